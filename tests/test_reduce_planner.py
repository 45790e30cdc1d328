"""The reduce planner's choice between the plain reduce (16-byte loads) and
the staged reduce (bulk copies through shared memory), checked on the CPU
through the library's test hook (host logic only: the addresses below are
never dereferenced).

The rule: the staged reduce runs when some row holds a full tile (2048
elements) and every accumulator is 16-byte aligned, and either a
contribution row starts off a 64-byte boundary or the rows hold at least
1 GiB of contributions."""
import pytest

Z = pytest.importorskip("fsdp_sharded_mixed_zero_gb300")

GIB = 1 << 30
BASE = 1 << 40                 # a 64-byte-aligned address


def form(dtype, n, rows, mode=0):
    return Z.zero_debug_reduce_form(dtype, n, rows, mode)


def test_aligned_rows_stage_from_one_gib():
    # 8 fp16 contributions: 16 bytes per element over the rows
    at = GIB // 16
    assert form(Z.ZERO_F16, 8, [(BASE, at, at)]) == "staged"
    assert form(Z.ZERO_F16, 8, [(BASE, at, at - 8)]) == "plain"       # 1 GiB - 128 B
    # the bytes of every row count (two rows of half the size)
    assert form(Z.ZERO_F16, 8, [(BASE, at, at // 2), (BASE + 64 * at, at, at // 2)]) == "staged"
    # fp32 contributions: 4 bytes per element
    assert form(Z.ZERO_F32, 8, [(BASE, GIB // 32, GIB // 32)]) == "staged"
    assert form(Z.ZERO_F32, 8, [(BASE, GIB // 32, GIB // 32 - 16)]) == "plain"
    # bf16 is a 2-byte encoding like fp16
    assert form(Z.ZERO_BF16, 4, [(BASE, GIB // 8, GIB // 8)]) == "staged"


def test_small_aligned_rows_stay_plain():
    # the tiny and small-group launches: rows 64-byte aligned, a few MB
    assert form(Z.ZERO_F16, 4, [(BASE, 1_050_112, 262_528)]) == "plain"
    assert form(Z.ZERO_F16, 8, [(BASE + 64 * k * 65_536, 65_536, 65_536) for k in range(8)]) \
        == "plain"


def test_misaligned_rows_stage_at_any_size():
    # a row stride that is not a multiple of 64 bytes (500,016 bytes)
    assert form(Z.ZERO_F16, 8, [(BASE, 250_008, 250_003)]) == "staged"
    # a first contribution off a 64-byte boundary (2-byte aligned slice)
    assert form(Z.ZERO_F16, 8, [(BASE + 14, 800_000_008, 100_000_001)]) == "staged"
    # 64 contributions 32 bytes off (the 1.5B shard's layout)
    assert form(Z.ZERO_F16, 64, [(BASE + 17 * 2 * 24_337_675, 24_337_680, 24_337_675)]) \
        == "staged"
    # one contributor: its row stride does not matter, only its start
    assert form(Z.ZERO_F16, 1, [(BASE, 250_003, 250_003)]) == "plain"
    assert form(Z.ZERO_F16, 1, [(BASE + 2, 250_003, 250_003)]) == "staged"


def test_shards_below_a_tile_stay_plain():
    # no row holds a full 2048-element tile: plain, whatever the alignment or size
    assert form(Z.ZERO_F16, 1000, [(BASE + 2, 38_000, 38)]) == "plain"
    assert form(Z.ZERO_F16, 8, [(BASE + 2, 2_047, 2_047)]) == "plain"
    assert form(Z.ZERO_F16, 8, [(BASE + 2, 2_048, 2_048)]) == "staged"


def test_accumulation_needs_aligned_accumulators():
    rows = [(BASE + 14, 250_008, 250_003, BASE + (1 << 30))]
    assert form(Z.ZERO_F16, 8, rows, mode=1) == "staged"
    assert form(Z.ZERO_F16, 8, rows, mode=2) == "staged"
    bad = [(BASE + 14, 250_008, 250_003, BASE + (1 << 30) + 8)]         # 8-byte aligned only
    assert form(Z.ZERO_F16, 8, bad, mode=1) == "plain"
    assert form(Z.ZERO_F16, 8, bad, mode=2) == "plain"


def test_bad_arguments_are_refused():
    with pytest.raises(Z.ZeroError):
        form(Z.ZERO_F16, 0, [(BASE, 4096, 4096)])
    with pytest.raises(Z.ZeroError):
        form(7, 8, [(BASE, 4096, 4096)])
    with pytest.raises(Z.ZeroError):
        form(Z.ZERO_F16, 8, [(BASE, 4096, 4096)], mode=3)
    with pytest.raises(Z.ZeroError):
        Z.zero_debug_reduce_form(Z.ZERO_F16, 8, [], 0)
