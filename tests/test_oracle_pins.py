"""Pins of the oracle to facts other than itself: the pages' printed figures,
closed forms of the Adam update, special cases that reduce to library
routines, brute force in exact rational arithmetic on tiny buffers, hand-traced
loss-scale sequences, and the ZeRO == DDP invariant.  CPU only.

Page references are by title and section:
  "DeepSpeed 与 FSDP" (docs.ifdog.com)                       -> DS-FSDP
  "PyTorch FSDP ... 源码级深度解析" (tbr8.org)                -> FSDP-SRC
  the ZeRO paper reading at 2kiu.com/news/5312103            -> ZeRO reading
"""
import math
import os
from fractions import Fraction as Fr

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
GB = 10 ** 9


# --------------------------------------------------------------------------
# Memory accounting: DS-FSDP §逐步推导 and §ZeRO-3 的数学总结; ZeRO reading §1.

def test_memory_pure_dp_10b(ora):
    # 20 + 20 + 40 + 40 + 40 = 160 GB for a 10B model; optimizer = 120 GB = 75 %
    p, g, o, tot = ora.memory_breakdown(0, 10 * GB, 8)
    assert (p, g, o, tot) == (20 * GB, 20 * GB, 120 * GB, 160 * GB)
    assert o * 4 == tot * 3


def test_memory_zero_stages_10b_n8(ora):
    # ZeRO-1: 20 + 20 + 15 = 55 GB (optimizer state 15 GB per GPU)
    assert ora.memory_breakdown(1, 10 * GB, 8) == (20 * GB, 20 * GB, 15 * GB, 55 * GB)
    # ZeRO-2: 20 + 2.5 + 15 = 37.5 GB
    assert ora.memory_breakdown(2, 10 * GB, 8) == (20 * GB, 2_500_000_000, 15 * GB,
                                                   37_500_000_000)
    # ZeRO-3: 2.5 + 2.5 + 15 = 20 GB
    assert ora.memory_breakdown(3, 10 * GB, 8) == (2_500_000_000, 2_500_000_000,
                                                   15 * GB, 20 * GB)


def test_memory_1p5b_and_175b(ora):
    # ZeRO reading §1: 1.5B -> fp16 params 3 GB, grads 3 GB; the figure 18 GB
    # is the 12-bytes-per-parameter optimizer state (12 * 1.5e9).  (The page's
    # own split "3 + 3 + 12 = 18" contradicts 12 bytes per parameter.)
    p, g, o, tot = ora.memory_breakdown(0, 1_500_000_000, 1)
    assert (p, g, o) == (3 * GB, 3 * GB, 18 * GB)
    assert tot == 24 * GB
    # 175B: fp16 params 350 GB, grads 350 GB, three fp32 states 700 GB each = 2100 GB
    p, g, o, tot = ora.memory_breakdown(0, 175 * GB, 1)
    assert (p, g, o) == (350 * GB, 350 * GB, 2100 * GB)


def test_memory_formula_limits_and_rounding(ora):
    # ZeRO-3 per-GPU memory tends to 0 as N grows; never below ceil(16 psi / N)
    assert ora.memory_breakdown(3, 10 * GB, 10 ** 6)[3] == 160_000
    # exact rational total, rounded up once: psi=1, N=3, ZeRO-1 -> 4 + 12/3 = 8
    assert ora.memory_breakdown(1, 1, 3)[3] == 8
    # psi=1, N=7, ZeRO-3 -> 16/7 -> 3 (parts 1, 1, 2 rounded separately)
    assert ora.memory_breakdown(3, 1, 7) == (1, 1, 2, 3)
    with pytest.raises(ValueError):
        ora.memory_breakdown(4, 1, 1)
    with pytest.raises(ValueError):
        ora.memory_breakdown(1, 1, 0)


# --------------------------------------------------------------------------
# Layout: FSDP-SRC §3.1 (_param_infos start/end), §3.3 (shard_size);
# DS-FSDP §FSDP 的分片粒度与 FlatParameter (chunk(world_size)[rank]).

def test_layout_workload_tables(ora):
    assert ora.layout([512 * 1024, 1024, 1024 * 512, 512], 4) == (1_050_112, 262_528, 1_050_112)
    assert ora.layout([10 ** 10], 8) == (10 ** 10, 1_250_000_000, 10 ** 10)
    assert ora.layout([1_557_611_200], 64) == (1_557_611_200, 24_337_675, 1_557_611_200)
    assert ora.layout([10], 4) == (10, 3, 12)
    assert ora.layout([0], 3) == (0, 0, 0)


def test_layout_matches_torch_chunk(ora):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    for _ in range(200):
        n = int(rng.integers(1, 500))
        N = int(rng.integers(1, 17))
        full, S, padded = ora.layout([n], N)
        assert full == n and padded == S * N and padded >= n and padded - n < N
        chunks = torch.arange(n).chunk(N)
        for r in range(N):
            want = chunks[r].tolist() if r < len(chunks) else []
            got = list(range(r * S, min((r + 1) * S, n)))
            assert got == want, (n, N, r)


def test_layout_numpy_array_split_demo(ora):
    # DS-FSDP §用 numpy 模拟: 16 parameters over 4 GPUs -> four shards of 4
    full, S, padded = ora.layout([16], 4)
    assert [len(s) for s in np.array_split(np.arange(16), 4)] == [S] * 4


def test_layout_rejects_bad_tables(ora):
    assert ora.layout_raw([0, 5], [4, 4], 2)[0] != 0      # gap between params
    assert ora.layout_raw([0, 3], [4, 4], 2)[0] != 0      # overlap
    assert ora.layout_raw([0], [4], 0)[0] != 0            # world_size 0
    assert ora.layout_raw([0], [-1], 1)[0] != 0
    assert ora.layout_raw([0, 2 ** 62], [2 ** 62, 2 ** 62], 1)[0] != 0  # int64 overflow


# --------------------------------------------------------------------------
# Number formats against numpy's / torch's IEEE-754 conversions (library).

def _structured_f32_patterns():
    rng = np.random.default_rng(7)
    hi = np.arange(1 << 19, dtype=np.uint32) << 13            # sign|exp|10 mantissa bits
    low = np.array([0, 1, 0xFFF, 0x1000, 0x1001, 0x1FFF], dtype=np.uint32)
    a = (hi[:, None] | low[None, :]).ravel()
    # whole binades around the fp16 subnormal range, the smallest subnormal
    # boundary and the overflow boundary, both signs
    parts = [a]
    for be in (101, 102, 103, 111, 112, 113, 142):
        m = np.arange(1 << 23, dtype=np.uint32)
        parts.append((np.uint32(be) << 23) | m)
        parts.append((np.uint32(0x100 + be) << 23) | m[::97])
    parts.append(rng.integers(0, 2 ** 32, size=1 << 22, dtype=np.uint64).astype(np.uint32))
    return np.concatenate(parts)


def test_cast_f16_matches_numpy(ora):
    u = _structured_f32_patterns()
    x = u.view(np.float32)
    got = ora.cast_array(x)
    want = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all(np.isnan(got[nan].view(np.float16)))


def test_cast_bf16_matches_torch(ora):
    torch = pytest.importorskip("torch")
    u = _structured_f32_patterns()
    # bf16's rounding point is bit 16: add all low-16 critical patterns
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    low = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    u = np.concatenate([u, (hi[:, None] | low[None, :]).ravel()])
    x = u.view(np.float32)
    got = ora.cast_array(x, to_bf16=True)
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    back = ora.decode_array(got[nan], from_bf16=True)
    assert np.all(np.isnan(back))


def test_decode_exhaustive(ora):
    torch = pytest.importorskip("torch")
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = ora.decode_array(h)
    want = h.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(f[~nan].view(np.uint32), want[~nan].view(np.uint32))
    assert np.all(np.isnan(f[nan]))
    b = ora.decode_array(h, from_bf16=True)
    wb = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nanb = np.isnan(wb)
    assert np.array_equal(b[~nanb].view(np.uint32), wb[~nanb].view(np.uint32))


# --------------------------------------------------------------------------
# Loss scale: hand-traced sequences (tests/golden, policy of the ZeRO reading
# §5.1 / §5.3).

def _load_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    return rows


@pytest.mark.parametrize("name,kw", [
    ("loss_scale_window2.txt", dict(dynamic=True, initial_scale_power=3, window=2,
                                    min_scale=1.0)),
    ("loss_scale_static.txt", dict(dynamic=False, static_scale=1.0, window=2)),
])
def test_scaler_hand_traced(ora, name, kw):
    hp = ora.hparams(**kw)
    st = ora.scaler_init(hp)
    for of, skipped, used, scale, good, t, ovf in _load_golden(name):
        assert st.scale == used
        coef, skip = ora.scaler_decide(hp, st, int(of), 0.5)
        assert skip == skipped
        assert st.as_tuple() == (scale, good, t, ovf)


def test_scaler_trace_through_full_step(ora):
    # the same trace, driven by real fp16 gradients with an injected +inf
    hp = ora.hparams(dynamic=True, initial_scale_power=3, window=2, min_scale=1.0,
                     lr=1e-3)
    st = ora.scaler_init(hp)
    n, N = 6, 2
    rng = np.random.default_rng(3)
    master = [rng.standard_normal(3).astype(np.float32) for _ in range(N)]
    m = [np.zeros(3, np.float32) for _ in range(N)]
    v = [np.zeros(3, np.float32) for _ in range(N)]
    out = np.zeros(6, np.uint16)
    for of, skipped, used, scale, good, t, ovf in _load_golden("loss_scale_window2.txt"):
        g = (rng.standard_normal((N, n)) * st.scale * 1e-2).astype(np.float16)
        if of:
            g[1, 4] = np.inf
        before = [a.copy() for a in master + m + v] + [out.copy()]
        res = ora.shard_step(hp, st, N, n, 3, [0, 1], g.view(np.uint16), n, 3,
                             master, m, v, out)
        assert (res.overflow, res.skipped, res.scale_used) == (of, skipped, used)
        assert st.as_tuple() == (scale, good, t, ovf)
        if skipped:   # a skipped step leaves master, m, v and the flat buffer alone
            after = [a for a in master + m + v] + [out]
            for x, y in zip(before, after):
                assert np.array_equal(x, y)


# --------------------------------------------------------------------------
# Reduce-scatter: DS-FSDP numpy demo (sum of the N gradients, then split),
# FSDP-SRC §3.3 (op AVG or SUM).

def test_reduce_scatter_is_sum_then_split(ora):
    rng = np.random.default_rng(11)
    N, n = 4, 16
    ints = rng.integers(-1000, 1000, size=(N, n))          # exact in fp16 and their sums
    grads = ints.astype(np.float16)
    full, S, padded = ora.layout([n], N)
    summed = ints.sum(axis=0)
    want_shards = np.array_split(summed, N)
    for r in range(N):
        g = ora.reduce_unscale(grads.view(np.uint16), n, r * S, N, S, r * S, full,
                               avg=False, scale=1.0)
        assert np.array_equal(g, want_shards[r].astype(np.float32))
        ga = ora.reduce_unscale(grads.view(np.uint16), n, r * S, N, S, r * S, full,
                                avg=True, scale=8.0)
        assert np.array_equal(ga, (want_shards[r] / (N * 8.0)).astype(np.float32))


def test_reduce_order_ld_offset_and_padding(ora):
    # N=3 contributors, 10 elements -> S=4, padded 12; garbage in the padding
    rng = np.random.default_rng(5)
    N, n, ld = 3, 10, 16
    full, S, padded = ora.layout([n], N)
    buf = (rng.standard_normal((N, ld)) * 7).astype(np.float16)
    buf[:, n:] = np.float16(np.inf)                          # beyond full_numel
    for r in range(N):
        g = ora.reduce_unscale(buf.view(np.uint16), ld, r * S, N, S, r * S, full,
                               avg=True, scale=4.0)
        acc = np.zeros(S, np.float32)
        for c in range(N):                                   # sequential fp32 sum
            acc = acc + buf[c, r * S:(r + 1) * S].astype(np.float32)
        want = (acc / np.float32(N)) / np.float32(4.0)
        valid = np.arange(r * S, (r + 1) * S) < n
        assert np.array_equal(g[valid], want[valid])
        assert np.all(g[~valid] == 0)


def test_sum_of_squares_is_exact(ora):
    # the exact sum of the exact squares, rounded once: math.fsum's answer
    rng = np.random.default_rng(2)
    g = rng.standard_normal(100_000).astype(np.float32)
    ss, of = ora.sum_of_squares(g)
    assert of == 0 and ss == math.fsum(float(x) * float(x) for x in g)
    # extreme magnitudes: subnormal, tiny, huge and mixed scales
    ext = np.array([2.0 ** -149, 2.0 ** -126, 3.0e-30, 1.0, 1.0e30, 3.4e38, 2.0 ** -149,
                    7.0, 1e-20], np.float32)
    exact = sum((Fr(float(x)) ** 2 for x in ext), Fr(0))
    assert ora.sum_of_squares(ext)[0] == float(exact)        # Fraction -> nearest double
    acc, _ = ora.norm_accumulate(np.ones(3, np.float32))
    assert ora.norm_sum(acc) == 3.0
    # order and splitting do not matter
    parts = [ora.norm_accumulate(c)[0] for c in np.array_split(g, 7)]
    tot = ora.ExactAcc()
    for p_ in parts[::-1]:
        ora.acc_merge(tot, p_)
    assert ora.norm_sum(tot) == ss
    g[123] = np.nan
    assert ora.sum_of_squares(g)[1] == 1
    g[123] = -np.inf
    assert ora.sum_of_squares(g)[1] == 1


def test_exact_accumulators_merge_with_carries(ora):
    # Merging two exact accumulators carries between 64-bit limbs.  Units are
    # 2^-298, so 2^84 sits at bit 382 (limb 5); two squares of 2^42 make 2^85
    # (limb 5's top bit) in each accumulator, and their merge 2^86 (limb 6).
    x = np.full(2, 2.0 ** 42, np.float32)
    a, b = ora.norm_accumulate(x)[0], ora.norm_accumulate(x)[0]
    assert ora.norm_sum(ora.acc_merge(a, b)) == 2.0 ** 86
    # Random magnitudes over the whole fp32 range, many squares of one binade
    # (so limbs fill and carry), split at random and merged in random order:
    # the exact sum rounded once (Fraction -> nearest double).
    rng = np.random.default_rng(11)
    for _ in range(10):
        wide = np.ldexp(rng.uniform(1.0, 2.0, 200), rng.integers(-149, 127, 200))
        same = np.ldexp(rng.uniform(1.9, 2.0, 300), 42)
        g = (np.concatenate([wide, same]) * rng.choice([-1.0, 1.0], 500)).astype(np.float32)
        rng.shuffle(g)
        exact = float(sum((Fr(float(v)) ** 2 for v in g), Fr(0)))
        cuts = np.sort(rng.choice(np.arange(1, g.size), 6, replace=False))
        parts = [ora.norm_accumulate(p)[0] for p in np.split(g, cuts)]
        tot = ora.ExactAcc()
        for k in rng.permutation(len(parts)):
            ora.acc_merge(tot, parts[k])
        assert ora.norm_sum(tot) == exact == ora.sum_of_squares(g)[0]


def test_sum_of_squares_rounding_ties(ora):
    # (2^26)^2 + (2^26)^2 + 1 = 2^53 + 1 is halfway between two doubles
    x = np.array([2.0 ** 26, 2.0 ** 26, 1.0], np.float32)   # 2^53 + 1 exactly
    assert ora.sum_of_squares(x)[0] == float(Fr(2 ** 53 + 1))   # ties to even: 2^53
    y = np.array([2.0 ** 26, 2.0 ** 26, 1.0, 1.0, 1.0], np.float32)  # 2^53 + 3
    assert ora.sum_of_squares(y)[0] == float(Fr(2 ** 53 + 3))   # ties to even: 2^53 + 4
    # a tie broken by the smallest possible square: (2^-149)^2 = 2^-298, the
    # lowest bit the exact sum can hold, lifts 2^53 + 1 above the halfway point
    z = np.array([2.0 ** 26, 2.0 ** 26, 1.0, 2.0 ** -149], np.float32)
    exact = Fr(2 ** 53 + 1) + Fr(1, 2 ** 298)
    assert ora.sum_of_squares(z)[0] == float(exact) == 2.0 ** 53 + 2


# --------------------------------------------------------------------------
# Adam closed forms: DS-FSDP §ZeRO-Offload (Adam with bias correction),
# decoupled weight decay (ZeRO reading §5.1, AdamW).

def _f32_ulp(x):
    x = np.abs(np.float32(x))
    return float(np.spacing(x))


def test_step1_closed_form(ora):
    # t=1, m=v=0, no clipping: theta1 = theta0 (1 - lr wd) - lr g / (|g| + eps)
    rng = np.random.default_rng(0)
    n = 4096
    lr, wd, eps = 1e-2, 0.1, 1e-8
    hp = ora.hparams(lr=lr, weight_decay=wd, eps=eps, max_grad_norm=0.0)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    th0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    th, m, v = th0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    ora.adamw_cast(hp, 1, 1.0, g, th, m, v)
    gd = g.astype(np.float64)
    want = th0.astype(np.float64) * (1 - lr * wd) - lr * gd / (np.abs(gd) + eps)
    # rounding error is a few ulps of the operands (theta0*d and lr), not of a
    # result that may cancel to near zero
    mag = np.maximum(np.abs(th0.astype(np.float64)), lr)
    ulps = np.abs(th - want) / np.array([_f32_ulp(x) for x in mag])
    assert ulps.max() <= 4, ulps.max()
    assert np.allclose(m, 0.1 * gd, rtol=3e-7, atol=0)
    assert np.allclose(v, 0.001 * gd * gd, rtol=5e-7, atol=0)


def test_zero_gradient_is_pure_decay(ora):
    hp = ora.hparams(lr=3e-5, weight_decay=0.01)
    th0 = np.linspace(-1, 1, 101).astype(np.float32)
    th, m, v = th0.copy(), np.zeros(101, np.float32), np.zeros(101, np.float32)
    out = ora.adamw_cast(hp, 1, 1.0, np.zeros(101, np.float32), th, m, v)
    decay = np.float32(1.0 - 3e-5 * 0.01)
    assert np.array_equal(th, th0 * decay)
    assert not m.any() and not v.any()
    assert np.array_equal(out, (th0 * decay).astype(np.float16).view(np.uint16))


def test_constant_gradient_closed_form(ora):
    # With a constant g the bias-corrected moments are exactly g and g^2 at
    # every t, so each step is theta <- theta*d - lr*g/(|g|+eps).
    rng = np.random.default_rng(4)
    n, T = 2048, 6
    lr, wd, eps = 1e-3, 0.05, 1e-8
    hp = ora.hparams(lr=lr, weight_decay=wd, eps=eps, max_grad_norm=0.0)
    g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    th0 = (rng.standard_normal(n) * 0.05).astype(np.float32)
    th, m, v = th0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(1, T + 1):
        ora.adamw_cast(hp, t, 1.0, g, th, m, v)
    gd = g.astype(np.float64)
    d = 1 - lr * wd
    s = gd / (np.abs(gd) + eps)
    want = th0.astype(np.float64) * d ** T - lr * s * sum(d ** k for k in range(T))
    assert np.max(np.abs(th - want)) <= 16 * _f32_ulp(0.1)
    assert np.allclose(m, (1 - 0.9 ** T) * gd, rtol=2e-6, atol=0)
    assert np.allclose(v, (1 - 0.999 ** T) * gd * gd, rtol=2e-6, atol=0)


def test_two_gradient_closed_form(ora):
    # t=2 after g1, g2: mh = (b1 g1 + g2)/(1+b1), vh = (b2 g1^2 + g2^2)/(1+b2)
    rng = np.random.default_rng(8)
    n = 2048
    lr, wd, eps, b1, b2 = 1e-3, 0.01, 1e-8, 0.9, 0.999
    hp = ora.hparams(lr=lr, weight_decay=wd, eps=eps, max_grad_norm=0.0)
    g1 = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    g2 = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    th0 = (rng.standard_normal(n) * 0.05).astype(np.float32)
    th, m, v = th0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    ora.adamw_cast(hp, 1, 1.0, g1, th, m, v)
    ora.adamw_cast(hp, 2, 1.0, g2, th, m, v)
    a, b = g1.astype(np.float64), g2.astype(np.float64)
    d = 1 - lr * wd
    th1 = th0.astype(np.float64) * d - lr * a / (np.abs(a) + eps)
    mh = (b1 * a + b) / (1 + b1)
    vh = (b2 * a * a + b * b) / (1 + b2)
    want = th1 * d - lr * mh / (np.sqrt(vh) + eps)
    assert np.max(np.abs(th - want)) <= 8 * _f32_ulp(0.2)
    # the betas must not be swapped: the swapped answer is far away
    mh_s = (b2 * a + b) / (1 + b2)
    vh_s = (b1 * a * a + b * b) / (1 + b1)
    swapped = th1 * d - lr * mh_s / (np.sqrt(vh_s) + eps)
    assert np.max(np.abs(swapped - want)) > 100 * _f32_ulp(0.2)


def test_skipped_step_does_not_advance_t(ora):
    # g1 applied, overflowing step skipped, g2 applied with t=2 (closed form)
    rng = np.random.default_rng(9)
    n, lr, wd, eps = 64, 1e-3, 0.0, 1e-8
    hp = ora.hparams(lr=lr, weight_decay=wd, eps=eps, max_grad_norm=0.0,
                     dynamic=True, initial_scale_power=0)
    st = ora.scaler_init(hp)
    g1 = rng.standard_normal(n).astype(np.float16)
    g2 = rng.standard_normal(n).astype(np.float16)
    bad = g2.copy()
    bad[7] = np.inf
    th0 = (rng.standard_normal(n) * 0.05).astype(np.float32)
    th, m, v = [th0.copy()], [np.zeros(n, np.float32)], [np.zeros(n, np.float32)]
    out = np.zeros(n, np.uint16)
    for gg in (g1, bad, g2):
        ora.shard_step(hp, st, 1, n, n, [0], gg.view(np.uint16), n, 0, th, m, v, out,
                       avg=False)
    assert st.step_t == 2 and st.overflow_count == 1
    a, b = g1.astype(np.float64), g2.astype(np.float64)
    th1 = th0.astype(np.float64) - lr * a / (np.abs(a) + eps)
    mh = (0.9 * a + b) / 1.9
    vh = (0.999 * a * a + b * b) / 1.999
    want = th1 - lr * mh / (np.sqrt(vh) + eps)
    assert np.max(np.abs(th[0] - want)) <= 8 * _f32_ulp(0.2)


def test_clip_coefficient_closed_form(ora):
    # one contributor, g = (3, 4) * 2^k -> norm exactly 5 * 2^k
    hp = ora.hparams(lr=1e-3, max_grad_norm=1.0, dynamic=False, static_scale=1.0)
    for k in (-3, 0, 2):
        st = ora.scaler_init(hp)
        g = np.array([3 * 2.0 ** k, 4 * 2.0 ** k, 0, 0], np.float16)
        th, m, v = [np.zeros(4, np.float32)], [np.zeros(4, np.float32)], [np.zeros(4, np.float32)]
        out = np.zeros(4, np.uint16)
        res = ora.shard_step(hp, st, 1, 4, 4, [0], g.view(np.uint16), 4, 0, th, m, v, out,
                             avg=False)
        norm = 5 * 2.0 ** k
        assert res.grad_norm == norm
        q = 1.0 / (norm + 1e-6)
        want_coef = np.float32(q) if q < 1 else np.float32(1.0)
        assert res.clip_coef == want_coef
        gc = np.float32(g[:2].astype(np.float32) * want_coef)
        assert np.array_equal(m[0][:2], np.float32(0.1) * gc)


def test_numpy_demo_special_case(ora):
    # DS-FSDP §用 numpy 模拟 ZeRO 分片过程: 4 GPUs, 16 parameters, gradients
    # summed then split, one Adam step with lr 1e-3, betas 0.9/0.999, eps 1e-8,
    # bias correction at t=1, no weight decay, no clipping, no loss scale.
    # numpy evaluates that script in float32 (float32 arrays, Python-float
    # scalars); the oracle must give the same bits on every shard.
    rng = np.random.default_rng(12)
    N, n = 4, 16
    full_param = rng.standard_normal(n).astype(np.float32)
    grads = [rng.standard_normal(n).astype(np.float16) for _ in range(N)]
    summed = np.zeros(n, np.float32)
    for gr in grads:
        summed = summed + gr.astype(np.float32)
    hp = ora.hparams(lr=1e-3, weight_decay=0.0, max_grad_norm=0.0, dynamic=False,
                     static_scale=1.0)
    st = ora.scaler_init(hp)
    master = [s.copy() for s in np.array_split(full_param, N)]
    m = [np.zeros(4, np.float32) for _ in range(N)]
    v = [np.zeros(4, np.float32) for _ in range(N)]
    out = np.zeros(n, np.uint16)
    ora.shard_step(hp, st, N, n, 4, list(range(N)), np.stack(grads).view(np.uint16), n, 4,
                   master, m, v, out, avg=False)
    lr, b1, b2, eps = 1e-3, 0.9, 0.999, 1e-8
    for r, g in enumerate(np.array_split(summed, N)):
        ms = np.zeros_like(g)
        vs = np.zeros_like(g)
        p = np.array_split(full_param, N)[r].copy()
        ms = b1 * ms + (1 - b1) * g
        vs = b2 * vs + (1 - b2) * g ** 2
        mh = ms / (1 - b1)
        vh = vs / (1 - b2)
        p -= lr * mh / (np.sqrt(vh) + eps)
        assert p.dtype == np.float32
        assert np.array_equal(master[r], p)
        assert np.array_equal(m[r], ms) and np.array_equal(v[r], vs)


# --------------------------------------------------------------------------
# Brute force in exact rational arithmetic, every fp32 rounding explicit.

def _rf32(q):
    """Round a rational to the nearest binary32 (ties to even); normal range."""
    if q == 0:
        return Fr(0)
    s = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fr(2) ** e > a:
        e -= 1
    while Fr(2) ** (e + 1) <= a:
        e += 1
    qe = max(e, -126) - 23
    x = a / Fr(2) ** qe
    k = x.numerator // x.denominator
    rem = x - k
    if rem > Fr(1, 2) or (rem == Fr(1, 2) and k % 2 == 1):
        k += 1
    return s * k * Fr(2) ** qe


def _sqrt_f32(q):
    """Correctly rounded binary32 square root of a non-negative rational."""
    if q == 0:
        return Fr(0)
    E = q.numerator.bit_length() - q.denominator.bit_length()
    while Fr(2) ** E > q:
        E -= 1
    while Fr(2) ** (E + 1) <= q:
        E += 1
    e = E // 2
    x = q * Fr(4) ** (23 - e)          # sqrt(x) = sqrt(q) / 2^(e-23), in [2^23, 2^24)
    k = math.isqrt(x.numerator // x.denominator)
    mid = Fr(2 * k + 1, 2) ** 2
    if x > mid or (x == mid and k % 2 == 1):
        k += 1
    return k * Fr(2) ** (e - 23)


def _F(x):
    return Fr(float(np.float32(x)))


def _brute_step(hp, grads, N, S, full, ranks, master, m, v, scale, t, avg, extra=0.0):
    """Rational re-derivation of one step; returns updated lists and outputs."""
    f = _rf32
    g_all = []
    for r in ranks:
        gr = []
        for i in range(S):
            idx = r * S + i
            if idx >= full:
                gr.append(Fr(0))
                continue
            acc = Fr(0)
            for c in range(N):
                acc = f(acc + Fr(float(grads[c, idx])))
            if avg:
                acc = f(acc / N)
            gr.append(f(acc / Fr(float(scale))))
        g_all.append(gr)
    ss = sum((x * x for gr in g_all for x in gr), Fr(0))
    norm = math.sqrt(float(ss) + extra)
    q = hp.max_grad_norm / (norm + 1e-6)
    coef = _F(q) if (hp.max_grad_norm > 0 and q < 1) else Fr(1)
    b1, b2 = _F(hp.beta1), _F(hp.beta2)
    omb1, omb2 = _F(1 - hp.beta1), _F(1 - hp.beta2)
    bc1, bc2 = _F(1 - hp.beta1 ** t), _F(1 - hp.beta2 ** t)
    decay = _F(1 - hp.lr * hp.weight_decay)
    lr, eps = _F(hp.lr), _F(hp.eps)
    outs = []
    for j in range(len(ranks)):
        for i in range(S):
            gc = f(g_all[j][i] * coef)
            mi = f(f(b1 * Fr(float(m[j][i]))) + f(omb1 * gc))
            vi = f(f(b2 * Fr(float(v[j][i]))) + f(omb2 * f(gc * gc)))
            mh = f(mi / bc1)
            vh = f(vi / bc2)
            th = f(Fr(float(master[j][i])) * decay)
            th = f(th - f(f(lr * mh) / f(_sqrt_f32(vh) + eps)))
            master[j][i], m[j][i], v[j][i] = float(th), float(mi), float(vi)
            outs.append(float(th))
    return norm, float(coef), outs


@pytest.mark.parametrize("N,n,avg,scale", [(2, 8, True, 1024.0), (3, 8, False, 1.0),
                                           (3, 8, True, 65536.0),
                                           # a static scale that is not a power of two:
                                           # the AVG division and the unscale each round
                                           (3, 8, True, 5.0)])
def test_brute_force_tiny(ora, N, n, avg, scale):
    rng = np.random.default_rng(N * 100 + n)
    full, S, padded = ora.layout([n], N)
    hp = ora.hparams(lr=1e-2, weight_decay=0.1, max_grad_norm=0.05, dynamic=False,
                     static_scale=scale)
    grads = (rng.standard_normal((N, padded)) * scale * 0.1).astype(np.float16)
    master = [(rng.standard_normal(S) * 0.3).astype(np.float32) for _ in range(N)]
    m = [(rng.standard_normal(S) * 1e-2).astype(np.float32) for _ in range(N)]
    v = [(np.abs(rng.standard_normal(S)) * 1e-4).astype(np.float32) for _ in range(N)]
    bm = [list(map(float, a)) for a in master]
    bmm = [list(map(float, a)) for a in m]
    bv = [list(map(float, a)) for a in v]
    st = ora.scaler_init(hp)
    out = np.zeros(padded, np.uint16)
    for t in (1, 2):
        res = ora.shard_step(hp, st, N, full, S, list(range(N)), grads.view(np.uint16),
                             padded, S, master, m, v, out, avg=avg)
        norm, coef, outs = _brute_step(hp, grads.astype(np.float32), N, S, full,
                                       list(range(N)), bm, bmm, bv, scale, t, avg)
        assert res.clip_coef == coef and res.clip_coef < 1
        assert abs(res.grad_norm - norm) <= 1e-12 * norm
        for j in range(N):
            assert np.array_equal(master[j], np.array(bm[j], np.float32))
            assert np.array_equal(m[j], np.array(bmm[j], np.float32))
            assert np.array_equal(v[j], np.array(bv[j], np.float32))
        want_out = np.array(outs, np.float32).astype(np.float16).view(np.uint16)
        assert np.array_equal(out, want_out)
        grads = (rng.standard_normal((N, padded)) * scale * 0.1).astype(np.float16)


def test_one_rank_with_the_others_norm_share_steps_like_all_ranks(ora):
    # The clip / skip decision is one decision over every rank's gradient (ZeRO
    # reading §5.3): a rank stepped alone with extra_norm_sq = the other ranks'
    # sum of squares (here math.fsum over their reduced gradients) takes the
    # decision of the all-ranks step and updates its shard the same way.
    rng = np.random.default_rng(21)
    N, n = 4, 4001
    full, S, padded = ora.layout([n], N)
    hp = ora.hparams(lr=1e-3, max_grad_norm=1.0, dynamic=False, static_scale=1.0)
    grads = (rng.standard_normal((N, padded)) * 0.05).astype(np.float16)
    grads[:, full:] = 0
    theta = (rng.standard_normal(padded) * 0.02).astype(np.float32)
    r = 2
    others = [ora.reduce_unscale(grads.view(np.uint16), padded, k * S, N, S, k * S, full,
                                 avg=True, scale=1.0) for k in range(N) if k != r]
    extra = math.fsum(float(x) * float(x) for g in others for x in g)
    st_all, st_one = ora.scaler_init(hp), ora.scaler_init(hp)
    all_state = [[theta[k * S:(k + 1) * S].copy() for k in range(N)],
                 [np.zeros(S, np.float32) for _ in range(N)],
                 [np.zeros(S, np.float32) for _ in range(N)]]
    one_state = [[theta[r * S:(r + 1) * S].copy()], [np.zeros(S, np.float32)],
                 [np.zeros(S, np.float32)]]
    out_all, out_one = np.zeros(padded, np.uint16), np.zeros(padded, np.uint16)
    ra = ora.shard_step(hp, st_all, N, full, S, list(range(N)), grads.view(np.uint16), padded,
                        S, *all_state, out_all)
    ro = ora.shard_step(hp, st_one, N, full, S, [r], grads.view(np.uint16), padded, S,
                        *one_state, out_one, extra_norm_sq=extra)
    assert ra.clip_coef < 1.0                                  # clipping is active
    assert abs(ro.grad_norm - ra.grad_norm) <= 4e-16 * ra.grad_norm
    assert (ro.overflow, ro.skipped, ro.clip_coef) == (ra.overflow, ra.skipped, ra.clip_coef)
    for x, y in zip(one_state, all_state):
        assert np.array_equal(x[0], y[r])
    assert np.array_equal(out_one[r * S:(r + 1) * S], out_all[r * S:(r + 1) * S])


# --------------------------------------------------------------------------
# ZeRO == DDP (ZeRO reading §5.2: same optimizer update sequence as DDP).

@pytest.mark.parametrize("N,n,bf16,avg", [(2, 1000, False, True), (3, 1001, False, True),
                                          (4, 4099, True, False), (8, 12345, False, True)])
def test_zero_equals_ddp(ora, N, n, bf16, avg):
    rng = np.random.default_rng(N + n)
    full, S, padded = ora.layout([n // 3, n - n // 3], N)
    scale_kw = dict(dynamic=False, static_scale=1.0) if bf16 else dict(dynamic=True)
    hp = ora.hparams(lr=1e-3, weight_decay=0.01, max_grad_norm=1.0, window=2, **scale_kw)
    st_z, st_d = ora.scaler_init(hp), ora.scaler_init(hp)
    th = (rng.standard_normal(padded) * 0.02).astype(np.float32)
    th[full:] = 0
    zm = [th[r * S:(r + 1) * S].copy() for r in range(N)]
    zmm = [np.zeros(S, np.float32) for _ in range(N)]
    zv = [np.zeros(S, np.float32) for _ in range(N)]
    dth, dm, dv = th[:full].copy(), np.zeros(full, np.float32), np.zeros(full, np.float32)
    zout = np.zeros(padded, np.uint16)
    dout = np.zeros(full, np.uint16)
    for step in range(5):
        g = rng.standard_normal((N, padded)) * (1e-1 if step != 1 else 1e-3)
        g = g * (1.0 if bf16 else st_z.scale)
        if bf16:
            import torch
            gh = torch.from_numpy(g.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        else:
            gh = g.astype(np.float16).view(np.uint16)
        gh = gh.copy()
        if step == 3 and not bf16:
            gh[N - 1, full // 2] = 0x7C00                      # +inf: skipped step
        if padded > full:
            gh[:, full:] = 0x7E00                              # NaN in padding: ignored
        rz = ora.shard_step(hp, st_z, N, full, S, list(range(N)), gh, padded, S,
                            zm, zmm, zv, zout, avg=avg, grad_is_bf16=bf16,
                            param_is_bf16=bf16)
        rd = ora.ddp_step(hp, st_d, N, full, gh, padded, dth, dm, dv, dout, avg=avg,
                          grad_is_bf16=bf16, param_is_bf16=bf16)
        assert (rz.overflow, rz.skipped, rz.grad_norm, rz.clip_coef) == \
               (rd.overflow, rd.skipped, rd.grad_norm, rd.clip_coef)
        assert st_z.as_tuple() == st_d.as_tuple()
        assert np.array_equal(np.concatenate(zm)[:full], dth)
        assert np.array_equal(np.concatenate(zmm)[:full], dm)
        assert np.array_equal(np.concatenate(zv)[:full], dv)
        assert np.array_equal(zout[:full], dout)
        assert not np.concatenate(zm)[full:].any()             # padding stays zero
    assert st_z.step_t == (5 if bf16 else 4)


# --------------------------------------------------------------------------
# fp32 contributions (reduce_dtype=float32, DS-FSDP §PyTorch FSDP 使用) and
# gradient accumulation across micro-steps (DS-FSDP §实践要点; ZeRO reading
# §5.1 contiguous_gradients).

def test_fp32_contributions_sum_then_split(ora):
    rng = np.random.default_rng(21)
    N, n = 4, 40
    ints = rng.integers(-2 ** 20, 2 ** 20, size=(N, n))       # exact in fp32, sums too
    grads = ints.astype(np.float32)
    full, S, padded = ora.layout([n], N)
    want = np.array_split(ints.sum(axis=0), N)
    for r in range(N):
        g = ora.reduce_unscale(grads, n, r * S, N, S, r * S, full, avg=False, scale=1.0)
        assert np.array_equal(g, want[r].astype(np.float32))


def test_fp32_contributions_sequential_order(ora):
    rng = np.random.default_rng(22)
    N, S = 5, 1000
    grads = rng.standard_normal((N, S)).astype(np.float32) * np.float32(1e3)
    g = ora.reduce_unscale(grads, S, 0, N, S, 0, S, avg=True, scale=4.0)
    acc = np.zeros(S, np.float32)
    for c in range(N):
        acc = acc + grads[c]
    assert np.array_equal(g, (acc / np.float32(N)) / np.float32(4.0))


def test_accumulation_is_the_sum_of_micro_steps(ora):
    rng = np.random.default_rng(23)
    N, n, K = 4, 64, 5
    full, S, padded = ora.layout([n], N)
    acc = [np.full(S, 7.0, np.float32) for _ in range(N)]     # overwritten by first=True
    total = np.zeros((N, padded), np.int64)
    for k in range(K):
        ints = rng.integers(-1000, 1000, size=(N, padded))
        total += ints
        ora.grad_accumulate(N, full, S, list(range(N)), ints.astype(np.float16).view(np.uint16),
                            padded, S, acc, first=(k == 0), avg=True)
    want = total.sum(axis=0) / N                              # exact: N is a power of two
    for r in range(N):
        assert np.array_equal(acc[r], want[r * S:(r + 1) * S].astype(np.float32))


@pytest.mark.parametrize("kind", ["f16", "bf16", "f32"])
def test_one_micro_step_equals_the_direct_step(ora, kind):
    # accumulate once (first=True), then step from the accumulator: the same
    # bits as the direct step on the same contributions
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(24)
    N, n = 3, 1001
    full, S, padded = ora.layout([n], N)
    x = rng.standard_normal((N, padded)) * 100.0
    if kind == "f16":
        grads, bf = x.astype(np.float16).view(np.uint16), False
    elif kind == "bf16":
        grads = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(
            torch.int16).numpy().view(np.uint16)
        bf = True
    else:
        grads, bf = x.astype(np.float32), False
    hp = ora.hparams(lr=1e-3, max_grad_norm=1.0, initial_scale_power=3)
    sa, sb = ora.scaler_init(hp), ora.scaler_init(hp)
    th = [(rng.standard_normal(S) * 0.02).astype(np.float32) for _ in range(N)]
    A = [[t.copy() for t in th], [np.zeros(S, np.float32) for _ in range(N)],
         [np.zeros(S, np.float32) for _ in range(N)], np.zeros(padded, np.uint16)]
    B = [[t.copy() for t in th], [np.zeros(S, np.float32) for _ in range(N)],
         [np.zeros(S, np.float32) for _ in range(N)], np.zeros(padded, np.uint16)]
    ra = ora.shard_step(hp, sa, N, full, S, list(range(N)), grads, padded, S, A[0], A[1], A[2],
                        A[3], avg=True, grad_is_bf16=bf)
    acc = [np.zeros(S, np.float32) for _ in range(N)]
    ora.grad_accumulate(N, full, S, list(range(N)), grads, padded, S, acc, first=True,
                        avg=True, grad_is_bf16=bf)
    rb = ora.shard_step_acc(hp, sb, N, full, S, list(range(N)), acc, B[0], B[1], B[2], B[3])
    assert (ra.overflow, ra.skipped, ra.grad_norm, ra.clip_coef, ra.scale_used) == \
           (rb.overflow, rb.skipped, rb.grad_norm, rb.clip_coef, rb.scale_used)
    assert sa.as_tuple() == sb.as_tuple()
    for xa, xb in zip(A[0] + A[1] + A[2] + [A[3]], B[0] + B[1] + B[2] + [B[3]]):
        assert np.array_equal(xa, xb)


def test_cancelling_micro_steps_give_pure_decay(ora):
    # micro-steps G and -G accumulate to exactly zero: the step is theta*decay
    rng = np.random.default_rng(25)
    N, n = 2, 500
    full, S, padded = ora.layout([n], N)
    G = (rng.standard_normal((N, padded)) * 1000).astype(np.float16)
    acc = [np.zeros(S, np.float32) for _ in range(N)]
    ora.grad_accumulate(N, full, S, [0, 1], G.view(np.uint16), padded, S, acc, first=True)
    ora.grad_accumulate(N, full, S, [0, 1], (-G).view(np.uint16), padded, S, acc, first=False)
    assert all(not a.any() for a in acc)
    hp = ora.hparams(lr=1e-2, weight_decay=0.1)
    st = ora.scaler_init(hp)
    th0 = [(rng.standard_normal(S) * 0.3).astype(np.float32) for _ in range(N)]
    th = [t.copy() for t in th0]
    m = [np.zeros(S, np.float32) for _ in range(N)]
    v = [np.zeros(S, np.float32) for _ in range(N)]
    res = ora.shard_step_acc(hp, st, N, full, S, [0, 1], acc, th, m, v,
                             np.zeros(padded, np.uint16))
    assert res.grad_norm == 0.0 and res.skipped == 0
    decay = np.float32(1.0 - 1e-2 * 0.1)
    for a, b in zip(th, th0):
        assert np.array_equal(a, b * decay)


def test_step_from_accumulator_overflow_and_padding(ora):
    N, n = 3, 10
    full, S, padded = ora.layout([n], N)                      # S=4, two padding elements
    hp = ora.hparams(initial_scale_power=4)
    st = ora.scaler_init(hp)
    acc = [np.ones(S, np.float32) for _ in range(N)]
    acc[2][3] = np.inf                                        # padding: ignored
    th = [np.zeros(S, np.float32) for _ in range(N)]
    m = [np.zeros(S, np.float32) for _ in range(N)]
    v = [np.zeros(S, np.float32) for _ in range(N)]
    res = ora.shard_step_acc(hp, st, N, full, S, [0, 1, 2], acc, th, m, v,
                             np.zeros(padded, np.uint16))
    assert res.overflow == 0 and abs(res.grad_norm - np.sqrt(10) / 16) < 1e-15
    acc[1][0] = np.nan
    res = ora.shard_step_acc(hp, st, N, full, S, [0, 1, 2], acc, th, m, v,
                             np.zeros(padded, np.uint16))
    assert res.overflow == 1 and res.skipped == 1 and st.scale == 8.0


# --------------------------------------------------------------------------
# ZeRO++ quantized weight all-gather payload (DS-FSDP §ZeRO++; ZeRO reading
# §4.2): int8 codes halve the fp16 payload; the receiver dequantizes.

def _q8_exact(p, block):
    """Rational re-derivation: scale = RN32(amax / 127), code = round-half-even
    of the fp32-rounded quotient, clamped."""
    codes, scales = [], []
    for b0 in range(0, len(p), block):
        blk = [Fr(float(x)) for x in p[b0:b0 + block]]
        amax = max(abs(x) for x in blk)
        scale = _rf32(amax / 127) if amax else Fr(0)
        scales.append(float(scale))
        for x in blk:
            if scale == 0:
                codes.append(0)
                continue
            v = _rf32(x / scale)
            k = v.numerator // v.denominator
            rem = v - k
            if rem > Fr(1, 2) or (rem == Fr(1, 2) and k % 2 == 1):
                k += 1
            codes.append(max(-127, min(127, int(k))))
    return np.array(codes, np.int8), np.array(scales, np.float32)


@pytest.mark.parametrize("n,block", [(1000, 256), (256, 256), (77, 32), (5, 8)])
def test_q8_matches_exact_rounding(ora, n, block):
    rng = np.random.default_rng(n)
    p = (rng.standard_normal(n) * 0.05).astype(np.float16).astype(np.float32)
    p[::17] = 0.0
    q, sc = ora.quantize_q8(p, block)
    wq, wsc = _q8_exact(p, block)
    assert np.array_equal(q, wq) and np.array_equal(sc, wsc)


def test_q8_properties(ora):
    rng = np.random.default_rng(40)
    p = (rng.standard_normal(100_000) * np.exp(rng.standard_normal(100_000))).astype(
        np.float16).astype(np.float32)
    q, sc = ora.quantize_q8(p, 256)
    assert q.min() >= -127 and q.max() <= 127
    deq = q.astype(np.float64) * np.repeat(sc.astype(np.float64), 256)[:p.size]
    # every block's largest magnitude maps to +-127, and the error is at most
    # half a quantization step (plus fp32 rounding of the quotient)
    for k in range(sc.size):
        blk = np.abs(p[k * 256:(k + 1) * 256])
        assert np.abs(q[k * 256:(k + 1) * 256]).max() == (127 if blk.max() > 0 else 0)
    step = np.repeat(sc.astype(np.float64), 256)[:p.size]
    assert np.all(np.abs(deq - p) <= step * (0.5 + 1e-5))
    # payload: 1 byte per parameter + one fp32 scale per 256 -> about half of fp16
    assert abs((p.size + 4 * sc.size) / (2 * p.size) - 0.5078) < 1e-3


def test_q8_special_values(ora):
    z, sz = ora.quantize_q8(np.zeros(10, np.float32), 4)
    assert not z.any() and not sz.any()
    p = np.array([1.0, -1.0, 0.5, np.nan, np.inf, -2.0, 3.0, 0.0], np.float32)
    q, sc = ora.quantize_q8(p, 4)
    assert list(q[:3]) == [127, -127, 64] and q[3] == 0        # 63.5 -> 64 (even)
    assert sc[1] == np.inf and list(q[4:]) == [0, 0, 0, 0]     # inf block: inf/inf -> NaN -> 0
