"""zero_shard_step_noalloc -- the shard step for callers that may not
allocate device memory (for instance code running under a framework whose
caching allocator owns all device memory, where zero_flat_init's cudaMalloc
is not allowed).

Each case runs three calls in a row through the C ABI, the second one with an
inf planted in one gradient contribution, beside the handle-based
zero_shard_step on an identical copy of the inputs and beside the oracle:
  - against the handle step: the same kernels run on the same bytes, so the
    result, the loss-scale state, master, m, v and the flat buffer must be
    bit-identical;
  - against the oracle: within the parity tolerances of the other GPU tests
    (overflow, skip and loss-scale state bit-exact);
  - the overflowing call must skip (state and slot untouched) and halve a
    dynamic scale, and the next clean call must match again.
The layouts take both reduce kernels through this entry point: contributor
rows whose starts are off a 64-byte boundary (the staged reduce) and rows
that all start on one (the vectorised reduce).  Oversized shards must be
refused with a clear error.  This file is collected last on purpose and
builds everything it uses itself, so it passes alone or after the other
tests."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import synth  # noqa: E402
from tests.gpu_helpers import (assert_params_close, assert_result, assert_state, f32,  # noqa: E402
                               host_grads, u16)

pytestmark = pytest.mark.gpu

F16, BF16, F32, SUM, AVG = 0, 1, 2, 0, 1
INF_CALL = 1
CASES = [
    # all four shards of a ragged FlatParameter, fp16, AVG, dynamic loss scale;
    # odd shard size: rank slices start 2-byte aligned (staged reduce)
    dict(name="all_shards_fp16_staged", full=300_001, N=4, ranks=[0, 1, 2, 3], dtype=F16,
         op=AVG, dynamic=True, layout="full"),
    # one rank's slice of an 8-way group, bf16, SUM, static scale; row
    # stride 500,000 bytes: rows 32 bytes off a 64-byte boundary (staged)
    dict(name="slice_bf16_staged", full=2_000_000, N=8, ranks=[5], dtype=BF16, op=SUM,
         dynamic=False, layout="slice"),
    # every contributor row and rank slice on a 64-byte boundary (the
    # vectorised reduce), fp16, AVG, dynamic
    dict(name="all_shards_fp16_aligned", full=4 * 65_536, N=4, ranks=[0, 1, 2, 3], dtype=F16,
         op=AVG, dynamic=True, layout="full"),
    # fp32 contributions (reduce_dtype=float32) and fp16 parameters; odd shard:
    # 4-byte-aligned rank slices (the staged reduce's fp32 form)
    dict(name="two_shards_fp32_contributions", full=400_001, N=3, ranks=[0, 2], dtype=F16,
         gdtype=F32, op=AVG, dynamic=True, layout="full"),
]


def _setup(case):
    N, full = case["N"], case["full"]
    S = -(-full // N)
    padded = S * N
    tdt = torch.float16 if case["dtype"] == F16 else torch.bfloat16
    ld = padded if case["layout"] == "full" else -(-S // 8) * 8
    gtdt = torch.float32 if case.get("gdtype") == F32 else tdt
    grads = torch.empty((N, ld), dtype=gtdt, device="cuda")
    states = []
    for _ in range(2):                                   # identical copies: A and B
        master = []
        for r in case["ranks"]:
            t = torch.empty(S, dtype=torch.float32, device="cuda")
            synth.normal_device(t, 21, synth.MASTER, r * S, 0.02)
            t[max(0, min(S, full - r * S)):].zero_()
            master.append(t)
        m = [torch.zeros(S, device="cuda") for _ in case["ranks"]]
        v = [torch.zeros(S, device="cuda") for _ in case["ranks"]]
        out = torch.zeros(padded, dtype=tdt, device="cuda")
        out.view(torch.int16).fill_(0x3C3C)
        states.append((master, m, v, out))
    return S, padded, ld, grads, states


def _gen(case, grads, S, step, scale):
    dt = synth.F32 if case.get("gdtype") == F32 else (
        synth.F16 if case["dtype"] == F16 else synth.BF16)
    r0 = case["ranks"][0]
    if case["layout"] == "full":
        synth.grads_device(grads, 21, step, 0, grads.shape[1], 1e-3, 1e-3, scale, dt,
                           zero_from=case["full"])
    else:
        synth.grads_device(grads, 21, step, r0 * S, S, 1e-3, 1e-3, scale, dt,
                           zero_from=case["full"])
    if step == INF_CALL:                        # one contribution of one stepped element
        col = 12_345 if case["layout"] == "slice" else r0 * S + 12_345
        grads[case["N"] - 1, col] = float("inf")


def _same_bits(a, b):
    return np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                          b.view(np.uint32) if b.dtype == np.float32 else b)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c["name"])
def test_noalloc_matches_handle_step_and_oracle(ora, case):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import fsdp_sharded_mixed_zero_gb300 as Z
    kw = dict(dynamic=case["dynamic"], lr=1e-3)
    hp = Z.hparams(**kw)
    ohp = ora.hparams(**kw)
    bf16 = case["dtype"] == BF16
    gdt = case.get("gdtype", case["dtype"])
    S, padded, ld, grads, (A, B) = _setup(case)
    flat = Z.ZeroFlat([(case["full"],)], case["N"], gdt, case["dtype"], case["op"], hp)
    state = Z.ScalerState(65536.0 if case["dynamic"] else 1.0, 0, 0, 0)
    mul = S if case["layout"] == "full" else 0
    stream = torch.cuda.current_stream()
    # the oracle's own copy of the state, updated by the oracle alone
    o_master = [f32(t).copy() for t in B[0]]
    o_m = [f32(t).copy() for t in B[1]]
    o_v = [f32(t).copy() for t in B[2]]
    o_out = u16(B[3]).copy()
    o_st = ora.scaler_init(ohp)
    try:
        for call in range(3):
            sc_a = flat.scaler_state()
            assert sc_a.as_tuple() == state.as_tuple() == o_st.as_tuple()
            _gen(case, grads, S, call, sc_a.scale)
            g_host = host_grads(grads)
            before_b = [f32(t).copy() for t in B[0]], u16(B[3]).copy()
            ra = flat.step(case["ranks"], grads, A[0], A[1], A[2], A[3],
                           grad_rank_offset_mul=mul)
            rb = Z.zero_shard_step_noalloc(
                case["full"], case["N"], gdt, case["dtype"], case["op"], hp, state,
                case["ranks"], grads.data_ptr(), ld, mul, [t.data_ptr() for t in B[0]],
                [t.data_ptr() for t in B[1]], [t.data_ptr() for t in B[2]], B[3].data_ptr(),
                0.0, stream.cuda_stream)
            scale_used = o_st.scale
            ro = ora.shard_step(ohp, o_st, case["N"], case["full"], S, case["ranks"], g_host,
                                ld, mul, o_master, o_m, o_v, o_out, avg=case["op"] == AVG,
                                grad_is_bf16=bf16, param_is_bf16=bf16)
            tag = " (call %d)" % call
            # the handle step: same kernels, same bytes -> the same bits
            assert (rb.overflow, rb.skipped, rb.grad_norm, rb.clip_coef, rb.scale_used) == \
                   (ra.overflow, ra.skipped, ra.grad_norm, ra.clip_coef, ra.scale_used), tag
            assert flat.scaler_state().as_tuple() == state.as_tuple(), tag
            for j in range(len(case["ranks"])):
                for x, y in zip((B[0][j], B[1][j], B[2][j]), (A[0][j], A[1][j], A[2][j])):
                    assert _same_bits(f32(x), f32(y)), "state differs from the handle step" + tag
            assert _same_bits(u16(B[3]), u16(A[3])), "flat buffer differs" + tag
            # the oracle
            assert_result(rb, (ro.overflow, ro.skipped, ro.grad_norm, ro.clip_coef, scale_used))
            assert state.as_tuple() == o_st.as_tuple(), tag
            for j in range(len(case["ranks"])):
                assert_state(f32(B[0][j]), f32(B[1][j]), f32(B[2][j]),
                             o_master[j], o_m[j], o_v[j], tag=tag)
            assert_params_close(u16(B[3]), o_out, bf16, "flat params" + tag)
            # the planted inf: skipped, nothing written, dynamic scale halved
            if call == INF_CALL:
                assert (rb.overflow, rb.skipped) == (1, 1)
                for j in range(len(case["ranks"])):
                    assert _same_bits(f32(B[0][j]), before_b[0][j])
                assert _same_bits(u16(B[3]), before_b[1])
                assert state.scale == (scale_used / 2 if case["dynamic"] else scale_used)
            else:
                assert (rb.overflow, rb.skipped) == (0, 0)
        assert state.step_t == 2 and state.overflow_count == 1
    finally:
        flat.close()


def test_noalloc_refuses_shards_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import fsdp_sharded_mixed_zero_gb300 as Z
    full, N = 80_000_000, 8                     # one shard of 1e7 params > ~8.3M floats
    S = full // N
    state = Z.ScalerState(65536.0, 0, 0, 0)
    g = torch.zeros((N, 16), dtype=torch.float16, device="cuda")   # never read
    t = torch.zeros(16, device="cuda")
    o = torch.zeros(16, dtype=torch.float16, device="cuda")
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_shard_step_noalloc(full, N, F16, F16, AVG, Z.hparams(), state, [3],
                                  g.data_ptr(), S, 0, [t.data_ptr()], [t.data_ptr()],
                                  [t.data_ptr()], o.data_ptr())
    assert e.value.status == 1
    assert "static scratch" in Z.zero_last_error()
    assert state.as_tuple() == (65536.0, 0, 0, 0)           # untouched
