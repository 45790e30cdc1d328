"""zero_shard_step_noalloc -- the shard step for callers that may not
allocate device memory (for instance code running under a framework whose
caching allocator owns all device memory, where zero_flat_init's cudaMalloc
is not allowed).  Two calls in a row through the C ABI must give what the
handle-based zero_shard_step gives on the same inputs, within the parity
tolerances of the other GPU tests; oversized shards must be refused with a
clear error.  This file is collected last on purpose and builds everything it
uses itself, so it passes alone or after the other tests."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import synth  # noqa: E402
from tests.gpu_helpers import (NORM_RTOL, assert_params_close, assert_state, f32,  # noqa: E402
                               u16)

pytestmark = pytest.mark.gpu

F16, BF16, SUM, AVG = 0, 1, 0, 1
CASES = [
    # all four shards of a ragged FlatParameter, fp16, AVG, dynamic loss scale
    dict(name="all_shards_fp16", full=300_001, N=4, ranks=[0, 1, 2, 3], dtype=F16, op=AVG,
         dynamic=True, layout="full"),
    # one rank's slice of an 8-way group, bf16, SUM, static scale
    dict(name="slice_bf16", full=2_000_000, N=8, ranks=[5], dtype=BF16, op=SUM,
         dynamic=False, layout="slice"),
]


def _setup(case, Z):
    N, full = case["N"], case["full"]
    S = -(-full // N)
    padded = S * N
    tdt = torch.float16 if case["dtype"] == F16 else torch.bfloat16
    ld = padded if case["layout"] == "full" else -(-S // 8) * 8
    grads = torch.empty((N, ld), dtype=tdt, device="cuda")
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
    dt = synth.F16 if case["dtype"] == F16 else synth.BF16
    if case["layout"] == "full":
        synth.grads_device(grads, 21, step, 0, grads.shape[1], 1e-3, 1e-3, scale, dt,
                           zero_from=case["full"])
    else:
        synth.grads_device(grads, 21, step, case["ranks"][0] * S, S, 1e-3, 1e-3, scale, dt,
                           zero_from=case["full"])


@pytest.mark.parametrize("case", CASES, ids=lambda c: c["name"])
def test_noalloc_matches_handle_step_two_calls(case):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import fsdp_sharded_mixed_zero_gb300 as Z
    hp = Z.hparams(dynamic=case["dynamic"], lr=1e-3)
    S, padded, ld, grads, (A, B) = _setup(case, Z)
    shapes = [(case["full"],)]
    flat = Z.ZeroFlat(shapes, case["N"], case["dtype"], case["dtype"], case["op"], hp)
    state = Z.ScalerState(65536.0 if case["dynamic"] else 1.0, 0, 0, 0)
    mul = S if case["layout"] == "full" else 0
    stream = torch.cuda.current_stream()
    try:
        for call in range(2):
            sc_a = flat.scaler_state()
            assert sc_a.as_tuple() == state.as_tuple()
            _gen(case, grads, S, call, sc_a.scale)
            ra = flat.step(case["ranks"], grads, A[0], A[1], A[2], A[3],
                           grad_rank_offset_mul=mul)
            rb = Z.zero_shard_step_noalloc(
                case["full"], case["N"], case["dtype"], case["dtype"], case["op"], hp, state,
                case["ranks"], grads.data_ptr(), ld, mul, [t.data_ptr() for t in B[0]],
                [t.data_ptr() for t in B[1]], [t.data_ptr() for t in B[2]], B[3].data_ptr(),
                0.0, stream.cuda_stream)
            assert (rb.overflow, rb.skipped, rb.scale_used) == \
                   (ra.overflow, ra.skipped, ra.scale_used)
            assert abs(rb.grad_norm - ra.grad_norm) <= NORM_RTOL * ra.grad_norm
            assert abs(rb.clip_coef - ra.clip_coef) <= NORM_RTOL * ra.clip_coef
            assert flat.scaler_state().as_tuple() == state.as_tuple()
            for j in range(len(case["ranks"])):
                assert_state(f32(B[0][j]), f32(B[1][j]), f32(B[2][j]),
                             f32(A[0][j]), f32(A[1][j]), f32(A[2][j]),
                             tag=" (call %d, rank %d)" % (call, case["ranks"][j]))
            assert_params_close(u16(B[3]), u16(A[3]), case["dtype"] == BF16,
                                "flat params (call %d)" % call)
        assert state.step_t == 2
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
