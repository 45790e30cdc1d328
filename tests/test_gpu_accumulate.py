"""GPU parity for fp32 (reduce_dtype=float32) contributions and for gradient
accumulation over micro-steps followed by the step from the accumulated fp32
shard: the CUDA path through the C ABI against the oracle, element by
element, including padding, an overflowing micro-step, several launches'
worth of ranks and unaligned accumulators."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth.workloads import AVG, BF16, F16, F32, SUM, Workload  # noqa: E402

import tests.oracle_runner as runner  # noqa: E402
from tests.gpu_helpers import (assert_params_close, assert_result, assert_state, f32,  # noqa: E402
                               host_grads, u16)
from tests.test_gpu_parity import run_parity  # noqa: E402

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _wl(name, shapes, N, ranks, dtype=F16, op=AVG, dynamic=True, steps=3, layout="full",
        micro=1, inf_at=None, hp=None):
    return Workload(name=name, description=name, shapes=shapes, world_size=N, ranks=ranks,
                    grad_dtype=dtype, op=op, dynamic=dynamic, steps=steps, sigma_g=1e-3,
                    sigma_n=1e-3, inf_at=inf_at, hp=hp or {}, grads_layout=layout,
                    micro_steps=micro)


# ------------------------------------------------------------ fp32 contributions

FP32 = [
    _wl("fp32_all_ragged", [(70_001,)], 4, [0, 1, 2, 3], dtype=F32, steps=4),
    _wl("fp32_slice_rank5", [(3_000_003,)], 8, [5], dtype=F32, layout="slice"),
    _wl("fp32_sum_static", [(20_000,), (17,)], 2, [0, 1], dtype=F32, op=SUM, dynamic=False),
]


@pytest.mark.parametrize("w", FP32, ids=lambda w: w.name)
def test_fp32_contributions(ora, w):
    run_parity(ora, w)


# ------------------------------------------------------------ accumulation

def run_accum_parity(ora, w):
    """w.steps optimizer steps of w.micro_steps micro-steps each."""
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    hp = ora.hparams(**w.hparams_kwargs())
    dw = DeviceWorkload(w, out_fill=0x5A5A)
    try:
        dw.alloc_acc()
        master = [f32(t).copy() for t in dw.master]
        m = [f32(t).copy() for t in dw.m]
        v = [f32(t).copy() for t in dw.v]
        out = u16(dw.out).copy()
        acc = [np.zeros(dw.S, np.float32) for _ in w.ranks]
        st = ora.scaler_init(hp)
        gbf16 = w.grad_dtype == BF16
        pbf16 = w.param_dtype == BF16
        skipped = []
        for step in range(w.steps):
            sc = dw.scaler()
            assert sc.as_tuple() == st.as_tuple()
            for k in range(w.micro_steps):
                micro = step * w.micro_steps + k
                dw.gen_grads(micro, sc.scale)
                g = host_grads(dw.grads)
                dw.accumulate(first=(k == 0))
                ora.grad_accumulate(w.world_size, dw.full, dw.S, w.ranks, g, w.grad_ld,
                                    w.grad_rank_mul, acc, first=(k == 0), avg=w.op == AVG,
                                    grad_is_bf16=gbf16)
                for j in range(len(w.ranks)):                # bit-exact accumulators
                    got = f32(dw.acc[j])
                    same = (got.view(np.uint32) == acc[j].view(np.uint32)) | \
                           (np.isnan(got) & np.isnan(acc[j]))
                    assert same.all(), "acc rank %d micro %d" % (w.ranks[j], micro)
            res = dw.step_accumulated()
            want = ora.shard_step_acc(hp, st, w.world_size, dw.full, dw.S, w.ranks, acc,
                                      master, m, v, out, param_is_bf16=pbf16)
            assert_result(res, (want.overflow, want.skipped, want.grad_norm, want.clip_coef,
                                want.scale_used))
            for j in range(len(w.ranks)):
                assert_state(f32(dw.master[j]), f32(dw.m[j]), f32(dw.v[j]), master[j], m[j],
                             v[j], tag=" (step %d, rank %d)" % (step, w.ranks[j]))
            assert_params_close(u16(dw.out), out, pbf16, "flat params (step %d)" % step)
            skipped.append(res.skipped)
        assert dw.scaler().as_tuple() == st.as_tuple()
        return skipped
    finally:
        dw.close()


ACCUM = [
    # 4 shards, 3 micro-steps, dynamic scale; micro-step 4 (step 1) overflows
    _wl("accum_tiny_inf", [(512, 1024), (1024,), (1024, 512), (512,)], 4, [0, 1, 2, 3],
        micro=3, steps=3, inf_at=(4, 2, 77)),
    # bf16 SUM, ragged shards with padding, 2 micro-steps
    _wl("accum_bf16_ragged", [(9_999,), (13,)], 8, list(range(8)), dtype=BF16, op=SUM,
        dynamic=False, micro=2, steps=3),
    # fp32 contributions, one rank of 8, 4 micro-steps
    _wl("accum_fp32_slice", [(2_000_000,)], 8, [6], dtype=F32, layout="slice", micro=4,
        steps=2),
    # more ranks than one launch takes
    _wl("accum_n70", [(70 * 33 + 1,)], 70, list(range(70)), micro=2, steps=2),
    # a static loss scale of 5: the norm pass and AdamW divide the accumulator
    # by a scale that is not a power of two (an IEEE division); rank slices
    # 8 bytes off 64-byte boundaries and 16-byte-aligned accumulator rows, so
    # the accumulation launches are staged
    _wl("accum_static_scale5", [(3 * 40_004 - 1,)], 3, [0, 1, 2], dynamic=False, micro=2,
        steps=2, hp=dict(static_scale=5.0)),
]


@pytest.mark.parametrize("w", ACCUM, ids=lambda w: w.name)
def test_accumulation_then_step(ora, w):
    skipped = run_accum_parity(ora, w)
    if w.inf_at is not None:
        assert skipped[w.inf_at[0] // w.micro_steps] == 1


def test_one_micro_step_equals_direct_step():
    """Accumulate once, step from the accumulator: the same bits as the direct
    step on the same contributions (two handles, same inputs).  The two norms
    are summed over different partitions (the direct step's odd shard takes
    the staged reduce, the accumulated step the plain norm pass), so they
    agree to ~1e-16 relative rather than bit for bit; the clip coefficient
    derived from them, and so every state bit, is the same."""
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = _wl("one_micro", [(100_003,)], 4, [0, 1, 2, 3], steps=2)
    a, b = DeviceWorkload(w), DeviceWorkload(w)
    b.alloc_acc()
    for step in range(2):
        a.gen_grads(step, a.scaler().scale)
        b.grads.copy_(a.grads)
        ra = a.step()
        b.accumulate(first=True)
        rb = b.step_accumulated()
        assert (ra.overflow, ra.skipped, ra.clip_coef) == (rb.overflow, rb.skipped, rb.clip_coef)
        assert abs(ra.grad_norm - rb.grad_norm) <= 1e-14 * ra.grad_norm
    for x, y in zip(a.master + a.m + a.v, b.master + b.m + b.v):
        assert torch.equal(x, y)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    a.close()
    b.close()


def test_unaligned_accumulators():
    """Accumulators that are only 4-byte aligned take the scalar paths and
    give the same bits."""
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    N, n = 4, 50_000
    f = Z.ZeroFlat([(n,)], N)
    S, P = f.shard_size, f.padded_numel
    g = torch.randn((N, P), device="cuda", generator=torch.Generator(device="cuda").manual_seed(3))
    g = (g * 100).to(torch.float16)
    buf_a = torch.zeros(N * S, device="cuda")
    buf_b = torch.zeros(N * S + 4, device="cuda")
    acc_a = [buf_a[r * S:(r + 1) * S] for r in range(N)]
    acc_b = [buf_b[1 + r * S:1 + (r + 1) * S] for r in range(N)]
    for first in (True, False, False):
        f.accumulate(list(range(N)), g, acc_a, first)
        f.accumulate(list(range(N)), g, acc_b, first)
    torch.cuda.synchronize()
    for x, y in zip(acc_a, acc_b):
        assert torch.equal(x, y)
    f.close()


def test_accumulate_argument_errors():
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    f = Z.ZeroFlat([(100,)], 4)
    g = torch.zeros((4, 100), dtype=torch.float16, device="cuda")
    acc = [torch.zeros(25, device="cuda")]
    with pytest.raises(Z.ZeroError):
        Z.zero_grad_accumulate(f.handle, [0], g.data_ptr(), 100, 0, [acc[0].data_ptr() + 2], True)
    with pytest.raises(Z.ZeroError):
        Z.zero_grad_accumulate(f.handle, [9], g.data_ptr(), 100, 0, [acc[0].data_ptr()], True)
    with pytest.raises(Z.ZeroError):
        Z.zero_shard_step_accumulated(f.handle, [0], [0], [acc[0].data_ptr()],
                                      [acc[0].data_ptr()], [acc[0].data_ptr()], g.data_ptr())
    f32_flat = Z.ZeroFlat([(100,)], 4, grad_dtype=Z.ZERO_F32)
    with pytest.raises(Z.ZeroError) as e:                 # fp32 contributions: 4-byte aligned
        Z.zero_shard_step(f32_flat.handle, [0], g.data_ptr() + 2, 100, 0, [acc[0].data_ptr()],
                          [acc[0].data_ptr()], [acc[0].data_ptr()], g.data_ptr())
    assert e.value.status == 3
    with pytest.raises(Z.ZeroError) as e:                 # parameters are never fp32
        Z.ZeroFlat([(100,)], 4, grad_dtype=Z.ZERO_F32, param_dtype=Z.ZERO_F32)
    assert e.value.status == 2
    f.close()
    f32_flat.close()


@pytest.mark.parametrize("scales", [(1e22, 1e-24, 1.0), (1e-24, 1e-24, 1e-24),
                                    (3e19, 3e19, 3e19), (1e-30, 1.0, 1e-30)])
def test_norm_extreme_magnitudes(ora, scales):
    """Squares that overflow or underflow fp32 while the values are finite:
    the norm (and so the clip) must still match the oracle's exact one."""
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    N, n = 2, 3 * 4096
    hp = Z.hparams(dynamic=False, lr=1e-3)
    f = Z.ZeroFlat([(n,)], N, grad_dtype=Z.ZERO_F32, hp=hp)
    S = f.shard_size
    rng = np.random.default_rng(31)
    g = rng.standard_normal((N, n)).astype(np.float64)
    for k, sc in enumerate(scales):
        g[:, k * 4096:(k + 1) * 4096] *= sc
    g = g.astype(np.float32)
    gd = torch.from_numpy(g).cuda()
    master = [torch.zeros(S, device="cuda") for _ in range(N)]
    m = [torch.zeros(S, device="cuda") for _ in range(N)]
    v = [torch.zeros(S, device="cuda") for _ in range(N)]
    out = torch.zeros(n, dtype=torch.float16, device="cuda")
    res = f.step([0, 1], gd, master, m, v, out)
    oh = ora.hparams(dynamic=False, lr=1e-3)
    st = ora.scaler_init(oh)
    hm = [np.zeros(S, np.float32) for _ in range(N)]
    hmm = [np.zeros(S, np.float32) for _ in range(N)]
    hv = [np.zeros(S, np.float32) for _ in range(N)]
    want = ora.shard_step(oh, st, N, n, S, [0, 1], g, n, S, hm, hmm, hv,
                          np.zeros(n, np.uint16), avg=True)
    assert res.overflow == want.overflow == 0
    assert abs(res.grad_norm - want.grad_norm) <= 1e-5 * want.grad_norm, \
        (res.grad_norm, want.grad_norm)
    assert abs(res.clip_coef - want.clip_coef) <= 1e-5 * want.clip_coef
    for j in range(N):
        assert_state(f32(master[j]), f32(m[j]), f32(v[j]), hm[j], hmm[j], hv[j])
    f.close()


def test_split_accumulated_step_equals_the_accumulated_step():
    """zero_shard_reduce_accumulated followed by zero_shard_apply (the split
    form a multi-rank caller uses) gives the bits of zero_shard_step_accumulated
    on the same accumulators -- ragged shard, four stepped ranks, an
    overflowing micro-step."""
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = _wl("split_acc", [(400_003,)], 4, [0, 1, 2, 3], steps=3, micro=2, inf_at=(2, 3, 11))
    a, b = DeviceWorkload(w), DeviceWorkload(w)
    a.alloc_acc()
    b.alloc_acc()
    ss = torch.zeros((), dtype=torch.float64, device="cuda")
    of = torch.zeros((), dtype=torch.int32, device="cuda")
    for step in range(w.steps):
        for k in range(2):
            a.gen_grads(2 * step + k, a.scaler().scale)
            b.grads.copy_(a.grads)
            a.accumulate(first=(k == 0))
            b.accumulate(first=(k == 0))
        ra = a.step_accumulated()
        b.flat.reduce_accumulated(w.ranks, b.acc, ss, of)
        rb = b.flat.apply(w.ranks, b.master, b.m, b.v, b.out, ss, of)
        assert (ra.overflow, ra.skipped, ra.clip_coef, ra.scale_used) == \
               (rb.overflow, rb.skipped, rb.clip_coef, rb.scale_used)
        if not ra.overflow:
            assert abs(ra.grad_norm - rb.grad_norm) <= 1e-14 * ra.grad_norm
        assert rb.skipped == (step == 1)
    for x, y in zip(a.master + a.m + a.v, b.master + b.m + b.v):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert a.scaler().as_tuple() == b.scaler().as_tuple()
    a.close()
    b.close()
