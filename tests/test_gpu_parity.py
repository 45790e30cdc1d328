"""GPU parity: the CUDA path (through the C ABI) against the oracle, element
by element, on the same seeded inputs: the three workloads the oracle finishes
in seconds at full size (tiny MLP, GPT-2 small, 1.5B rank 17 with an injected
inf), and the edge cases (ragged shards, padding, N=1, N=3 AVG division, more
stepped ranks than one launch takes, an empty FlatParameter, unaligned
pointers, misaligned output slots, determinism, resume)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth import workloads as W  # noqa: E402
from synth.workloads import AVG, BF16, F16, SUM, Workload  # noqa: E402

import tests.oracle_runner as runner  # noqa: E402
from tests.gpu_helpers import (assert_params_close, assert_result, assert_state, f32,  # noqa: E402
                               host_grads, u16)

pytestmark = pytest.mark.gpu

SENTINEL = 0x5A5A            # flat-buffer fill: slots not stepped must keep it


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def run_parity(ora, w, steps=None, out_fill=SENTINEL, extra_norm_sq=0.0):
    """Step workload w on the GPU and in the oracle; compare after every step."""
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    hp = ora.hparams(**w.hparams_kwargs())
    dw = DeviceWorkload(w, out_fill=out_fill)
    try:
        master = [f32(t).copy() for t in dw.master]
        m = [f32(t).copy() for t in dw.m]
        v = [f32(t).copy() for t in dw.v]
        out = u16(dw.out).copy()
        st = ora.scaler_init(hp)
        gbf16 = w.grad_dtype == BF16
        bf16 = w.param_dtype == BF16
        results = []
        for step in range(steps if steps is not None else w.warm_steps + w.steps):
            sc = dw.scaler()
            assert sc.as_tuple() == st.as_tuple(), (step, sc.as_tuple(), st.as_tuple())
            dw.gen_grads(step, sc.scale)
            g = host_grads(dw.grads)
            res = dw.step(extra_norm_sq=extra_norm_sq)
            want = runner.shard_step(hp, st, w.world_size, dw.full, dw.S, w.ranks, g,
                                     w.grad_ld, w.grad_rank_mul, master, m, v, out,
                                     avg=w.op == AVG, grad_is_bf16=gbf16, param_is_bf16=bf16,
                                     extra_norm_sq=extra_norm_sq)
            assert_result(res, want)
            for j in range(len(w.ranks)):
                assert_state(f32(dw.master[j]), f32(dw.m[j]), f32(dw.v[j]), master[j], m[j],
                             v[j], tag=" (step %d, rank %d)" % (step, w.ranks[j]))
            assert_params_close(u16(dw.out), out, bf16, "flat params (step %d)" % step)
            results.append((res.overflow, res.skipped, res.grad_norm, res.clip_coef))
        assert dw.scaler().as_tuple() == st.as_tuple()
        return results
    finally:
        dw.close()


# ------------------------------------------------------------ the workloads

def test_tiny_mlp_all_four_shards(ora):
    res = run_parity(ora, W.TINY)
    assert len(res) == 5 and not any(r[1] for r in res)


def test_gpt2_small_all_eight_shards_bf16_clipped(ora):
    res = run_parity(ora, W.GPT2)
    assert len(res) == 20
    assert all(r[3] < 1.0 for r in res), "clipping must be active (norm > 1)"


def test_1p5b_rank17_inf_skip_and_halve(ora):
    res = run_parity(ora, W.GPT_1P5B)
    assert [r[1] for r in res] == [0, 0, 0, 1, 0, 0, 0, 0, 0, 0]


# ------------------------------------------------------------ edge cases

def _wl(name, shapes, N, ranks, dtype=F16, op=AVG, dynamic=True, steps=4, layout="full",
        inf_at=None, hp=None, **kw):
    return Workload(name=name, description=name, shapes=shapes, world_size=N, ranks=ranks,
                    grad_dtype=dtype, op=op, dynamic=dynamic, steps=steps, sigma_g=1e-3,
                    sigma_n=1e-3, inf_at=inf_at, hp=hp or {}, grads_layout=layout, **kw)


EDGE = [
    # ragged shards (S=27), padding (3 elements), unaligned rows -> scalar paths,
    # misaligned output slots, a fast-growing dynamic scale and an overflow
    _wl("ragged", [(7, 13), (5,), (3, 3)], 4, [0, 1, 2, 3], steps=6, inf_at=(2, 1, 4),
        hp=dict(initial_scale_power=4, window=2)),
    # AVG over a world size that is not a power of two: true division
    _wl("avg_n3", [(1001,)], 3, [0, 1, 2], sigma_m=1e-5, sigma_v=1e-8),
    # more stepped ranks than one launch handles (64): two launches per kernel
    _wl("n70", [(70 * 41 - 5,)], 70, list(range(70)), steps=3),
    # one rank owns everything
    _wl("world1_bf16_sum", [(4096,), (100,)], 1, [0], dtype=BF16, op=SUM, dynamic=False),
    # vector path with a ragged tail on a single stepped rank of a slice layout
    _wl("slice_tail", [(8 * 50_000 * 3 + 7,)], 3, [1], layout="slice"),
    # many blocks, vector path, one stepped rank, misaligned slot (S odd)
    _wl("multi_block_odd_slot", [(3_000_001,)], 8, [3], layout="slice", steps=3),
    # clipping off, weight decay off
    _wl("no_clip_no_wd", [(9999,)], 2, [0, 1], hp=dict(max_grad_norm=0.0, weight_decay=0.0)),
    # every step overflows until the scale reaches its floor
    _wl("floor", [(4096,)], 2, [0, 1], steps=3, hp=dict(initial_scale_power=1, min_scale=1.0)),
    # a large world: 1000 contributions (AVG by true division) of a 38-element
    # shard; rank 973 holds 31 elements and 7 of padding, rank 999's slice is
    # all padding (full_numel = 37,005 < 999 * 38)
    _wl("n1000_tiny_shards", [(37_005,)], 1000, [0, 973, 999], steps=3, inf_at=(1, 640, 5)),
    # 256 contributions through the staged reduce: odd shard (4,097), rows
    # 8,208 bytes apart (16 bytes off a 64-byte boundary)
    _wl("n256_staged", [(256 * 4_097,)], 256, [201], layout="slice", steps=3),
    # a static loss scale that is not a power of two: the unscale is an IEEE
    # division (not an exact reciprocal multiply) after the AVG division by 3;
    # plain reduce (aligned rows) and staged reduce (odd shard) both
    _wl("static_scale5_n3_aligned", [(3 * 65_536,)], 3, [0, 1, 2], dynamic=False,
        hp=dict(static_scale=5.0)),
    _wl("static_scale5_n3_staged", [(3 * 30_001,)], 3, [0, 1, 2], dynamic=False,
        hp=dict(static_scale=5.0)),
]


@pytest.mark.parametrize("w", EDGE, ids=lambda w: w.name)
def test_edge_cases(ora, w):
    run_parity(ora, w)


def test_extra_norm_sq_from_other_ranks(ora):
    run_parity(ora, _wl("extra", [(50_000,)], 4, [2], layout="slice"), extra_norm_sq=0.37)


def test_empty_flat_parameter(ora):
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    f = Z.ZeroFlat([(0,)], 2, hp=Z.hparams())
    assert (f.full_numel, f.shard_size, f.padded_numel) == (0, 0, 0)
    t = torch.empty(8, dtype=torch.float32, device="cuda")
    g = torch.empty((2, 8), dtype=torch.float16, device="cuda")
    o = torch.empty(8, dtype=torch.float16, device="cuda")
    res = f.step([0, 1], g, [t, t], [t, t], [t, t], o)
    assert (res.overflow, res.skipped, res.grad_norm, res.clip_coef) == (0, 0, 0.0, 1.0)
    assert f.scaler_state().step_t == 1
    f.close()


def test_overflow_nan_skips(ora):
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    dw = DeviceWorkload(_wl("nan", [(5000,)], 2, [0, 1]))
    dw.gen_grads(0, dw.scaler().scale)
    dw.grads[1, 4321] = float("nan")
    before = [t.clone() for t in dw.master + dw.m + dw.v] + [dw.out.clone()]
    res = dw.step()
    assert res.overflow == 1 and res.skipped == 1
    for a, b in zip(before, dw.master + dw.m + dw.v + [dw.out]):
        assert torch.equal(a.view(torch.int16) if a.element_size() == 2 else a,
                           b.view(torch.int16) if b.element_size() == 2 else b)
    sc = dw.scaler()
    assert (sc.scale, sc.good_steps, sc.step_t, sc.overflow_count) == (32768.0, 0, 0, 1)
    dw.close()


def test_unaligned_pointers_match_aligned(ora):
    """Scalar paths (grads rows and master/m/v not 16-byte aligned) give the
    same bits as the vector paths."""
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    N, n = 4, 40_000
    f_a = Z.ZeroFlat([(n,)], N)
    f_b = Z.ZeroFlat([(n,)], N)
    S, P = f_a.shard_size, f_a.padded_numel
    gen = torch.Generator(device="cuda").manual_seed(0)
    gbuf = torch.empty((N * P + 16,), dtype=torch.float16, device="cuda")
    gbuf.normal_(0, 30.0, generator=gen)
    g_al = gbuf[:N * P].view(N, P)
    g_un = gbuf[1:1 + N * P].view(N, P)
    g_copy = g_un.clone()                           # aligned copy of the same values
    states = []
    for f, base_off in ((f_a, 0), (f_b, 1)):
        bufs = [torch.zeros(N * S + 8, dtype=torch.float32, device="cuda") for _ in range(3)]
        bufs[0][base_off:base_off + N * S].normal_(0, 0.02, generator=torch.Generator(
            device="cuda").manual_seed(1))
        views = [[b[base_off + r * S: base_off + (r + 1) * S] for r in range(N)] for b in bufs]
        out = torch.zeros(P, dtype=torch.float16, device="cuda")
        states.append((views, out))
    for _ in range(3):
        ra = f_a.step(list(range(N)), g_copy, *states[0][0], states[0][1])
        rb = f_b.step(list(range(N)), g_un, *states[1][0], states[1][1])
        assert (ra.overflow, ra.skipped, ra.grad_norm, ra.clip_coef) == \
               (rb.overflow, rb.skipped, rb.grad_norm, rb.clip_coef)
    for xa, xb in zip(sum(states[0][0], []), sum(states[1][0], [])):
        assert torch.equal(xa, xb)
    assert torch.equal(states[0][1].view(torch.int16), states[1][1].view(torch.int16))
    f_a.close()
    f_b.close()


def test_deterministic_bits(ora):
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    outs = []
    for _ in range(2):
        dw = DeviceWorkload(W.TINY)
        norms = []
        for step in range(3):
            dw.gen_grads(step, dw.scaler().scale)
            norms.append(dw.step().grad_norm)
        outs.append((norms, [t.clone() for t in dw.master + dw.m + dw.v], dw.out.clone()))
        dw.close()
    assert outs[0][0] == outs[1][0]
    for a, b in zip(outs[0][1], outs[1][1]):
        assert torch.equal(a, b)
    assert torch.equal(outs[0][2].view(torch.int16), outs[1][2].view(torch.int16))


def test_resume_from_saved_state(ora):
    """Checkpoint (master/m/v/flat buffer + loss-scale state), continue,
    restore, continue again: the same bits."""
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = _wl("resume", [(30_000,)], 2, [0, 1], steps=5, hp=dict(initial_scale_power=5, window=2))
    dw = DeviceWorkload(w)
    for step in range(3):
        dw.gen_grads(step, dw.scaler().scale)
        dw.step()
    saved = [t.clone() for t in dw.master + dw.m + dw.v + [dw.out]]
    saved_sc = dw.scaler()
    runs = []
    for _ in range(2):
        for t, s in zip(dw.master + dw.m + dw.v + [dw.out], saved):
            t.copy_(s)
        dw.flat.set_scaler_state(saved_sc)
        norms = []
        for step in range(3, 5):
            dw.gen_grads(step, dw.scaler().scale)
            norms.append(dw.step().grad_norm)
        runs.append((norms, dw.scaler().as_tuple(),
                     [t.clone() for t in dw.master + dw.m + dw.v + [dw.out]]))
    assert runs[0][0] == runs[1][0] and runs[0][1] == runs[1][1]
    for a, b in zip(runs[0][2], runs[1][2]):
        assert torch.equal(a.view(torch.int16) if a.element_size() == 2 else a,
                           b.view(torch.int16) if b.element_size() == 2 else b)
    dw.close()


def test_step_argument_errors(ora):
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    f = Z.ZeroFlat([(100,)], 4)
    S = f.shard_size
    g = torch.zeros((4, 100), dtype=torch.float16, device="cuda")
    t = [torch.zeros(S, device="cuda") for _ in range(4)]
    o = torch.zeros(100, dtype=torch.float16, device="cuda")
    with pytest.raises(Z.ZeroError) as e:
        f.step([0, 0], g, t[:2], t[:2], t[:2], o)     # duplicate rank
    assert e.value.status == 1
    with pytest.raises(Z.ZeroError):
        f.step([4], g, t[:1], t[:1], t[:1], o)         # rank out of range
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_shard_step(f.handle, [0], g.data_ptr() + 1, 100, 0, [t[0].data_ptr()],
                          [t[1].data_ptr()], [t[2].data_ptr()], o.data_ptr())
    assert e.value.status == 3                         # odd address
    with pytest.raises(Z.ZeroError):
        Z.zero_shard_step(f.handle, [0], g.data_ptr(), 10, 0, [t[0].data_ptr()],
                          [t[1].data_ptr()], [t[2].data_ptr()], o.data_ptr())  # ld < S
    with pytest.raises(Z.ZeroError):
        f.step([0], g, t[:1], t[:1], t[:1], o, extra_norm_sq=float("nan"))
    bad = Z.ScalerState(0.0, 0, 0, 0)
    with pytest.raises(Z.ZeroError):
        f.set_scaler_state(bad)
    assert f.scaler_state().step_t == 0                # nothing ran
    f.close()


def test_learning_rate_schedule(ora):
    """A warm-up then decay schedule set between steps (zero_flat_set_lr)
    matches the oracle stepping with the same rates."""
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = _wl("lr_sched", [(60_001,)], 4, [0, 1, 2, 3], steps=5)
    lrs = [1e-5, 2e-5, 3e-5, 1.5e-5, 0.0]
    dw = DeviceWorkload(w)
    try:
        master = [f32(t).copy() for t in dw.master]
        m = [f32(t).copy() for t in dw.m]
        v = [f32(t).copy() for t in dw.v]
        out = u16(dw.out).copy()
        kw = w.hparams_kwargs()
        st = ora.scaler_init(ora.hparams(**kw))
        for step, lr in enumerate(lrs):
            dw.flat.set_lr(lr)
            kw["lr"] = lr
            hp = ora.hparams(**kw)
            dw.gen_grads(step, dw.scaler().scale)
            g = host_grads(dw.grads)
            res = dw.step()
            want = runner.shard_step(hp, st, w.world_size, dw.full, dw.S, w.ranks, g, w.grad_ld,
                                     w.grad_rank_mul, master, m, v, out, avg=True)
            assert_result(res, want)
            for j in range(len(w.ranks)):
                assert_state(f32(dw.master[j]), f32(dw.m[j]), f32(dw.v[j]), master[j], m[j],
                             v[j], tag=" (lr %g)" % lr)
        import fsdp_sharded_mixed_zero_gb300 as Z
        with pytest.raises(Z.ZeroError):
            dw.flat.set_lr(float("nan"))
    finally:
        dw.close()
