"""The step split at its global decision (zero_shard_reduce, then
zero_shard_apply with device totals): bit-identical to zero_shard_step on one
handle; and for a group of FlatParameters (one handle each, different shapes,
world sizes and layouts) stepped with one clip norm and one loss-scale
decision -- the totals summed across the group on the device -- equal to the
oracle's single global decision over all of them, including an overflow in
one member that skips every member."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth.workloads import AVG, F16, F32, Workload  # noqa: E402

import tests.oracle_runner as runner  # noqa: E402
from tests.gpu_helpers import (NORM_RTOL, assert_params_close, assert_state, f32,  # noqa: E402
                               host_grads, u16)

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _wl(name, shapes, N, ranks, dtype=F16, steps=3, layout="full", inf_at=None, seed=1):
    return Workload(name=name, description=name, shapes=shapes, world_size=N, ranks=ranks,
                    grad_dtype=dtype, op=AVG, dynamic=True, steps=steps, sigma_g=1e-3,
                    sigma_n=1e-3, inf_at=inf_at, grads_layout=layout, seed=seed)


def _totals():
    return (torch.zeros((), dtype=torch.float64, device="cuda"),
            torch.zeros((), dtype=torch.int32, device="cuda"))


def test_split_equals_direct_step_bit_for_bit():
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = _wl("split_one", [(200_003,), (17,)], 4, [0, 1, 2, 3], steps=4, inf_at=(2, 1, 5))
    a, b = DeviceWorkload(w), DeviceWorkload(w)
    ss, of = _totals()
    try:
        for step in range(w.steps):
            a.gen_grads(step, a.scaler().scale)
            b.grads.copy_(a.grads)
            ra = a.step()
            b.flat.reduce(w.ranks, b.grads, ss, of, grad_rank_offset_mul=w.grad_rank_mul)
            rb = b.flat.apply(w.ranks, b.master, b.m, b.v, b.out, ss, of)
            assert (ra.overflow, ra.skipped, ra.grad_norm, ra.clip_coef, ra.scale_used) == \
                   (rb.overflow, rb.skipped, rb.grad_norm, rb.clip_coef, rb.scale_used)
        for x, y in zip(a.master + a.m + a.v, b.master + b.m + b.v):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
        assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
        assert a.scaler().as_tuple() == b.scaler().as_tuple()
    finally:
        a.close()
        b.close()


GROUP = [
    _wl("member_all_shards", [(512, 1024), (1024,), (1024, 512), (512,)], 4, [0, 1, 2, 3],
        seed=11),
    _wl("member_slice_rank3", [(300_001,)], 8, [3], layout="slice", inf_at=(1, 2, 77), seed=12),
    _wl("member_fp32_odd", [(50_001,), (7,)], 2, [0, 1], dtype=F32, seed=13),
]


def test_group_of_flat_parameters_takes_one_decision(ora):
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    hp = ora.hparams(**GROUP[0].hparams_kwargs())
    members = [DeviceWorkload(w, out_fill=0x5A5A) for w in GROUP]
    try:
        state = [([f32(t).copy() for t in d.master], [f32(t).copy() for t in d.m],
                  [f32(t).copy() for t in d.v], u16(d.out).copy()) for d in members]
        st = ora.scaler_init(hp)
        totals = [_totals() for _ in members]
        for step in range(3):
            for d in members:
                assert d.scaler().as_tuple() == st.as_tuple()
            scale = st.scale
            grads = []
            for w, d in zip(GROUP, members):
                d.gen_grads(step, scale)
                grads.append(host_grads(d.grads))
            for w, d, (ss, of) in zip(GROUP, members, totals):
                d.flat.reduce(w.ranks, d.grads, ss, of, grad_rank_offset_mul=w.grad_rank_mul)
            total_ss = torch.stack([t[0] for t in totals]).sum()       # the group's totals
            any_of = torch.stack([t[1] for t in totals]).max()
            results = [d.flat.apply(w.ranks, d.master, d.m, d.v, d.out, total_ss, any_of)
                       for w, d in zip(GROUP, members)]
            # the oracle: every member's reduced gradient, one exact norm, one decision
            gs = []
            for w, d, g in zip(GROUP, members, grads):
                for r in w.ranks:
                    x = np.empty(max(d.S, 1), np.float32)[:d.S]
                    runner.reduce_rank(g, w.grad_ld, r * w.grad_rank_mul, w.world_size, d.S,
                                       r * d.S, d.full, True, scale, False, x)
                    gs.append(x)
            acc, of = runner.norm_exact(gs)
            norm = float(np.sqrt(ora.norm_sum(acc)))
            coef, skip = ora.scaler_decide(hp, st, of, norm)
            for res in results:
                assert (res.overflow, res.skipped, res.scale_used) == (of, skip, scale)
                if not of:
                    assert abs(res.grad_norm - norm) <= NORM_RTOL * norm
                    assert abs(res.clip_coef - coef) <= NORM_RTOL * coef
            k = 0
            for w, d, (master, m, v, out) in zip(GROUP, members, state):
                for j, r in enumerate(w.ranks):
                    if not skip:
                        ora.adamw_cast(hp, st.step_t, coef, gs[k], master[j], m[j], v[j],
                                       out=out[r * d.S:(r + 1) * d.S])
                    k += 1
                    assert_state(f32(d.master[j]), f32(d.m[j]), f32(d.v[j]), master[j], m[j],
                                 v[j], tag=" (%s, step %d, rank %d)" % (w.name, step, r))
                assert_params_close(u16(d.out), out, False, "%s params (step %d)" % (w.name, step))
            assert skip == (step == 1)                   # member 2's inf skips every member
        for d in members:
            assert d.scaler().as_tuple() == st.as_tuple()
    finally:
        for d in members:
            d.close()


def test_split_misuse_is_refused():
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = _wl("misuse", [(40_000,)], 4, [0, 1, 2, 3], steps=1)
    d = DeviceWorkload(w)
    ss, of = _totals()
    try:
        d.gen_grads(0, d.scaler().scale)
        with pytest.raises(Z.ZeroError) as e:                     # no pending reduce
            d.flat.apply(w.ranks, d.master, d.m, d.v, d.out, ss, of)
        assert e.value.status == 1
        d.flat.reduce(w.ranks, d.grads, ss, of, grad_rank_offset_mul=w.grad_rank_mul)
        with pytest.raises(Z.ZeroError) as e:                     # other ranks
            d.flat.apply([0, 1], d.master[:2], d.m[:2], d.v[:2], d.out, ss, of)
        assert e.value.status == 1
        d.step()                                                  # a step in between
        with pytest.raises(Z.ZeroError) as e:
            d.flat.apply(w.ranks, d.master, d.m, d.v, d.out, ss, of)
        assert e.value.status == 1
        with pytest.raises(Z.ZeroError) as e:                     # misaligned total
            Z.zero_shard_reduce(d.flat.handle, w.ranks, d.grads.data_ptr(), d.grads.stride(0),
                                w.grad_rank_mul, ss.data_ptr() + 4, of.data_ptr())
        assert e.value.status == 3
    finally:
        d.close()


def test_apply_partials_totals_thousands_of_partials():
    """zero_shard_apply_partials with 5000 per-rank partials (the all-gathered
    form of the cross-rank exchange): the decision kernel's fixed-order fp64
    total matches the exactly rounded sum to ~1e-15, the clip coefficient
    follows from it, and one set flag among them skips the step."""
    _need_gpu()
    import math
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = _wl("partials", [(50_000,)], 1, [0], steps=1, layout="slice")
    dw = DeviceWorkload(w)
    ss, of = _totals()
    rng = np.random.default_rng(3)
    n = 5000
    parts = rng.random(n) * rng.choice([1e-6, 1e-3, 1.0], n)       # magnitudes far apart
    norm_sq = torch.from_numpy(parts).cuda()
    try:
        for overflow_at in (None, 4321):
            flags = torch.zeros(n, dtype=torch.int32, device="cuda")
            if overflow_at is not None:
                flags[overflow_at] = 1
            sc = dw.scaler()
            dw.gen_grads(0, sc.scale)
            dw.flat.reduce(w.ranks, dw.grads, ss, of, grad_rank_offset_mul=0)
            res = dw.flat.apply_partials(w.ranks, dw.master, dw.m, dw.v, dw.out, norm_sq, flags)
            if overflow_at is None:
                norm = math.sqrt(math.fsum(parts))
                assert (res.overflow, res.skipped) == (0, 0)
                assert abs(res.grad_norm - norm) <= 1e-14 * norm, (res.grad_norm, norm)
                coef = float(np.float32(1.0 / (norm + 1e-6)))
                assert abs(res.clip_coef - coef) <= NORM_RTOL * coef
            else:
                assert (res.overflow, res.skipped) == (1, 1)
                assert dw.scaler().scale == sc.scale / 2
    finally:
        dw.close()
