"""Group steps (zero_group_step): the FlatParameters of one rank -- one
handle each, different shapes, layouts and shard sizes -- stepped with one
clip norm and one loss-scale decision in one reduce launch and one AdamW
launch per 64 (member, rank) rows.  Compared with the oracle's single global
decision over all members (exact norm of the union, one ora_scaler_decide,
AdamW per member), a one-member group with zero_shard_step bit for bit, and
the launch count checked with the CUDA profiler."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth.workloads import AVG, BF16, F16, F32, SUM, Workload  # noqa: E402

import tests.oracle_runner as runner  # noqa: E402
from tests.gpu_helpers import (NORM_RTOL, assert_params_close, assert_state, f32,  # noqa: E402
                               host_grads, u16)

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _wl(name, shapes, N, ranks, layout="full", inf_at=None, seed=1, steps=3, hp=None,
        dtype=F16, op=AVG, dynamic=True):
    return Workload(name=name, description=name, shapes=shapes, world_size=N, ranks=ranks,
                    grad_dtype=dtype, op=op, dynamic=dynamic, steps=steps, sigma_g=1e-3,
                    sigma_n=1e-3, inf_at=inf_at, grads_layout=layout, seed=seed, hp=hp or {})


def _args(w, d):
    return dict(ranks=w.ranks, grads=d.grads, master=d.master, m=d.m, v=d.v, out=d.out,
                grad_rank_offset_mul=w.grad_rank_mul)


def _decode(u):
    return u.view(np.float16).astype(np.float32)


def run_group_parity(ora, ws, steps=3, lr_at=None, q8=False, q8_only=()):
    """Step the members ws as one group on the GPU and in the oracle, each
    member with its own parameter group's lr and weight decay; lr_at: {step:
    lr} set on the whole group before that step.  q8: zero_group_step_q8, the
    int8 payload checked bit for bit against the oracle's quantizer of every
    member's parameters; members in q8_only pass no 16-bit output."""
    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    kws = [dict(w.hparams_kwargs()) for w in ws]
    hp = ora.hparams(**kws[0])
    ds = [DeviceWorkload(w, out_fill=0x5A5A) for w in ws]
    group = Z.ZeroGroup([d.flat for d in ds])
    try:
        state = [([f32(t).copy() for t in d.master], [f32(t).copy() for t in d.m],
                  [f32(t).copy() for t in d.v], u16(d.out).copy()) for d in ds]
        st = ora.scaler_init(hp)
        skipped = []
        if q8:
            nbs = [-(-d.S // 256) for d in ds]
            q8s = [torch.full((d.padded,), 0x55, dtype=torch.int8, device="cuda") for d in ds]
            scs = [torch.full((w.world_size * nb,), -1.0, device="cuda")
                   for w, nb in zip(ws, nbs)]
            want_q = [np.full(d.padded, 0x55, np.int8) for d in ds]
            want_s = [np.full(w.world_size * nb, -1.0, np.float32) for w, nb in zip(ws, nbs)]
        for step in range(steps):
            if lr_at and step in lr_at:
                group.set_lr(lr_at[step])
                for kw in kws:
                    kw["lr"] = lr_at[step]
            hps = [ora.hparams(**kw) for kw in kws]
            assert group.scaler_state().as_tuple() == st.as_tuple()
            scale = st.scale
            grads = []
            for d in ds:
                d.gen_grads(step, scale)
                grads.append(host_grads(d.grads))
            if q8:
                margs = [_args(w, d) for w, d in zip(ws, ds)]
                for k, a in enumerate(margs):
                    a.update(q8=q8s[k], q8_scales=scs[k])
                    if k in q8_only:
                        a["out"] = None
                res = group.step_q8(margs)
            else:
                res = group.step([_args(w, d) for w, d in zip(ws, ds)])
            gs = []
            for w, d, g in zip(ws, ds, grads):
                for r in w.ranks:
                    x = np.empty(max(d.S, 1), np.float32)[:d.S]
                    runner.reduce_rank(g, w.grad_ld, r * w.grad_rank_mul, w.world_size, d.S,
                                       r * d.S, d.full, w.op == AVG, scale,
                                       w.grad_dtype == BF16, x)
                    gs.append(x)
            acc, of = runner.norm_exact(gs)
            norm = float(np.sqrt(ora.norm_sum(acc)))
            coef, skip = ora.scaler_decide(hp, st, of, norm)
            assert (res.overflow, res.skipped, res.scale_used) == (of, skip, scale)
            if not of:
                assert abs(res.grad_norm - norm) <= NORM_RTOL * norm
                assert abs(res.clip_coef - coef) <= NORM_RTOL * coef
            k = 0
            for w, d, hpk, (master, m, v, out) in zip(ws, ds, hps, state):
                for j, r in enumerate(w.ranks):
                    if not skip:
                        ora.adamw_cast(hpk, st.step_t, coef, gs[k], master[j], m[j], v[j],
                                       param_is_bf16=w.param_dtype == BF16,
                                       out=out[r * d.S:(r + 1) * d.S])
                    k += 1
                    assert_state(f32(d.master[j]), f32(d.m[j]), f32(d.v[j]), master[j], m[j],
                                 v[j], tag=" (%s, step %d, rank %d)" % (w.name, step, r))
                if q8 and ws.index(w) in q8_only:
                    assert bool((d.out.view(torch.int16) == 0x5A5A).all())
                else:
                    assert_params_close(u16(d.out), out, w.param_dtype == BF16,
                                        "%s params (step %d)" % (w.name, step))
            if q8:
                for i, (w, d, (_, _, _, out)) in enumerate(zip(ws, ds, state)):
                    S, nb = d.S, nbs[i]
                    if not skip:
                        for r in w.ranks:
                            qq, ss = ora.quantize_q8(
                                np.ascontiguousarray(_decode(out[r * S:(r + 1) * S])), 256)
                            want_q[i][r * S:(r + 1) * S] = qq
                            want_s[i][r * nb:(r + 1) * nb] = ss
                    assert np.array_equal(q8s[i].cpu().numpy(), want_q[i]), \
                        "%s codes (step %d)" % (w.name, step)
                    assert np.array_equal(scs[i].cpu().numpy().view(np.uint32),
                                          want_s[i].view(np.uint32)), \
                        "%s scales (step %d)" % (w.name, step)
            skipped.append(skip)
        assert group.scaler_state().as_tuple() == st.as_tuple()
        return skipped
    finally:
        group.close()
        for d in ds:
            d.close()


def test_group_step_with_int8_payload(ora):
    """zero_group_step_q8: four members (one slice, one staged, one q8-only
    without the 16-bit output, one with its own rates), an overflow skipping
    every member and leaving every payload as it was."""
    _need_gpu()
    ws = [
        _wl("attn_all_shards", [(256, 768), (768,)], 8, list(range(8)), seed=51),
        _wl("mlp_slice_rank5", [(768, 3072), (3072,)], 8, [5], layout="slice", seed=52,
            inf_at=(1, 6, 1000)),
        _wl("odd_all_shards", [(80_001,)], 8, list(range(8)), seed=53),
        _wl("norms_q8_only", [(768,), (768,), (777,)], 8, [0, 3, 7], seed=54,
            hp=dict(lr=1e-4, weight_decay=0.0)),
    ]
    assert run_group_parity(ora, ws, q8=True, q8_only=(3,)) == [0, 1, 0]


@pytest.mark.parametrize("dtype,op,dynamic", [(BF16, SUM, False), (F32, AVG, True)],
                         ids=["bf16_sum_static", "fp32_contributions"])
def test_group_other_dtypes(ora, dtype, op, dynamic):
    """Groups whose members take bf16 contributions summed at a static scale
    (bf16 parameters), or fp32 contributions (fp16 parameters): one staged
    member (rows off 64 bytes), one slice, one all-shards; own rates in one."""
    _need_gpu()
    kw = dict(dtype=dtype, op=op, dynamic=dynamic)
    ws = [
        _wl("all_shards", [(512, 768), (768,)], 8, list(range(8)), seed=81, **kw),
        _wl("odd_rows", [(80_001,)], 8, list(range(8)), seed=82, **kw),
        _wl("slice_rank4", [(768, 3072)], 8, [4], layout="slice", seed=83,
            hp=dict(lr=1e-4, weight_decay=0.0), **kw),
    ]
    assert run_group_parity(ora, ws) == [0, 0, 0]


def test_group_members_keep_their_own_rates(ora):
    """Parameter groups in one group: weights with decay, biases and norms
    without, a head with its own learning rate; then one learning rate set on
    the whole group (each member keeps its weight decay)."""
    _need_gpu()
    ws = [
        _wl("weights_decay", [(768, 3072)], 8, [1, 6], seed=41, steps=4,
            hp=dict(lr=3e-5, weight_decay=0.01)),
        _wl("bias_norm_no_decay", [(3072,), (768,), (768,)], 8, list(range(8)), seed=42,
            steps=4, hp=dict(lr=3e-5, weight_decay=0.0)),
        _wl("head_own_lr", [(80_032,)], 8, list(range(8)), seed=43, steps=4,
            hp=dict(lr=1e-3, weight_decay=0.1)),
    ]
    assert run_group_parity(ora, ws, steps=4, lr_at={2: 2e-5}) == [0, 0, 0, 0]


def test_group_of_four_flat_parameters(ora):
    _need_gpu()
    ws = [
        _wl("attn_all_shards", [(256, 768), (768,)], 8, list(range(8)), seed=21),
        _wl("mlp_slice_rank5", [(768, 3072), (3072,)], 8, [5], layout="slice", seed=22,
            inf_at=(1, 6, 1000)),
        _wl("odd_all_shards", [(80_001,)], 8, list(range(8)), seed=23),     # staged rows
        _wl("norm_small", [(768,), (768,)], 8, [0, 3], seed=24),            # below one tile
    ]
    assert run_group_parity(ora, ws) == [0, 1, 0]


def test_group_of_seventy_members_in_two_launches_each(ora):
    _need_gpu()
    ws = [_wl("m%02d" % k, [(2_000 + 37 * k,)], 4, [k % 4], layout="slice", seed=100 + k,
              steps=2) for k in range(70)]
    assert run_group_parity(ora, ws, steps=2) == [0, 0]
    # launch count: 70 rows -> 2 reduce launches and 2 AdamW launches
    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    from torch.profiler import ProfilerActivity, profile
    ds = [DeviceWorkload(w) for w in ws]
    group = Z.ZeroGroup([d.flat for d in ds])
    try:
        for d in ds:
            d.gen_grads(0, group.scaler_state().scale)
        args = [_args(w, d) for w, d in zip(ws, ds)]
        names = []
        for _ in range(2):                   # the profiler's first session may be empty
            with profile(activities=[ProfilerActivity.CUDA]) as prof:
                group.step(args, want_result=False)
                torch.cuda.synchronize()
            names = [e.name for e in prof.events() if "zg::" in e.name or "kernel" in e.name]
            if names:
                break
        if names:
            assert sum("reduce" in n for n in names) == 2, names
            assert sum("adamw" in n for n in names) == 2, names
    finally:
        group.close()
        for d in ds:
            d.close()


def test_one_member_group_equals_the_shard_step():
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = _wl("solo", [(300_007,)], 4, [0, 1, 2, 3], inf_at=(1, 3, 9), steps=4)
    a, b = DeviceWorkload(w), DeviceWorkload(w)
    group = Z.ZeroGroup([b.flat])
    try:
        for step in range(w.steps):
            a.gen_grads(step, a.scaler().scale)
            b.grads.copy_(a.grads)
            ra = a.step()
            rb = group.step([_args(w, b)])
            assert (ra.overflow, ra.skipped, ra.grad_norm, ra.clip_coef, ra.scale_used) == \
                   (rb.overflow, rb.skipped, rb.grad_norm, rb.clip_coef, rb.scale_used)
        for x, y in zip(a.master + a.m + a.v, b.master + b.m + b.v):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
        assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
        assert a.scaler().as_tuple() == group.scaler_state().as_tuple()
    finally:
        group.close()
        a.close()
        b.close()


def test_group_rejects_mismatched_members():
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    f4 = Z.ZeroFlat([(1000,)], 4)
    f8 = Z.ZeroFlat([(1000,)], 8)
    f4b = Z.ZeroFlat([(1000,)], 4, hp=Z.hparams(eps=1e-6))
    try:
        for members in ([f4, f8], [f4, f4b], [f4, f4]):     # world, eps, listed twice
            with pytest.raises(Z.ZeroError) as e:
                Z.ZeroGroup(members)
            assert e.value.status == 1
    finally:
        for f in (f4, f8, f4b):
            f.close()


def _wl_micro(name, shapes, N, ranks, micro, layout="full", inf_at=None, seed=1, steps=3,
              hp=None):
    w = _wl(name, shapes, N, ranks, layout=layout, inf_at=inf_at, seed=seed, steps=steps, hp=hp)
    w.micro_steps = micro
    return w


def run_group_accum_parity(ora, ws, micro, steps=3):
    """steps group steps of `micro` micro-steps each: zero_group_accumulate
    against the oracle's per-member accumulation (bit for bit), then
    zero_group_step_accumulated against one global decision over every
    member's g = acc / scale (padding zero)."""
    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    hps = [ora.hparams(**w.hparams_kwargs()) for w in ws]
    hp = hps[0]
    ds = [DeviceWorkload(w, out_fill=0x5A5A) for w in ws]
    for d in ds:
        d.alloc_acc()
    group = Z.ZeroGroup([d.flat for d in ds])
    try:
        state = [([f32(t).copy() for t in d.master], [f32(t).copy() for t in d.m],
                  [f32(t).copy() for t in d.v], u16(d.out).copy()) for d in ds]
        accs = [[np.zeros(d.S, np.float32) for _ in w.ranks] for w, d in zip(ws, ds)]
        st = ora.scaler_init(hp)
        skipped = []
        for step in range(steps):
            assert group.scaler_state().as_tuple() == st.as_tuple()
            scale = st.scale
            for k in range(micro):
                for w, d, acc in zip(ws, ds, accs):
                    d.gen_grads(step * micro + k, scale)
                    ora.grad_accumulate(w.world_size, d.full, d.S, w.ranks, host_grads(d.grads),
                                        w.grad_ld, w.grad_rank_mul, acc, first=(k == 0),
                                        avg=w.op == AVG)
                group.accumulate([dict(ranks=w.ranks, grads=d.grads, acc=d.acc,
                                       grad_rank_offset_mul=w.grad_rank_mul)
                                  for w, d in zip(ws, ds)], first_micro_step=(k == 0))
                for w, d, acc in zip(ws, ds, accs):
                    for j, r in enumerate(w.ranks):
                        got = f32(d.acc[j])
                        same = (got.view(np.uint32) == acc[j].view(np.uint32)) | \
                               (np.isnan(got) & np.isnan(acc[j]))
                        assert same.all(), "%s acc rank %d micro %d" % (w.name, r, k)
            res = group.step_accumulated([dict(ranks=w.ranks, acc=d.acc, master=d.master,
                                               m=d.m, v=d.v, out=d.out)
                                          for w, d in zip(ws, ds)])
            gs = []
            for w, d, acc in zip(ws, ds, accs):
                for j, r in enumerate(w.ranks):
                    g = acc[j] / np.float32(scale)
                    g[max(d.full - r * d.S, 0):] = 0.0
                    gs.append(g)
            nacc, of = runner.norm_exact(gs)
            norm = float(np.sqrt(ora.norm_sum(nacc)))
            coef, skip = ora.scaler_decide(hp, st, of, norm)
            assert (res.overflow, res.skipped, res.scale_used) == (of, skip, scale)
            if not of:
                assert abs(res.grad_norm - norm) <= NORM_RTOL * norm
                assert abs(res.clip_coef - coef) <= NORM_RTOL * coef
            k = 0
            for w, d, hpk, (master, m, v, out) in zip(ws, ds, hps, state):
                for j, r in enumerate(w.ranks):
                    if not skip:
                        ora.adamw_cast(hpk, st.step_t, coef, gs[k], master[j], m[j], v[j],
                                       param_is_bf16=w.param_dtype == BF16,
                                       out=out[r * d.S:(r + 1) * d.S])
                    k += 1
                    assert_state(f32(d.master[j]), f32(d.m[j]), f32(d.v[j]), master[j], m[j],
                                 v[j], tag=" (%s, step %d, rank %d)" % (w.name, step, r))
                assert_params_close(u16(d.out), out, False, "%s params (step %d)" % (w.name, step))
            skipped.append(skip)
        assert group.scaler_state().as_tuple() == st.as_tuple()
        return skipped
    finally:
        group.close()
        for d in ds:
            d.close()


def test_group_accumulation_staged_rows(ora):
    """Aligned accumulators, one member whose rows start off 64 bytes (the
    staged reduce), an overflow in micro-step 4 (step 1) of another member."""
    _need_gpu()
    ws = [
        _wl_micro("attn_all_shards", [(256, 768), (768,)], 8, list(range(8)), 3, seed=31),
        _wl_micro("odd_rows_all_shards", [(80_032,)], 8, list(range(8)), 3, seed=32),
        _wl_micro("mlp_slice_rank2", [(768, 3072)], 8, [2], 3, layout="slice", seed=33,
                  inf_at=(4, 2, 500), hp=dict(lr=1e-4, weight_decay=0.0)),
    ]
    assert run_group_accum_parity(ora, ws, micro=3) == [0, 1, 0]
    # the accumulate launch of this group is the staged reduce
    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    from torch.profiler import ProfilerActivity, profile
    ds = [DeviceWorkload(w) for w in ws]
    for d in ds:
        d.alloc_acc()
        d.gen_grads(0, 1.0)
    group = Z.ZeroGroup([d.flat for d in ds])
    try:
        args = [dict(ranks=w.ranks, grads=d.grads, acc=d.acc, grad_rank_offset_mul=w.grad_rank_mul)
                for w, d in zip(ws, ds)]
        names = []
        for _ in range(2):                   # the profiler's first session may be empty
            with profile(activities=[ProfilerActivity.CUDA]) as prof:
                group.accumulate(args, first_micro_step=True)
                torch.cuda.synchronize()
            names = [e.name for e in prof.events() if "kernel" in e.name]
            if names:
                break
        if names:
            assert any("reduce_staged_kernel" in n for n in names), names
    finally:
        group.close()
        for d in ds:
            d.close()


def test_group_accumulation_plain_rows_and_many_members(ora):
    """An odd shard size (accumulators off 16 bytes: the plain reduce for the
    whole group) and 70 members (two launches per call)."""
    _need_gpu()
    ws = [_wl_micro("m%02d" % k, [(1_001 + 37 * k,)], 4, [k % 4], 2, layout="slice",
                    seed=200 + k, steps=2) for k in range(69)]
    ws.append(_wl_micro("odd_s", [(4 * 2_501,)], 4, [0, 1, 2, 3], 2, seed=300, steps=2))
    assert run_group_accum_parity(ora, ws, micro=2, steps=2) == [0, 0]


@pytest.mark.parametrize("gpu_share", [0.0, 0.5, 1.0])
def test_group_offload_equals_group_step(gpu_share):
    """zero_group_step_offload (state in pinned host memory, the update split
    between the GPU and the host threads) against zero_group_step on twin
    handles: identical state, parameters and results every step, a skipped
    step included; members with their own rates and one misaligned (staged)."""
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    ws = [
        _wl("two_segments", [(8 * ((1 << 24) + 12_345),)], 8, [0], layout="slice", seed=61,
            steps=4, inf_at=(2, 3, 99)),
        _wl("mid_slice", [(3 * (1 << 20) + 12_345,)], 8, [2], layout="slice", seed=64, steps=4),
        _wl("odd_all", [(80_001,)], 8, list(range(8)), seed=62, steps=4,
            hp=dict(lr=1e-4, weight_decay=0.0)),
        _wl("small_two", [(5_000,), (77,)], 8, [0, 3], seed=63, steps=4),
    ]
    da = [DeviceWorkload(w) for w in ws]
    db = [DeviceWorkload(w) for w in ws]
    ga = Z.ZeroGroup([d.flat for d in da])
    gb = Z.ZeroGroup([d.flat for d in db])
    try:
        host = [[[t.detach().cpu().pin_memory() for t in getattr(d, name)]
                 for name in ("master", "m", "v")] for d in db]
        for step in range(4):
            for a, b in zip(da, db):
                a.gen_grads(step, ga.scaler_state().scale)
                b.grads.copy_(a.grads)
            ra = ga.step([_args(w, d) for w, d in zip(ws, da)])
            bargs = []
            for w, d, (hm, hmm, hv) in zip(ws, db, host):
                x = _args(w, d)
                x.update(master=hm, m=hmm, v=hv)
                bargs.append(x)
            rb = gb.step_offload(bargs, gpu_share=gpu_share)
            assert (ra.overflow, ra.skipped, ra.grad_norm, ra.clip_coef, ra.scale_used) == \
                   (rb.overflow, rb.skipped, rb.grad_norm, rb.clip_coef, rb.scale_used)
            assert rb.skipped == (step == 2)
        torch.cuda.synchronize()
        for a, b, (hm, hmm, hv) in zip(da, db, host):
            for x, y in zip(a.master + a.m + a.v, hm + hmm + hv):
                assert torch.equal(x.cpu().view(torch.int32), y.view(torch.int32))
            assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
        assert ga.scaler_state().as_tuple() == gb.scaler_state().as_tuple()
    finally:
        ga.close()
        gb.close()
        for d in da + db:
            d.close()


def test_group_argument_errors_name_the_member():
    """Every group entry point validates every member before launching: a bad
    argument of member 1 is refused with the member named, and nothing runs
    (the group's loss-scale state is unchanged)."""
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    ws = [_wl("a", [(4_000,)], 4, [0, 1, 2, 3], seed=71), _wl("b", [(1_000,)], 4, [1], seed=72,
                                                              layout="slice")]
    ds = [DeviceWorkload(w) for w in ws]
    for d in ds:
        d.alloc_acc()
        d.gen_grads(0, 65536.0)
    group = Z.ZeroGroup([d.flat for d in ds])
    try:
        before = group.scaler_state().as_tuple()

        q8s = [torch.zeros(d.padded, dtype=torch.int8, device="cuda") for d in ds]
        scs = [torch.zeros(4 * -(-d.S // 256), device="cuda") for d in ds]

        def refused(call, status, **bad):
            args = [_args(w, d) for w, d in zip(ws, ds)]
            for a, d, q, c in zip(args, ds, q8s, scs):
                a.update(acc=d.acc, q8=q, q8_scales=c)
            args[1].update(bad)
            with pytest.raises(Z.ZeroError) as e:
                call(args)
            assert e.value.status == status, str(e.value)
            assert "member 1" in str(e.value), str(e.value)

        bad_rank = dict(ranks=[4])                                  # rank >= world size
        refused(group.step, 1, **bad_rank)
        refused(lambda a: group.step_q8(a), 1, q8=None)             # no int8 outputs
        sc = torch.zeros(64, dtype=torch.uint8, device="cuda")
        refused(lambda a: group.step_q8(a), 3, q8_scales=sc[1:])    # misaligned scales
        refused(lambda a: group.accumulate(a, True), 1, **bad_rank)
        refused(lambda a: group.step_accumulated(a), 3,
                acc=[ds[1].acc[0].view(torch.uint8)[2:].view(torch.uint8)])  # misaligned acc
        refused(lambda a: group.step_offload(a), 1, **bad_rank)
        for bad in (-0.5, 2.0):
            with pytest.raises(Z.ZeroError) as e:
                group.step_offload([_args(w, d) for w, d in zip(ws, ds)], gpu_share=bad)
            assert e.value.status == 1
        torch.cuda.synchronize()
        assert group.scaler_state().as_tuple() == before
    finally:
        group.close()
        for d in ds:
            d.close()


def test_group_resume_from_saved_state():
    """Checkpoint a group mid-run (every member's master/m/v/flat buffer and
    the group's loss-scale state), build a new group over the same handles,
    restore, continue: the same bits as the uninterrupted group (the scale
    grows inside the window on the way)."""
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    hp = dict(initial_scale_power=5, window=2)
    ws = [_wl("r0", [(30_000,)], 4, [0, 1, 2, 3], seed=91, steps=6, hp=hp),
          _wl("r1", [(9_001,), (17,)], 4, [2], layout="slice", seed=92, steps=6,
              hp=dict(hp, weight_decay=0.0))]
    ds = [DeviceWorkload(w) for w in ws]

    def tensors():
        return [t for d in ds for t in d.master + d.m + d.v + [d.out]]

    group = Z.ZeroGroup([d.flat for d in ds])
    try:
        for step in range(3):
            for d in ds:
                d.gen_grads(step, group.scaler_state().scale)
            group.step([_args(w, d) for w, d in zip(ws, ds)])
        saved = [t.clone() for t in tensors()]
        saved_sc = group.scaler_state()
        runs = []
        for _ in range(2):
            group.close()
            group = Z.ZeroGroup([d.flat for d in ds])          # a new group object
            for t, x in zip(tensors(), saved):
                t.copy_(x)
            group.set_scaler_state(saved_sc)
            norms = []
            for step in range(3, 6):
                for d in ds:
                    d.gen_grads(step, group.scaler_state().scale)
                norms.append(group.step([_args(w, d) for w, d in zip(ws, ds)]).grad_norm)
            runs.append((norms, group.scaler_state().as_tuple(), [t.clone() for t in tensors()]))
        assert runs[0][0] == runs[1][0] and runs[0][1] == runs[1][1]
        assert runs[0][1][0] != saved_sc.scale                    # the scale moved
        for a, b in zip(runs[0][2], runs[1][2]):
            assert torch.equal(a.view(torch.int16) if a.element_size() == 2 else a,
                               b.view(torch.int16) if b.element_size() == 2 else b)
    finally:
        group.close()
        for d in ds:
            d.close()


def test_group_step_captured_in_a_cuda_graph_equals_eager():
    """A group step (staged and plain rows, per-member rates) captured once in
    a CUDA graph and replayed: the same bits and loss-scale state as the same
    group stepped eagerly on twin handles."""
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    ws = [_wl("g0", [(512, 1024), (1024,)], 4, [0, 1, 2, 3], seed=101),
          _wl("g1", [(40_001,)], 4, [0, 1, 2, 3], seed=102, hp=dict(weight_decay=0.0)),
          _wl("g2", [(3_000,)], 4, [3], layout="slice", seed=103)]
    da = [DeviceWorkload(w) for w in ws]
    db = [DeviceWorkload(w) for w in ws]
    ga = Z.ZeroGroup([d.flat for d in da])
    gb = Z.ZeroGroup([d.flat for d in db])
    try:
        for a, b in zip(da, db):
            a.gen_grads(0, ga.scaler_state().scale)
            b.grads.copy_(a.grads)
        args_a = [_args(w, d) for w, d in zip(ws, da)]
        args_b = [_args(w, d) for w, d in zip(ws, db)]
        # first step eagerly: the members' scratch and the group's partials are
        # allocated here, not during capture
        ga.step(args_a, want_result=False)
        gb.step(args_b, want_result=False)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            gb.step(args_b, stream=s, want_result=False)
        torch.cuda.current_stream().wait_stream(s)
        for _ in range(3):
            ga.step(args_a, want_result=False)
            graph.replay()
        torch.cuda.synchronize()
        assert ga.scaler_state().as_tuple() == gb.scaler_state().as_tuple()
        assert gb.scaler_state().step_t == 4
        for a, b in zip(da, db):
            for x, y in zip(a.master + a.m + a.v + [a.out], b.master + b.m + b.v + [b.out]):
                if x.element_size() == 2:
                    x, y = x.view(torch.int16), y.view(torch.int16)
                assert torch.equal(x, y)
    finally:
        ga.close()
        gb.close()
        for d in da + db:
            d.close()
