"""The threaded composition of the oracle's pieces equals ora_shard_step
(and ora_shard_step_acc) bit for bit, so large GPU parity runs may use it."""
import numpy as np
import pytest

import tests.oracle_runner as runner


@pytest.mark.parametrize("N,n,bf16,avg,ranks", [
    (4, 3_000_001, False, True, [0, 1, 2, 3]),
    (3, 1_000_003, True, False, [1]),
    (8, 5_000_000, False, True, [2, 5]),
])
def test_threaded_matches_shard_step(ora, monkeypatch, N, n, bf16, avg, ranks):
    monkeypatch.setattr(runner, "CHUNK", 1 << 18)
    rng = np.random.default_rng(n)
    full, S, padded = ora.layout([n], N)
    hp = ora.hparams(lr=1e-3, max_grad_norm=1.0, dynamic=not bf16, window=2,
                     initial_scale_power=4)
    sa, sb = ora.scaler_init(hp), ora.scaler_init(hp)
    th = [(rng.standard_normal(S) * 0.02).astype(np.float32) for _ in ranks]
    ma = [t.copy() for t in th]
    mb = [t.copy() for t in th]
    m_a = [np.zeros(S, np.float32) for _ in ranks]
    m_b = [np.zeros(S, np.float32) for _ in ranks]
    v_a = [np.zeros(S, np.float32) for _ in ranks]
    v_b = [np.zeros(S, np.float32) for _ in ranks]
    oa = np.zeros(padded, np.uint16)
    ob = np.zeros(padded, np.uint16)
    for step in range(3):
        g = (rng.standard_normal((N, padded)) * 16).astype(np.float16).view(np.uint16)
        if step == 1:
            g[N - 1, ranks[0] * S + 7] = 0x7C00
        ra = ora.shard_step(hp, sa, N, full, S, ranks, g, padded, S, ma, m_a, v_a, oa,
                            avg=avg, grad_is_bf16=bf16, param_is_bf16=bf16, extra_norm_sq=0.25)
        rb = runner.shard_step(hp, sb, N, full, S, ranks, g, padded, S, mb, m_b, v_b, ob,
                               avg=avg, grad_is_bf16=bf16, param_is_bf16=bf16,
                               extra_norm_sq=0.25)
        assert (ra.overflow, ra.skipped, ra.grad_norm, ra.clip_coef, ra.scale_used) == rb
        assert sa.as_tuple() == sb.as_tuple()
        for x, y in zip(ma + m_a + v_a + [oa], mb + m_b + v_b + [ob]):
            assert np.array_equal(x, y)


def test_group_composition_equals_the_concatenated_step(ora):
    """The composition the group parity tests use -- each member's reduced
    gradient, one exact norm over all members, one decision, AdamW per
    member -- equals the oracle's own step over the members' concatenation
    (one FlatParameter, N=1: no padding, the same elements in the same
    places), bit for bit, overflow step included."""
    rng = np.random.default_rng(7)
    sizes = [1_003, 40_000, 7]
    total = sum(sizes)
    hp = ora.hparams(lr=1e-3, max_grad_norm=1.0, window=2, initial_scale_power=4)
    st_cat, st_grp = ora.scaler_init(hp), ora.scaler_init(hp)
    theta = (rng.standard_normal(total) * 0.02).astype(np.float32)
    cat = [theta.copy(), np.zeros(total, np.float32), np.zeros(total, np.float32)]
    out_cat = np.zeros(total, np.uint16)
    offs = np.cumsum([0] + sizes)
    grp = [[theta[a:b].copy(), np.zeros(b - a, np.float32), np.zeros(b - a, np.float32)]
           for a, b in zip(offs[:-1], offs[1:])]
    out_grp = [np.zeros(n, np.uint16) for n in sizes]
    for step in range(4):
        g = (rng.standard_normal((1, total)) * 8).astype(np.float16).view(np.uint16)
        if step == 2:
            g[0, offs[1] + 5] = 0x7C00                    # +inf in member 1
        r = ora.shard_step(hp, st_cat, 1, total, total, [0], g, total, 0, [cat[0]], [cat[1]],
                           [cat[2]], out_cat)
        scale = st_grp.scale
        gs = []
        for k, (a, b) in enumerate(zip(offs[:-1], offs[1:])):
            x = np.empty(b - a, np.float32)
            member = np.ascontiguousarray(g[:, a:b])
            runner.reduce_rank(member, b - a, 0, 1, b - a, 0, b - a, True, scale, False, x)
            gs.append(x)
        acc, of = runner.norm_exact(gs)
        norm = float(np.sqrt(ora.norm_sum(acc)))
        coef, skip = ora.scaler_decide(hp, st_grp, of, norm)
        if not skip:
            for k, x in enumerate(gs):
                ora.adamw_cast(hp, st_grp.step_t, coef, x, grp[k][0], grp[k][1], grp[k][2],
                               out=out_grp[k])
        assert (r.overflow, r.skipped, r.clip_coef) == (of, skip, coef)
        if not of:
            assert r.grad_norm == norm
        assert st_cat.as_tuple() == st_grp.as_tuple()
        for i in range(3):
            assert np.array_equal(cat[i], np.concatenate([m[i] for m in grp]))
        assert np.array_equal(out_cat, np.concatenate(out_grp))
    assert st_cat.overflow_count == 1


@pytest.mark.parametrize("N,n,ranks", [(4, 2_000_003, [0, 3]), (8, 1_000_000, [5])])
def test_threaded_matches_shard_step_acc(ora, monkeypatch, N, n, ranks):
    monkeypatch.setattr(runner, "CHUNK", 1 << 18)
    rng = np.random.default_rng(n + 1)
    full, S, padded = ora.layout([n], N)
    hp = ora.hparams(lr=1e-3, max_grad_norm=1.0, window=2, initial_scale_power=4)
    sa, sb = ora.scaler_init(hp), ora.scaler_init(hp)
    th = [(rng.standard_normal(S) * 0.02).astype(np.float32) for _ in ranks]
    st_a = [[t.copy() for t in th], [np.zeros(S, np.float32) for _ in ranks],
            [np.zeros(S, np.float32) for _ in ranks]]
    st_b = [[t.copy() for t in th], [np.zeros(S, np.float32) for _ in ranks],
            [np.zeros(S, np.float32) for _ in ranks]]
    oa = np.zeros(padded, np.uint16)
    ob = np.zeros(padded, np.uint16)
    for step in range(3):
        # accumulators as the accumulation leaves them: garbage in the padding
        # (the step must ignore it), an inf at step 1
        acc = [(rng.standard_normal(S) * 64).astype(np.float32) for _ in ranks]
        if step == 1:
            acc[-1][3] = np.inf
        ra = ora.shard_step_acc(hp, sa, N, full, S, ranks, acc, *st_a, oa, extra_norm_sq=0.5)
        rb = runner.shard_step_acc(hp, sb, N, full, S, ranks, acc, *st_b, ob, extra_norm_sq=0.5)
        assert (ra.overflow, ra.skipped, ra.grad_norm, ra.clip_coef, ra.scale_used) == rb
        assert sa.as_tuple() == sb.as_tuple()
        for x, y in zip(st_a[0] + st_a[1] + st_a[2] + [oa], st_b[0] + st_b[1] + st_b[2] + [ob]):
            assert np.array_equal(x, y)
    assert sa.overflow_count == 1


def test_unscale_acc_pads_with_zero(ora):
    acc = np.array([2.0, -6.0, 1.0, 5.0], np.float32)
    g = ora.unscale_acc(acc, 10, 12, 4.0)             # flat indices 10..13, full_numel 12
    assert g.tolist() == [0.5, -1.5, 0.0, 0.0]
