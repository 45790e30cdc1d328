"""The threaded composition of the oracle's pieces equals ora_shard_step bit
for bit (so large GPU parity runs may use it)."""
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
