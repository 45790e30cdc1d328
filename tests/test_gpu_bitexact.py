"""Bit-exact elementwise parity: with the clip coefficient the GPU used
injected into the oracle (the decision still the oracle's), the updated fp32
master, m and v and the 16-bit flat slot must equal the oracle's bit for bit
-- every per-element operation is one IEEE fp32 operation on both sides, so
only the norm's summation order may differ, and that enters through the
coefficient alone.  The GPU's coefficient must also be within the norm
tolerance of the oracle's own.  Layouts: all shards fp16 with an overflow
step, bf16 SUM, fp32 contributions, a misaligned full layout (staged reduce,
re-aligned output stores) and one rank's slice."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth.workloads import AVG, BF16, F16, F32, SUM, Workload  # noqa: E402

import tests.oracle_runner as runner  # noqa: E402
from tests.gpu_helpers import NORM_RTOL, f32, host_grads, u16  # noqa: E402

pytestmark = pytest.mark.gpu


def _wl(name, numel, N, ranks, dtype=F16, op=AVG, dynamic=True, steps=3, layout="full",
        inf_at=None):
    return Workload(name=name, description=name, shapes=[(numel,)], world_size=N, ranks=ranks,
                    grad_dtype=dtype, op=op, dynamic=dynamic, steps=steps, sigma_g=1e-3,
                    sigma_n=1e-3, inf_at=inf_at, grads_layout=layout)


CASES = [
    _wl("f16_all_shards_inf", 4 * 250_000, 4, [0, 1, 2, 3], steps=4, inf_at=(1, 2, 11)),
    _wl("bf16_sum_static", 8 * 120_000 + 5, 8, list(range(8)), dtype=BF16, op=SUM, dynamic=False),
    _wl("f32_contributions", 2 * 300_000, 2, [0, 1], dtype=F32),
    _wl("f16_full_odd_shard", 8 * 100_001 - 1, 8, list(range(8))),
    _wl("f16_slice_rank6", 8 * 1_000_003, 8, [6], layout="slice"),
]


def _same32(a, b):
    return np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_update_is_bit_exact_given_the_coefficient(ora, w):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    hp = ora.hparams(**w.hparams_kwargs())
    dw = DeviceWorkload(w, out_fill=0x5A5A)
    try:
        master = [f32(t).copy() for t in dw.master]
        m = [f32(t).copy() for t in dw.m]
        v = [f32(t).copy() for t in dw.v]
        out = u16(dw.out).copy()
        st = ora.scaler_init(hp)
        applied = 0
        for step in range(w.steps):
            dw.gen_grads(step, dw.scaler().scale)
            g = host_grads(dw.grads)
            res = dw.step()
            of, skip, norm, coef, _ = runner.shard_step(
                hp, st, w.world_size, dw.full, dw.S, w.ranks, g, w.grad_ld, w.grad_rank_mul,
                master, m, v, out, avg=w.op == AVG, grad_is_bf16=w.grad_dtype == BF16,
                param_is_bf16=w.param_dtype == BF16, coef_override=res.clip_coef)
            assert (res.overflow, res.skipped) == (of, skip)
            if not skip:
                applied += 1
                assert abs(res.clip_coef - coef) <= NORM_RTOL * coef
            for j in range(len(w.ranks)):
                what = " (step %d, rank %d)" % (step, w.ranks[j])
                assert _same32(f32(dw.master[j]), master[j]), "master" + what
                assert _same32(f32(dw.m[j]), m[j]), "m" + what
                assert _same32(f32(dw.v[j]), v[j]), "v" + what
            assert np.array_equal(u16(dw.out), out), "flat params (step %d)" % step
        assert applied >= 1
    finally:
        dw.close()
