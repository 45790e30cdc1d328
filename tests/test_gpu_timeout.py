"""The staged reduce's bounded waits, made to run out without any fault:
through the test hook every stage of bulk copies expects more bytes than its
copies deliver, so the copies land but nothing completes the wait.  Each
block gives up after one second; the step must report ZERO_ERR_TIMEOUT, be
skipped (state, moments and parameters untouched) and counted as an overflow
by the loss-scale state machine; the device error word is cleared, and the
next step on the same handle must match the oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth.workloads import AVG, F16, Workload  # noqa: E402

import tests.oracle_runner as runner  # noqa: E402
from tests.gpu_helpers import (assert_params_close, assert_result, assert_state, f32,  # noqa: E402
                               host_grads, u16)

pytestmark = pytest.mark.gpu

ZERO_ERR_TIMEOUT = 6


def test_staged_wait_timeout_reports_skips_and_recovers(ora):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    # full layout, odd shard size: rank 1's slices are 2-byte aligned -> staged reduce
    w = Workload(name="timeout", description="timeout", shapes=[(2 * 10_001,)], world_size=2,
                 ranks=[0, 1], grad_dtype=F16, op=AVG, dynamic=True, steps=1, sigma_g=1e-3,
                 sigma_n=1e-3, grads_layout="full")
    hp = ora.hparams(**w.hparams_kwargs())
    dw = DeviceWorkload(w, out_fill=0x5A5A)
    try:
        master = [f32(t).copy() for t in dw.master]
        m = [f32(t).copy() for t in dw.m]
        v = [f32(t).copy() for t in dw.v]
        out = u16(dw.out).copy()
        st = ora.scaler_init(hp)
        scale0 = dw.scaler().scale
        dw.gen_grads(0, scale0)
        Z.zero_debug_set_stage_tx_pad(16)
        try:
            with pytest.raises(Z.ZeroError) as e:
                dw.step()
        finally:
            Z.zero_debug_set_stage_tx_pad(0)
        assert e.value.status == ZERO_ERR_TIMEOUT
        torch.cuda.synchronize()                       # the context is still usable
        for j in range(2):
            assert np.array_equal(f32(dw.master[j]).view(np.uint32), master[j].view(np.uint32))
            assert np.array_equal(f32(dw.m[j]), m[j]) and np.array_equal(f32(dw.v[j]), v[j])
        assert np.array_equal(u16(dw.out), out)
        sc = dw.scaler()
        assert (sc.scale, sc.good_steps, sc.step_t, sc.overflow_count) == (scale0 / 2, 0, 0, 1)
        # the oracle takes the same skip, then both run a normal step
        ora.scaler_decide(hp, st, 1, 0.0)
        assert dw.scaler().as_tuple() == st.as_tuple()
        dw.gen_grads(1, dw.scaler().scale)
        g = host_grads(dw.grads)
        res = dw.step()
        want = runner.shard_step(hp, st, w.world_size, dw.full, dw.S, w.ranks, g, w.grad_ld,
                                 w.grad_rank_mul, master, m, v, out, avg=True)
        assert_result(res, want)
        assert res.skipped == 0
        for j in range(2):
            assert_state(f32(dw.master[j]), f32(dw.m[j]), f32(dw.v[j]), master[j], m[j], v[j])
        assert_params_close(u16(dw.out), out, False, "flat params after recovery")
    finally:
        dw.close()
