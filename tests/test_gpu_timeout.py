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


def test_accumulation_timeout_voids_the_next_step(ora):
    """A staged accumulation launch whose waits run out has no partials to
    carry an overflow; its error word must still void the step taken from the
    accumulators: that step reports ZERO_ERR_TIMEOUT, is skipped (state,
    moments and parameters untouched, the scale halved), and the next
    accumulation and step on the same handle match the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    # rank 1's contributor slices start 40 bytes into a 64-byte unit, the
    # accumulator rows are 16-byte aligned: the staged accumulate
    w = Workload(name="acc_timeout", description="acc_timeout", shapes=[(2 * 10_004,)],
                 world_size=2, ranks=[0, 1], grad_dtype=F16, op=AVG, dynamic=True, steps=1,
                 sigma_g=1e-3, sigma_n=1e-3, grads_layout="full")
    hp = ora.hparams(**w.hparams_kwargs())
    dw = DeviceWorkload(w, out_fill=0x5A5A)
    try:
        dw.alloc_acc()
        master = [f32(t).copy() for t in dw.master]
        m = [f32(t).copy() for t in dw.m]
        v = [f32(t).copy() for t in dw.v]
        out = u16(dw.out).copy()
        st = ora.scaler_init(hp)
        scale0 = dw.scaler().scale
        dw.gen_grads(0, scale0)
        Z.zero_debug_set_stage_tx_pad(16)
        try:
            dw.accumulate(first=True)
            torch.cuda.synchronize()
        finally:
            Z.zero_debug_set_stage_tx_pad(0)
        with pytest.raises(Z.ZeroError) as e:
            dw.step_accumulated()
        assert e.value.status == ZERO_ERR_TIMEOUT
        for j in range(2):
            assert np.array_equal(f32(dw.master[j]).view(np.uint32), master[j].view(np.uint32))
            assert np.array_equal(f32(dw.m[j]), m[j]) and np.array_equal(f32(dw.v[j]), v[j])
        assert np.array_equal(u16(dw.out), out)
        sc = dw.scaler()
        assert (sc.scale, sc.good_steps, sc.step_t, sc.overflow_count) == (scale0 / 2, 0, 0, 1)
        ora.scaler_decide(hp, st, 1, 0.0)
        # recovery: a clean accumulation and step, against the oracle
        dw.gen_grads(1, dw.scaler().scale)
        g = host_grads(dw.grads)
        dw.accumulate(first=True)
        acc = [np.zeros(dw.S, np.float32) for _ in w.ranks]
        ora.grad_accumulate(w.world_size, dw.full, dw.S, w.ranks, g, w.grad_ld, w.grad_rank_mul,
                            acc, first=True, avg=True)
        res = dw.step_accumulated()
        want = ora.shard_step_acc(hp, st, w.world_size, dw.full, dw.S, w.ranks, acc, master, m,
                                  v, out)
        assert_result(res, (want.overflow, want.skipped, want.grad_norm, want.clip_coef,
                            want.scale_used))
        assert res.skipped == 0
        for j in range(2):
            assert_state(f32(dw.master[j]), f32(dw.m[j]), f32(dw.v[j]), master[j], m[j], v[j])
        assert_params_close(u16(dw.out), out, False, "flat params after recovery")
    finally:
        dw.close()
