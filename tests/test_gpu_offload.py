"""GPU parity of the ZeRO-Offload step (zero_shard_step_offload): the reduce,
norm and decision on the GPU, AdamW on the host cores over fp32 state in host
memory, and the 16-bit parameters copied back into the device flat buffer.
Compared with the oracle element by element on every step (skip steps
included), and bit for bit with the all-GPU step on the same inputs."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth.workloads import AVG, BF16, F16, F32, SUM, Workload  # noqa: E402

import tests.oracle_runner as runner  # noqa: E402
from tests.gpu_helpers import (assert_params_close, assert_result, assert_state, f32,  # noqa: E402
                               host_grads, u16)

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _wl(name, shapes, N, ranks, dtype=F16, op=AVG, dynamic=True, steps=3, layout="full",
        inf_at=None):
    return Workload(name=name, description=name, shapes=shapes, world_size=N, ranks=ranks,
                    grad_dtype=dtype, op=op, dynamic=dynamic, steps=steps, sigma_g=1e-3,
                    sigma_n=1e-3, inf_at=inf_at, grads_layout=layout)


def _host_copies(ts, pin):
    out = []
    for t in ts:
        c = t.detach().cpu()
        out.append(c.pin_memory() if pin else c.clone())
    return out


CASES = [
    (_wl("tiny_inf_skip", [(512, 1024), (1024,), (1024, 512), (512,)], 4, [0, 1, 2, 3],
         steps=4, inf_at=(2, 1, 9)), True, 0, 0.5),
    (_wl("bf16_sum_ragged", [(40_001,), (33,)], 8, list(range(8)), dtype=BF16, op=SUM,
         dynamic=False), False, 3, 0.0),
    (_wl("slice_rank3", [(3_000_001,)], 8, [3], layout="slice"), True, 0, 0.4),
    (_wl("fp32_contrib", [(100_003,)], 2, [0, 1], dtype=F32), False, 1, 0.0),
    (_wl("n70_two_launches", [(70 * 33 + 5,)], 70, list(range(70)), steps=2), True, 0, 1.0),
    (_wl("multi_segment", [(2 * (1 << 24) + 12_345,)], 1, [0], steps=2), True, 0, 0.3),
    (_wl("gpu_only_pinned", [(1_000_003,)], 4, [0, 1, 2, 3], steps=3, inf_at=(1, 0, 5)),
     True, 0, 1.0),
]


@pytest.mark.parametrize("w,pin,n_threads,gpu_share", CASES, ids=[c[0].name for c in CASES])
def test_offload_step_matches_oracle(ora, w, pin, n_threads, gpu_share):
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    hp = ora.hparams(**w.hparams_kwargs())
    dw = DeviceWorkload(w, out_fill=0x5A5A)
    try:
        hm, hmm, hv = (_host_copies(x, pin) for x in (dw.master, dw.m, dw.v))
        master = [x.numpy().copy() for x in hm]
        m = [x.numpy().copy() for x in hmm]
        v = [x.numpy().copy() for x in hv]
        out = u16(dw.out).copy()
        st = ora.scaler_init(hp)
        pbf16 = w.param_dtype == BF16
        skipped = []
        for step in range(w.steps):
            sc = dw.scaler()
            assert sc.as_tuple() == st.as_tuple()
            dw.gen_grads(step, sc.scale)
            g = host_grads(dw.grads)
            before = u16(dw.out).copy()
            res = dw.flat.step_offload(w.ranks, dw.grads, hm, hmm, hv, dw.out,
                                       grad_rank_offset_mul=w.grad_rank_mul, n_threads=n_threads,
                                       gpu_share=gpu_share)
            want = runner.shard_step(hp, st, w.world_size, dw.full, dw.S, w.ranks, g, w.grad_ld,
                                     w.grad_rank_mul, master, m, v, out, avg=w.op == AVG,
                                     grad_is_bf16=w.grad_dtype == BF16, param_is_bf16=pbf16)
            assert_result(res, want)
            torch.cuda.synchronize()
            for j in range(len(w.ranks)):
                assert_state(hm[j].numpy(), hmm[j].numpy(), hv[j].numpy(), master[j], m[j], v[j],
                             tag=" (step %d, rank %d)" % (step, w.ranks[j]))
            assert_params_close(u16(dw.out), out, pbf16, "flat params (step %d)" % step)
            if res.skipped:
                assert np.array_equal(u16(dw.out), before), "a skipped step wrote params"
            skipped.append(res.skipped)
        assert dw.scaler().as_tuple() == st.as_tuple()
        if w.inf_at is not None:
            assert skipped[w.inf_at[0]] == 1
    finally:
        dw.close()


@pytest.mark.parametrize("gpu_share", [0.0, 0.3, 0.7, 1.0])
def test_offload_equals_device_step_bit_for_bit(gpu_share):
    """The same inputs through the all-GPU step and the offload step (two
    handles), for several splits of each shard between the GPU and the host
    threads: identical master, m, v, parameters and results."""
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = _wl("bits", [(1_000_007,), (99,)], 4, [0, 1, 2, 3], steps=3, inf_at=(1, 2, 5))
    a, b = DeviceWorkload(w), DeviceWorkload(w)
    try:
        hm, hmm, hv = (_host_copies(x, True) for x in (b.master, b.m, b.v))
        for step in range(w.steps):
            a.gen_grads(step, a.scaler().scale)
            b.grads.copy_(a.grads)
            ra = a.step()
            rb = b.flat.step_offload(w.ranks, b.grads, hm, hmm, hv, b.out,
                                     grad_rank_offset_mul=w.grad_rank_mul, gpu_share=gpu_share)
            assert (ra.overflow, ra.skipped, ra.grad_norm, ra.clip_coef, ra.scale_used) == \
                   (rb.overflow, rb.skipped, rb.grad_norm, rb.clip_coef, rb.scale_used)
        torch.cuda.synchronize()
        for x, y in zip(a.master + a.m + a.v, hm + hmm + hv):
            assert torch.equal(x.cpu().view(torch.int32), y.view(torch.int32))
        assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
        assert a.scaler().as_tuple() == b.scaler().as_tuple()
    finally:
        a.close()
        b.close()


def test_offload_argument_errors():
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    f = Z.ZeroFlat([(100,)], 4)
    g = torch.zeros((4, 100), dtype=torch.float16, device="cuda")
    host = torch.zeros(25)
    out = torch.zeros(100, dtype=torch.float16, device="cuda")
    p = [host.data_ptr()]
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_shard_step_offload(f.handle, [0], g.data_ptr(), 100, 0, p, p, p, out.data_ptr(),
                                  n_threads=-1)
    assert e.value.status == 1
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_shard_step_offload(f.handle, [0], g.data_ptr(), 100, 0, [host.data_ptr() + 2], p,
                                  p, out.data_ptr())
    assert e.value.status == 3
    with pytest.raises(Z.ZeroError):
        Z.zero_shard_step_offload(f.handle, [4], g.data_ptr(), 100, 0, p, p, p, out.data_ptr())
    for bad in (-0.1, 1.5, float("nan")):
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_shard_step_offload(f.handle, [0], g.data_ptr(), 100, 0, p, p, p,
                                      out.data_ptr(), gpu_share=bad)
        assert e.value.status == 1
    f.close()
