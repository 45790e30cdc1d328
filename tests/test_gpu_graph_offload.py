"""Three ways of running the same step: captured in a CUDA graph and
replayed (launch-bound small shards), with the fp32 master/m/v resident in
pinned host memory (optimizer state offloaded to the host, read and written
by the GPU kernels over the host link), and with bf16 gradients but fp16
parameters.  Each must give the bits of the plain device step, or the
oracle's."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth import workloads as W  # noqa: E402
from synth.workloads import AVG, BF16, F16, Workload  # noqa: E402

from tests.test_gpu_parity import run_parity  # noqa: E402

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _same(a, b):
    for x, y in zip(a, b):
        if x.element_size() == 2:
            x, y = x.view(torch.int16), y.view(torch.int16)
        assert torch.equal(x.cpu(), y.cpu())


def test_cuda_graph_replay_equals_eager():
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = W.TINY
    eager, graphed = DeviceWorkload(w), DeviceWorkload(w)
    steps = 4
    eager.gen_grads(0, eager.scaler().scale)
    graphed.grads.copy_(eager.grads)
    # first step eagerly: the handle allocates its scratch here, not during capture
    eager.step(want_result=False)
    graphed.step(want_result=False)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        graphed.step(want_result=False, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(steps - 1):
        eager.step(want_result=False)
        g.replay()
    torch.cuda.synchronize()
    assert eager.scaler().as_tuple() == graphed.scaler().as_tuple()
    assert graphed.scaler().step_t == steps
    _same(eager.master + eager.m + eager.v + [eager.out],
          graphed.master + graphed.m + graphed.v + [graphed.out])
    eager.close()
    graphed.close()


def test_optimizer_state_in_pinned_host_memory():
    """master/m/v in page-locked host memory: the kernels stream them over the
    host link; the bits equal those of device-resident state."""
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = Workload(name="offload", description="offload", shapes=[(1_000_003,)], world_size=4,
                 ranks=[0, 1, 2, 3], grad_dtype=F16, op=AVG, dynamic=True, steps=3,
                 sigma_g=1e-3, sigma_n=1e-3)
    dev = DeviceWorkload(w)
    host = DeviceWorkload(w)
    hstate = [[t.cpu().pin_memory() for t in ts] for ts in (host.master, host.m, host.v)]
    for step in range(w.steps):
        dev.gen_grads(step, dev.scaler().scale)
        host.grads.copy_(dev.grads)
        ra = dev.step()
        rb = host.flat.step(w.ranks, host.grads, *hstate, host.out,
                            grad_rank_offset_mul=w.grad_rank_mul)
        assert (ra.overflow, ra.skipped, ra.grad_norm, ra.clip_coef) == \
               (rb.overflow, rb.skipped, rb.grad_norm, rb.clip_coef)
    _same(dev.master + dev.m + dev.v + [dev.out], hstate[0] + hstate[1] + hstate[2] + [host.out])
    dev.close()
    host.close()


def test_bf16_grads_fp16_params(ora):
    w = Workload(name="bf16_to_fp16", description="bf16 grads, fp16 params",
                 shapes=[(40_001,), (7,)], world_size=4, ranks=[0, 1, 2, 3], grad_dtype=BF16,
                 op=AVG, dynamic=False, steps=3, sigma_g=1e-3, sigma_n=1e-3, pdtype=F16)
    run_parity(ora, w)


@pytest.mark.parametrize("numel,form", [(2_000_017, "staged"), (8 * 65_536, "plain")],
                         ids=["staged_bulk_copies", "plain_loads"])
def test_gradients_in_pinned_host_memory(numel, form):
    """The contributions read straight from page-locked host memory (no copy):
    the bits of the device-resident step -- through the staged reduce's bulk
    copies (slice rows 16 bytes off 64-byte boundaries) and through the plain
    reduce's 16-byte loads (aligned rows, a small reduce)."""
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = Workload(name="hostgrads", description="hostgrads", shapes=[(numel,)], world_size=8,
                 ranks=[5], grad_dtype=F16, op=AVG, dynamic=True, steps=3, sigma_g=1e-3,
                 sigma_n=1e-3, grads_layout="slice")
    dev, hst = DeviceWorkload(w), DeviceWorkload(w)
    pinned = torch.empty(dev.grads.shape, dtype=dev.grads.dtype, pin_memory=True)
    for step in range(w.steps):
        dev.gen_grads(step, dev.scaler().scale)
        pinned.copy_(dev.grads)
        ra = dev.step()
        rb = hst.flat.step(w.ranks, pinned, hst.master, hst.m, hst.v, hst.out,
                           grad_rank_offset_mul=0)
        assert (ra.overflow, ra.skipped, ra.grad_norm, ra.clip_coef) == \
               (rb.overflow, rb.skipped, rb.grad_norm, rb.clip_coef)
        assert dev.flat.reduce_form() == hst.flat.reduce_form() == form
    _same(dev.master + dev.m + dev.v + [dev.out], hst.master + hst.m + hst.v + [hst.out])
    dev.close()
    hst.close()
