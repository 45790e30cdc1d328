"""The device generator gives the host generator's bits (so the oracle can
regenerate any input the GPU consumed)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
import synth  # noqa: E402

pytestmark = pytest.mark.gpu


def test_device_equals_host_generator():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    n = 3_000_017
    for kind, first, sigma, absval in ((synth.MASTER, 0, 0.02, False),
                                       (synth.MOMENT_V, 5 * 10 ** 9, 1e-8, True)):
        t = torch.empty(n, dtype=torch.float32, device="cuda")
        synth.normal_device(t, 11, kind, first, sigma, absval=absval)
        h = synth.normal_host(11, kind, first, n, sigma, absval=absval)
        assert np.array_equal(t.cpu().numpy().view(np.uint32), h.view(np.uint32))
    for dtype in (synth.F16, synth.BF16):
        g = torch.empty((3, n + 5), dtype=torch.float16, device="cuda")
        synth.grads_device(g, 4, 7, 10 ** 9, n, 1e-3, 2e-3, scale=4096.0 if dtype == 0 else 1.0,
                           dtype=dtype, zero_from=10 ** 9 + n - 10)
        d = g[:, :n].view(torch.int16).cpu().numpy().view(np.uint16)
        h = synth.grads_host(4, 7, 3, 10 ** 9, n, 1e-3, 2e-3, scale=4096.0 if dtype == 0 else 1.0,
                             dtype=dtype, zero_from=10 ** 9 + n - 10)
        assert np.array_equal(d, h)
