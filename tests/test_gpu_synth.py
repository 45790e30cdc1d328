"""The device generator draws the host generator's distribution: the same
Philox words, and the platform's own logf / sqrtf / cos in Box-Muller, so
values agree to a few ulp (tests that compare the GPU with the oracle hand the
oracle the GPU's bytes, so bit identity is not needed)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
import synth  # noqa: E402

pytestmark = pytest.mark.gpu


def _decode(u, bf16):
    if bf16:
        return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return u.view(np.float16).astype(np.float64)


def test_device_matches_host_generator():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    n = 3_000_017
    for kind, first, sigma, absval in ((synth.MASTER, 0, 0.02, False),
                                       (synth.MOMENT_V, 5 * 10 ** 9, 1e-8, True)):
        t = torch.empty(n, dtype=torch.float32, device="cuda")
        synth.normal_device(t, 11, kind, first, sigma, absval=absval)
        d = t.cpu().numpy().astype(np.float64)
        h = synth.normal_host(11, kind, first, n, sigma, absval=absval).astype(np.float64)
        # a few ulp of the value, or of sigma where the cosine is near zero
        assert np.all(np.abs(d - h) <= 1e-6 * np.abs(h) + 1e-6 * sigma)
    for dtype in (synth.F16, synth.BF16):
        g = torch.empty((3, n + 5), dtype=torch.float16, device="cuda")
        synth.grads_device(g, 4, 7, 10 ** 9, n, 1e-3, 2e-3, scale=4096.0 if dtype == 0 else 1.0,
                           dtype=dtype, zero_from=10 ** 9 + n - 10)
        d = g[:, :n].view(torch.int16).cpu().numpy().view(np.uint16)
        h = synth.grads_host(4, 7, 3, 10 ** 9, n, 1e-3, 2e-3, scale=4096.0 if dtype == 0 else 1.0,
                             dtype=dtype, zero_from=10 ** 9 + n - 10)
        # g and n each agree to a few fp32 ulp; their sum can cancel, so the
        # bound is absolute (in units of the gradient's scale) plus one ulp of
        # the 16-bit cast
        bf16 = dtype == synth.BF16
        dd, hh = _decode(d, bf16), _decode(h, bf16)
        s = 4096.0 if dtype == 0 else 1.0
        ulp = 2.0 ** (-7 if bf16 else -10)
        assert np.all(np.abs(dd - hh) <= ulp * np.abs(hh) + 1e-6 * 3e-3 * s * 6)
        assert np.mean(d == h) > 0.99
        assert not d[:, n - 10:].any()
