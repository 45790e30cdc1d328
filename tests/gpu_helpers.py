"""Comparison of the CUDA path with the oracle, with the tolerances the
target states: fp32 master within 1e-6 relative (absolute floor 1e-10), m and
v within 1e-5 relative, the global norm within 1e-5 relative, 16-bit params
within 1 ulp, and the overflow flag, skip decision, loss scale and its
counters bit-exact.  (Expected in practice: bit-exact everywhere except where
the clip coefficient, derived from the differently-summed norm, differs by an
ulp.)"""
import numpy as np

MASTER_RTOL, MASTER_ATOL = 1e-6, 1e-10
MV_RTOL, MV_ATOL = 1e-5, 1e-30
NORM_RTOL = 1e-5
PARAM_ULP = 1


def u16(t):
    """16-bit CUDA/CPU tensor -> numpy uint16 encodings."""
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def host_grads(t):
    """Gradient contributions as the oracle takes them: uint16 encodings of a
    16-bit tensor, or the float32 values of an fp32 one."""
    import torch
    if t.dtype == torch.float32:
        return t.detach().cpu().numpy()
    return u16(t)


def f32(t):
    return t.detach().cpu().numpy()


def _key16(u, bf16):
    """Monotonic integer key of 16-bit float encodings (ulp distance = key
    difference, across the sign too)."""
    u = u.astype(np.int32)
    mag = u & 0x7FFF
    return np.where(u & 0x8000, -mag, mag)


def assert_params_close(got, want, bf16=False, what="params"):
    assert got.shape == want.shape, (got.shape, want.shape)
    gnan = (got & 0x7FFF) > (0x7F80 if bf16 else 0x7C00)
    wnan = (want & 0x7FFF) > (0x7F80 if bf16 else 0x7C00)
    assert np.array_equal(gnan, wnan), what + ": NaN positions differ"
    d = np.abs(_key16(got[~gnan], bf16) - _key16(want[~wnan], bf16))
    if d.size:
        assert d.max() <= PARAM_ULP, "%s: %d ulp at %d" % (what, d.max(), int(np.argmax(d)))


def assert_rel(got, want, rtol, atol, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    lim = np.maximum(rtol * np.abs(want), atol)
    bad = err > lim
    if bad.any():
        k = int(np.argmax(err / lim))
        raise AssertionError("%s: %d elements off, worst at %d: got %r want %r" %
                             (what, int(bad.sum()), k, got[k], want[k]))


def assert_result(res, ora_tuple):
    of, skip, norm, coef, scale_used = ora_tuple
    assert res.overflow == of and res.skipped == skip
    assert res.scale_used == scale_used
    if not of:
        assert abs(res.grad_norm - norm) <= NORM_RTOL * norm + 1e-300, (res.grad_norm, norm)
        assert abs(res.clip_coef - coef) <= NORM_RTOL * coef, (res.clip_coef, coef)


def assert_state(master_g, m_g, v_g, master_o, m_o, v_o, tag=""):
    assert_rel(master_g, master_o, MASTER_RTOL, MASTER_ATOL, "master" + tag)
    assert_rel(m_g, m_o, MV_RTOL, MV_ATOL, "m" + tag)
    assert_rel(v_g, v_o, MV_RTOL, MV_ATOL, "v" + tag)


def bit_exact_fraction(a, b):
    return float(np.mean(a.view(np.uint32) == b.view(np.uint32))) if a.size else 1.0
