"""The host half of the ZeRO-Offload step (zero_offload_adamw_host): AdamW
and the 16-bit cast on the CPU cores, called through the C ABI with no GPU.

- against the oracle's AdamW + cast, bit for bit, over random shards with
  ragged sizes, both parameter dtypes, several step counts and clip
  coefficients, and any thread count;
- its fp16 rounding against numpy's float16 conversion and its bf16 rounding
  against torch's bfloat16 conversion (both round to nearest even), over
  every rounding boundary, subnormals, overflow and special values: with
  lr = 0 and no decay the update leaves theta as it is and the output is the
  cast alone;
- argument errors.
"""
import numpy as np
import pytest

import fsdp_sharded_mixed_zero_gb300 as Z


def _host_step(hp, t, coef, g, th, m, v, bf16=False, n_threads=0):
    out = np.zeros(max(g.size, 1), np.uint16)
    Z.zero_offload_adamw_host(hp, t, coef, g.ctypes.data, th.ctypes.data, m.ctypes.data,
                              v.ctypes.data, out.ctypes.data, g.size,
                              Z.ZERO_BF16 if bf16 else Z.ZERO_F16, n_threads)
    return out[:g.size]


def _ora_hp(ora, hp):
    return ora.hparams(lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps,
                       weight_decay=hp.weight_decay, max_grad_norm=hp.max_grad_norm)


def _state(rng, n, scale=1e-3):
    g = (rng.standard_normal(n) * scale).astype(np.float32)
    th = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * scale * 0.1).astype(np.float32)
    v = (np.abs(rng.standard_normal(n)) * scale * scale * 0.01).astype(np.float32)
    return g, th, m, v


def _same(a, b):
    return np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("n", [1, 7, 2048, 65_536 + 3, 300_001])
@pytest.mark.parametrize("bf16", [False, True], ids=["f16", "bf16"])
@pytest.mark.parametrize("t,coef", [(1, 1.0), (2, 0.37), (57, 1.0), (40_000, 0.0123)])
def test_matches_oracle_bit_for_bit(ora, n, bf16, t, coef):
    rng = np.random.default_rng(n * 31 + t)
    hp = Z.hparams(lr=1e-3, weight_decay=0.01)
    g, th, m, v = _state(rng, n)
    a = [x.copy() for x in (th, m, v)]
    b = [x.copy() for x in (th, m, v)]
    got = _host_step(hp, t, coef, g, *a, bf16=bf16)
    want = ora.adamw_cast(_ora_hp(ora, hp), t, np.float32(coef), g, *b, param_is_bf16=bf16)
    for x, y, what in zip(a, b, ("master", "m", "v")):
        assert _same(x, y), what
    assert np.array_equal(got, want)


def test_thread_count_does_not_change_bits():
    rng = np.random.default_rng(5)
    n = 5 * 65_536 + 11
    hp = Z.hparams(lr=3e-4)
    g, th, m, v = _state(rng, n)
    outs = []
    for nt in (1, 3, 0):
        s = [x.copy() for x in (th, m, v)]
        outs.append((_host_step(hp, 3, 0.5, g, *s, n_threads=nt), s))
    for out, s in outs[1:]:
        assert np.array_equal(out, outs[0][0])
        for x, y in zip(s, outs[0][1]):
            assert _same(x, y)


def _cast_only(theta, bf16):
    """The update with lr = 0, no decay, zero gradient and moments leaves
    theta unchanged; the output is then its 16-bit encoding."""
    n = theta.size
    hp = Z.hparams(lr=0.0, weight_decay=0.0)
    th = theta.copy()
    z = np.zeros(n, np.float32)
    out = _host_step(hp, 1, 1.0, z.copy(), th, z.copy(), z.copy(), bf16=bf16)
    fin = np.isfinite(theta)
    assert _same(th[fin], theta[fin])
    return out


def _boundary_values():
    """fp32 values at and around every fp16 and bf16 rounding boundary: the
    representable 16-bit values, the midpoints between neighbours (ties) and
    one fp32 ulp either side, over the whole exponent range, plus zeros,
    infinities, NaNs, fp32 subnormals and the largest finite values."""
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (h[:-1] + h[1:]) / 2
    vals = [h, mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)).astype(np.float64),
            np.nextafter(mids.astype(np.float32), np.float32(0)).astype(np.float64),
            np.array([65504.0, 65519.99, 65520.0, 65536.0, 1e6, 3.4e38])]
    b = (np.arange(0, 0x7F80, 7, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    bm = ((np.arange(0, 0x7F80, 7, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    vals += [b, bm.astype(np.float64),
             (((np.arange(0, 0x7F80, 7, dtype=np.uint32) << 16) | 0x18000)).view(np.float32)
             .astype(np.float64)]
    x = np.concatenate(vals).astype(np.float32)
    x = np.concatenate([x, -x, np.array([0.0, -0.0, np.inf, -np.inf, np.nan], np.float32),
                        np.array([1, 2, 0x7FFFFF, 0x807FFFFF, 0x7F7FFFFF, 0xFF7FFFFF,
                                  0x7FC00001, 0xFF800001], np.uint32).view(np.float32)])
    return x


def test_f16_rounding_matches_numpy():
    x = _boundary_values()
    got = _cast_only(x, bf16=False)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all((got[nan] & 0x7C00) == 0x7C00) and np.all((got[nan] & 0x03FF) != 0)


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = _boundary_values()
    got = _cast_only(x, bf16=True)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all((got[nan] & 0x007F) != 0)


def test_argument_errors():
    hp = Z.hparams()
    a = np.zeros(8, np.float32)
    o = np.zeros(8, np.uint16)
    p = [a.ctypes.data] * 4

    def call(**kw):
        args = dict(hp=hp, step_t=1, clip_coef=1.0, g_ptr=p[0], master_ptr=p[1], m_ptr=p[2],
                    v_ptr=p[3], out_ptr=o.ctypes.data, n=8, param_dtype=Z.ZERO_F16, n_threads=1)
        args.update(kw)
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_offload_adamw_host(**args)
        return e.value.status

    assert call(step_t=0) == 1
    assert call(n=-1) == 1
    assert call(n_threads=-2) == 1
    assert call(g_ptr=0) == 1
    assert call(param_dtype=Z.ZERO_F32) == 2
    assert call(m_ptr=p[2] + 2) == 3
    assert call(out_ptr=o.ctypes.data + 1) == 3
    assert call(hp=Z.hparams(beta1=1.0)) == 1
    Z.zero_offload_adamw_host(hp, 1, 1.0, 0, 0, 0, 0, 0, 0)      # n = 0: nothing to do
