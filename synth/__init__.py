"""Seeded synthetic inputs for the ZeRO shard step (shared by the oracle side
and the CUDA side; no optimizer arithmetic lives here).

Every tensor is a pure function of (seed, stream id, flat element index):
Philox4x32-10 bits turned into approximately normal values by a four-term
Irwin-Hall sum.  The host generator (threads) and the device generator (CUDA)
give identical bits, so the oracle can regenerate any element it checks.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

MASTER, MOMENT_M, MOMENT_V, GRAD_SHARED, GRAD_NOISE = 1, 2, 3, 4, 5
F16, BF16, F32 = 0, 1, 2

_lib = None


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(_build.build())
        L.synth_philox4x32_10.argtypes = [C.POINTER(C.c_uint32)] * 3
        L.synth_stream_id.argtypes = [C.c_uint32] * 3
        L.synth_stream_id.restype = C.c_uint32
        L.synth_normal_f32_host.argtypes = [C.c_uint32, C.c_uint32, C.c_uint64, C.c_int64,
                                            C.c_double, C.c_int, C.c_void_p, C.c_int]
        L.synth_grads_host.argtypes = [C.c_uint32, C.c_uint32, C.c_int32, C.c_int32,
                                       C.c_double, C.c_double, C.c_float, C.c_int,
                                       C.c_uint64, C.c_int64, C.c_uint64, C.c_void_p,
                                       C.c_int64, C.c_int]
        L.synth_normal_f32_device.argtypes = [C.c_uint32, C.c_uint32, C.c_uint64, C.c_int64,
                                              C.c_double, C.c_int, C.c_void_p, C.c_void_p]
        L.synth_grads_device.argtypes = [C.c_uint32, C.c_uint32, C.c_int32, C.c_int32,
                                         C.c_double, C.c_double, C.c_float, C.c_int,
                                         C.c_uint64, C.c_int64, C.c_uint64, C.c_void_p,
                                         C.c_int64, C.c_void_p]
        _lib = L
    return _lib


def _threads():
    return max(1, min(32, os.cpu_count() or 1))


def philox(ctr, key):
    c = (C.c_uint32 * 4)(*ctr)
    k = (C.c_uint32 * 2)(*key)
    o = (C.c_uint32 * 4)()
    lib().synth_philox4x32_10(c, k, o)
    return list(o)


def stream_id(kind, step=0, contrib=0):
    return int(lib().synth_stream_id(kind, step, contrib))


def normal_host(seed, kind, first, n, sigma, absval=False, step=0, contrib=0):
    out = np.empty(max(n, 1), np.float32)
    rc = lib().synth_normal_f32_host(seed, stream_id(kind, step, contrib), first, n, sigma,
                                     int(absval), out.ctypes.data_as(C.c_void_p), _threads())
    assert rc == 0
    return out[:n]


def grads_host(seed, step, n_contrib, first, n, sigma_g, sigma_n, scale=1.0, dtype=F16,
               zero_from=None, c0=0):
    """uint16 encodings [n_contrib, n] (fp16 via the compiler's conversion,
    bf16 via torch's conversion of the fp32 pre-cast values), or the fp32
    values themselves for dtype F32."""
    zero_from = (1 << 64) - 1 if zero_from is None else zero_from
    if dtype == F16:
        out = np.empty((n_contrib, max(n, 1)), np.uint16)
        rc = lib().synth_grads_host(seed, step, c0, n_contrib, sigma_g, sigma_n, scale, 0,
                                    first, n, zero_from, out.ctypes.data_as(C.c_void_p),
                                    out.shape[1], _threads())
        assert rc == 0
        return out[:, :n]
    import torch
    f = np.empty((n_contrib, max(n, 1)), np.float32)
    rc = lib().synth_grads_host(seed, step, c0, n_contrib, sigma_g, sigma_n, scale, 2,
                                first, n, zero_from, f.ctypes.data_as(C.c_void_p),
                                f.shape[1], _threads())
    assert rc == 0
    if dtype == F32:
        return np.ascontiguousarray(f[:, :n])
    b = torch.from_numpy(f[:, :n].copy()).to(torch.bfloat16)
    return b.view(torch.int16).numpy().view(np.uint16)


def normal_device(tensor, seed, kind, first, sigma, absval=False, step=0, contrib=0,
                  stream=None):
    """Fill a contiguous float32 CUDA tensor."""
    import torch
    assert tensor.dtype == torch.float32 and tensor.is_cuda and tensor.is_contiguous()
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = lib().synth_normal_f32_device(seed, stream_id(kind, step, contrib), first,
                                       tensor.numel(), sigma, int(absval),
                                       C.c_void_p(tensor.data_ptr()), C.c_void_p(s.cuda_stream))
    assert rc == 0


def grads_device(tensor, seed, step, first, n, sigma_g, sigma_n, scale=1.0, dtype=F16,
                 zero_from=None, c0=0, n_contrib=None, stream=None):
    """Fill rows of a 2-D CUDA tensor [n_contrib, ld] (16-bit for F16/BF16,
    float32 for F32; uses the first n columns of each row)."""
    import torch
    assert tensor.dim() == 2 and tensor.is_cuda
    assert tensor.element_size() == (4 if dtype == F32 else 2)
    assert tensor.stride(1) == 1
    nc = tensor.shape[0] if n_contrib is None else n_contrib
    zero_from = (1 << 64) - 1 if zero_from is None else zero_from
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = lib().synth_grads_device(seed, step, c0, nc, sigma_g, sigma_n, scale, dtype, first,
                                  n, zero_from, C.c_void_p(tensor.data_ptr()),
                                  tensor.stride(0), C.c_void_p(s.cuda_stream))
    assert rc == 0
