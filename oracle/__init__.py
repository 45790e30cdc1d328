"""Python access to the oracle (plain C CPU restatement of the ZeRO shard step).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.  The arithmetic lives
in ``zero_oracle.c``; this module only marshals numpy arrays.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


class Hparams(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("eps", C.c_double), ("weight_decay", C.c_double),
                ("max_grad_norm", C.c_double), ("dynamic_loss_scale", C.c_int32),
                ("initial_scale_power", C.c_int32), ("loss_scale_window", C.c_int32),
                ("pad_", C.c_int32),
                ("static_loss_scale", C.c_double), ("min_loss_scale", C.c_double)]


class Scaler(C.Structure):
    _fields_ = [("scale", C.c_float), ("good_steps", C.c_int32),
                ("step_t", C.c_int64), ("overflow_count", C.c_int64)]

    def as_tuple(self):
        return (self.scale, self.good_steps, self.step_t, self.overflow_count)


class ExactAcc(C.Structure):
    """Exact fixed-point accumulator of squares (640 bits, unit 2^-298)."""
    _fields_ = [("w", C.c_uint64 * 10)]


class Result(C.Structure):
    _fields_ = [("overflow", C.c_int32), ("skipped", C.c_int32),
                ("grad_norm", C.c_double), ("clip_coef", C.c_float),
                ("scale_used", C.c_float)]


def hparams(lr=3e-5, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
            max_grad_norm=1.0, dynamic=True, initial_scale_power=16,
            window=1000, static_scale=1.0, min_scale=1.0):
    """ds_config-style hyper-parameters (defaults: the AdamW / fp16 / clipping
    values of the DeepSpeed config printed in the ZeRO reading, §5.1)."""
    return Hparams(lr, beta1, beta2, eps, weight_decay, max_grad_norm,
                   1 if dynamic else 0, initial_scale_power, window, 0,
                   static_scale, min_scale)


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        i64p = C.POINTER(C.c_int64)
        u64p = C.POINTER(C.c_uint64)
        L.ora_layout.argtypes = [i64p, i64p, C.c_int32, C.c_int32, i64p, i64p, i64p]
        L.ora_memory_breakdown.argtypes = [C.c_int32, C.c_uint64, C.c_int32,
                                           u64p, u64p, u64p, u64p]
        L.ora_f16_to_f32.argtypes = [C.c_uint16]
        L.ora_f16_to_f32.restype = C.c_float
        L.ora_bf16_to_f32.argtypes = [C.c_uint16]
        L.ora_bf16_to_f32.restype = C.c_float
        L.ora_f32_to_f16.argtypes = [C.c_float]
        L.ora_f32_to_f16.restype = C.c_uint16
        L.ora_f32_to_bf16.argtypes = [C.c_float]
        L.ora_f32_to_bf16.restype = C.c_uint16
        L.ora_scaler_init.argtypes = [C.POINTER(Hparams), C.POINTER(Scaler)]
        L.ora_reduce_unscale.argtypes = [C.c_int32, C.c_void_p, C.c_int64, C.c_int64,
                                         C.c_int32, C.c_int64, C.c_int64, C.c_int64,
                                         C.c_int32, C.c_float, C.c_void_p]
        L.ora_norm_accumulate.argtypes = [C.c_void_p, C.c_int64, C.POINTER(ExactAcc),
                                          C.POINTER(C.c_int32)]
        L.ora_norm_sum.argtypes = [C.POINTER(ExactAcc)]
        L.ora_norm_sum.restype = C.c_double
        L.ora_acc_merge.argtypes = [C.POINTER(ExactAcc), C.POINTER(ExactAcc)]
        L.ora_scaler_decide.argtypes = [C.POINTER(Hparams), C.POINTER(Scaler), C.c_int32,
                                        C.c_double, C.POINTER(C.c_float),
                                        C.POINTER(C.c_int32)]
        L.ora_adamw_cast.argtypes = [C.POINTER(Hparams), C.c_int64, C.c_float, C.c_void_p,
                                     C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64,
                                     C.c_void_p, C.c_int32]
        L.ora_shard_step.argtypes = [C.POINTER(Hparams), C.POINTER(Scaler), C.c_int32,
                                     C.c_int64, C.c_int64, C.c_int32, C.c_int32, C.c_int32,
                                     C.POINTER(C.c_int32), C.c_int32, C.c_void_p,
                                     C.c_int64, C.c_int64, C.POINTER(C.c_void_p),
                                     C.POINTER(C.c_void_p), C.POINTER(C.c_void_p),
                                     C.c_void_p, C.c_double, C.POINTER(Result)]
        L.ora_cast_array.argtypes = [C.c_void_p, C.c_int64, C.c_void_p, C.c_int32]
        L.ora_decode_array.argtypes = [C.c_void_p, C.c_int64, C.c_void_p, C.c_int32]
        L.ora_grad_accumulate.argtypes = [C.c_int32, C.c_int64, C.c_int64, C.c_int32, C.c_int32,
                                          C.POINTER(C.c_int32), C.c_int32, C.c_void_p,
                                          C.c_int64, C.c_int64, C.POINTER(C.c_void_p),
                                          C.c_int32]
        L.ora_shard_step_acc.argtypes = [C.POINTER(Hparams), C.POINTER(Scaler), C.c_int32,
                                         C.c_int64, C.c_int64, C.c_int32, C.POINTER(C.c_int32),
                                         C.c_int32, C.POINTER(C.c_void_p),
                                         C.POINTER(C.c_void_p), C.POINTER(C.c_void_p),
                                         C.POINTER(C.c_void_p), C.c_void_p, C.c_double,
                                         C.POINTER(Result)]
        L.ora_unscale_acc.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_int64, C.c_float,
                                      C.c_void_p]
        L.ora_quantize_q8.argtypes = [C.c_void_p, C.c_int64, C.c_int32, C.c_void_p, C.c_void_p]
        L.ora_ddp_step.argtypes = [C.POINTER(Hparams), C.POINTER(Scaler), C.c_int32,
                                   C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                   C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p,
                                   C.c_void_p, C.POINTER(Result)]
        _lib = L
    return _lib


def _grad_kind(grads, grad_is_bf16):
    """Contribution encoding: 0 fp16 / 1 bf16 (uint16 arrays), 2 fp32."""
    if isinstance(grads, np.ndarray) and grads.dtype == np.float32:
        assert grads.flags.c_contiguous
        return 2
    _check(grads, np.uint16)
    return 1 if grad_is_bf16 else 0


def _ptr_array(arrs, n=None, dtype=np.float32):
    for a in arrs:
        _check(a, dtype)
        if n is not None:
            assert a.size == n
    return (C.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _ptr(a):
    return a.ctypes.data_as(C.c_void_p)


def _check(a, dtype):
    assert isinstance(a, np.ndarray) and a.dtype == dtype and a.flags.c_contiguous, \
        (type(a), getattr(a, "dtype", None))
    return a


def layout(numels, world_size):
    """(full_numel, shard_size, padded_numel) of a FlatParameter built from
    parameters of the given element counts, concatenated in order."""
    numels = np.asarray(numels, dtype=np.int64)
    starts = np.concatenate([[0], np.cumsum(numels)[:-1]]).astype(np.int64)
    out = [C.c_int64() for _ in range(3)]
    rc = lib().ora_layout(starts.ctypes.data_as(C.POINTER(C.c_int64)),
                          numels.ctypes.data_as(C.POINTER(C.c_int64)),
                          len(numels), world_size, *[C.byref(o) for o in out])
    if rc:
        raise ValueError("ora_layout failed: %d" % rc)
    return tuple(o.value for o in out)


def layout_raw(starts, numels, world_size):
    """ora_layout on an explicit (starts, numels) table; returns (rc, triple)."""
    starts = np.asarray(starts, dtype=np.int64)
    numels = np.asarray(numels, dtype=np.int64)
    out = [C.c_int64() for _ in range(3)]
    rc = lib().ora_layout(starts.ctypes.data_as(C.POINTER(C.c_int64)),
                          numels.ctypes.data_as(C.POINTER(C.c_int64)),
                          len(numels), world_size, *[C.byref(o) for o in out])
    return rc, tuple(o.value for o in out)


def memory_breakdown(stage, psi, world_size):
    """(params, grads, optimizer, total) bytes per GPU."""
    out = [C.c_uint64() for _ in range(4)]
    rc = lib().ora_memory_breakdown(stage, psi, world_size, *[C.byref(o) for o in out])
    if rc:
        raise ValueError("ora_memory_breakdown failed: %d" % rc)
    return tuple(o.value for o in out)


def f32_to_f16_bits(x):
    return int(lib().ora_f32_to_f16(float(x)))


def f32_to_bf16_bits(x):
    return int(lib().ora_f32_to_bf16(float(x)))


def f16_bits_to_f32(h):
    return lib().ora_f16_to_f32(int(h))


def bf16_bits_to_f32(h):
    return lib().ora_bf16_to_f32(int(h))


def cast_array(x, to_bf16=False):
    """fp32 array -> 16-bit encodings (uint16) by the oracle's RNE casts."""
    _check(x, np.float32)
    out = np.empty(max(x.size, 1), dtype=np.uint16)
    lib().ora_cast_array(_ptr(x), x.size, _ptr(out), int(to_bf16))
    return out[:x.size]


def decode_array(h, from_bf16=False):
    """16-bit encodings (uint16) -> fp32 values."""
    _check(h, np.uint16)
    out = np.empty(max(h.size, 1), dtype=np.float32)
    lib().ora_decode_array(_ptr(h), h.size, _ptr(out), int(from_bf16))
    return out[:h.size]


def quantize_q8(p, block=256):
    """(codes int8 [n], scales float32 [ceil(n/block)]) of decoded params p."""
    _check(p, np.float32)
    n = p.size
    q = np.empty(max(n, 1), np.int8)
    sc = np.empty(max(-(-n // block), 1), np.float32)
    lib().ora_quantize_q8(_ptr(p), n, block, _ptr(q), _ptr(sc))
    return q[:n], sc[:-(-n // block)]


def scaler_init(hp):
    st = Scaler()
    lib().ora_scaler_init(C.byref(hp), C.byref(st))
    return st


def reduce_unscale(grads_u16, ld, rank_off, n_contrib, count, first_flat_index,
                   full_numel, avg, scale, grad_is_bf16=False, out=None):
    """Reduced, unscaled fp32 gradient of `count` elements (into `out` if given).
    grads_u16: uint16 fp16/bf16 encodings, or a float32 array of fp32 contributions."""
    kind = _grad_kind(grads_u16, grad_is_bf16)
    g = np.empty(max(count, 1), dtype=np.float32) if out is None else _check(out, np.float32)
    assert g.size >= count
    lib().ora_reduce_unscale(kind, _ptr(grads_u16), ld, rank_off, n_contrib,
                             count, first_flat_index, full_numel, int(avg), scale, _ptr(g))
    return g[:count]


def norm_accumulate(g, acc=None, overflow=0):
    """Add the exact squares of g to `acc` (a new accumulator if None);
    returns (acc, overflow)."""
    _check(g, np.float32)
    acc = ExactAcc() if acc is None else acc
    of = C.c_int32(overflow)
    lib().ora_norm_accumulate(_ptr(g), g.size, C.byref(acc), C.byref(of))
    return acc, of.value


def norm_sum(acc):
    """The accumulated sum of squares rounded to the nearest double."""
    return lib().ora_norm_sum(C.byref(acc))


def acc_merge(dst, src):
    lib().ora_acc_merge(C.byref(dst), C.byref(src))
    return dst


def sum_of_squares(g):
    acc, of = norm_accumulate(g)
    return norm_sum(acc), of


def scaler_decide(hp, st, overflow, norm):
    coef = C.c_float()
    skip = C.c_int32()
    lib().ora_scaler_decide(C.byref(hp), C.byref(st), int(overflow), float(norm),
                            C.byref(coef), C.byref(skip))
    return coef.value, skip.value


def adamw_cast(hp, t, coef, g, theta, m, v, param_is_bf16=False, out=None):
    """In-place AdamW on theta, m, v (fp32); returns the 16-bit cast as uint16
    (written into `out` if given)."""
    for a in (g, theta, m, v):
        _check(a, np.float32)
    n = g.size
    assert theta.size == n and m.size == n and v.size == n
    if out is None:
        out = np.empty(max(n, 1), dtype=np.uint16)
    else:
        _check(out, np.uint16)
        assert out.size >= n
    lib().ora_adamw_cast(C.byref(hp), t, coef, _ptr(g), _ptr(theta), _ptr(m), _ptr(v),
                         n, _ptr(out), int(param_is_bf16))
    return out[:n]


def shard_step(hp, st, world_size, full_numel, shard_size, ranks, grads_u16, ld,
               rank_mul, master, m, v, flat_out, avg=True, grad_is_bf16=False,
               param_is_bf16=False, extra_norm_sq=0.0):
    """One ZeRO shard step on the listed ranks; master/m/v are lists of fp32
    arrays (one per stepped rank), flat_out a uint16 array of padded_numel.
    grads_u16: uint16 fp16/bf16 encodings, or float32 fp32 contributions."""
    kind = _grad_kind(grads_u16, grad_is_bf16)
    _check(flat_out, np.uint16)
    ranks_a = (C.c_int32 * len(ranks))(*ranks)
    arrs = []
    for lst in (master, m, v):
        assert len(lst) == len(ranks)
        for a in lst:
            _check(a, np.float32)
            assert a.size == shard_size
        arrs.append((C.c_void_p * len(lst))(*[a.ctypes.data for a in lst]))
    res = Result()
    rc = lib().ora_shard_step(C.byref(hp), C.byref(st), world_size, full_numel,
                              shard_size, kind, int(param_is_bf16), int(avg),
                              ranks_a, len(ranks), _ptr(grads_u16), ld, rank_mul,
                              arrs[0], arrs[1], arrs[2], _ptr(flat_out),
                              float(extra_norm_sq), C.byref(res))
    if rc:
        raise ValueError("ora_shard_step failed: %d" % rc)
    return res


def grad_accumulate(world_size, full_numel, shard_size, ranks, grads, ld, rank_mul, acc,
                    first, avg=True, grad_is_bf16=False):
    """acc[j] (fp32 arrays, one per stepped rank) = reduce(grads) if first,
    else acc[j] + reduce(grads)."""
    kind = _grad_kind(grads, grad_is_bf16)
    ranks_a = (C.c_int32 * len(ranks))(*ranks)
    rc = lib().ora_grad_accumulate(world_size, full_numel, shard_size, kind, int(avg), ranks_a,
                                   len(ranks), _ptr(grads), ld, rank_mul,
                                   _ptr_array(acc, shard_size), int(bool(first)))
    if rc:
        raise ValueError("ora_grad_accumulate failed: %d" % rc)


def unscale_acc(acc, first_flat_index, full_numel, scale, out=None):
    """g = acc / scale for real elements, 0 for padding (flat index >= full_numel)."""
    _check(acc, np.float32)
    out = np.empty(acc.size, np.float32) if out is None else out
    _check(out, np.float32)
    assert out.size == acc.size
    lib().ora_unscale_acc(_ptr(acc), acc.size, first_flat_index, full_numel, float(scale),
                          _ptr(out))
    return out


def shard_step_acc(hp, st, world_size, full_numel, shard_size, ranks, acc, master, m, v,
                   flat_out, param_is_bf16=False, extra_norm_sq=0.0):
    """The optimizer step on accumulated fp32 shards acc[j]."""
    _check(flat_out, np.uint16)
    ranks_a = (C.c_int32 * len(ranks))(*ranks)
    res = Result()
    rc = lib().ora_shard_step_acc(C.byref(hp), C.byref(st), world_size, full_numel, shard_size,
                                  int(param_is_bf16), ranks_a, len(ranks),
                                  _ptr_array(acc, shard_size), _ptr_array(master, shard_size),
                                  _ptr_array(m, shard_size), _ptr_array(v, shard_size),
                                  _ptr(flat_out), float(extra_norm_sq), C.byref(res))
    if rc:
        raise ValueError("ora_shard_step_acc failed: %d" % rc)
    return res


def ddp_step(hp, st, n_contrib, full_numel, grads_u16, ld, master, m, v, out,
             avg=True, grad_is_bf16=False, param_is_bf16=False):
    for a in (master, m, v):
        _check(a, np.float32)
    kind = _grad_kind(grads_u16, grad_is_bf16)
    _check(out, np.uint16)
    res = Result()
    rc = lib().ora_ddp_step(C.byref(hp), C.byref(st), n_contrib, full_numel,
                            kind, int(param_is_bf16), int(avg),
                            _ptr(grads_u16), ld, _ptr(master), _ptr(m), _ptr(v),
                            _ptr(out), C.byref(res))
    if rc:
        raise ValueError("ora_ddp_step failed: %d" % rc)
    return res
