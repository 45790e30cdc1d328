"""GB300 ZeRO shard optimizer step on a FlatParameter -- Python binding.

A thin ctypes layer over ``libzero_gb300.so`` (the C ABI in include/zero.h):
the functions keep the C names and only marshal arguments.  Every step of the
path runs in the library's CUDA kernels; there is no CPU or PyTorch fallback,
and importing this module fails loudly if the library has not been built
(``python -m fsdp_sharded_mixed_zero_gb300.build`` or ``__graft_entry__.build()``).

PyTorch is used only to hand over device pointers and CUDA streams.
"""
import ctypes as C
import os

__all__ = [
    "ZERO_OK", "ZERO_F16", "ZERO_BF16", "ZERO_F32", "ZERO_SUM", "ZERO_AVG", "ZeroError",
    "ParamInfo", "Hparams", "ScalerState", "StepResult", "hparams", "param_infos",
    "zero_flat_init", "zero_flat_layout", "zero_shard_step", "zero_loss_scaler_state",
    "zero_set_loss_scaler_state", "zero_memory_bytes", "zero_flat_device_bytes",
    "zero_flat_free", "zero_flat_profile_enable", "zero_flat_profile_read",
    "zero_flat_profile_reduce_form",
    "zero_shard_step_noalloc", "zero_grad_accumulate", "zero_shard_step_accumulated",
    "zero_shard_step_q8", "ZERO_Q8_BLOCK", "zero_flat_set_lr", "zero_shard_step_offload",
    "zero_offload_adamw_host", "zero_debug_set_stage_tx_pad", "zero_debug_reduce_form",
    "zero_shard_reduce",
    "zero_shard_apply", "zero_shard_apply_partials", "zero_shard_apply_partials_q8",
    "zero_shard_reduce_accumulated",
    "GroupMember", "ZeroGroup", "zero_group_init", "zero_group_step",
    "zero_group_step_q8", "zero_group_step_accumulated", "zero_group_step_offload",
    "zero_group_accumulate", "zero_group_loss_scaler_state", "zero_group_set_loss_scaler_state",
    "zero_group_set_lr", "zero_group_free",
    "zero_status_string", "zero_last_error", "ZeroFlat",
    "LIB_PATH",
]

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libzero_gb300.so")

ZERO_OK = 0
ZERO_F16, ZERO_BF16, ZERO_F32 = 0, 1, 2
ZERO_SUM, ZERO_AVG = 0, 1
ZERO_Q8_BLOCK = 256


class ZeroError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = "%s: %s (%s)" % (where, _lib.zero_status_string(status).decode(),
                               _lib.zero_last_error().decode())
        super().__init__(msg)


class ParamInfo(C.Structure):
    _fields_ = [("offset", C.c_int64), ("numel", C.c_int64), ("ndim", C.c_int32),
                ("dtype", C.c_int32), ("shape", C.c_int64 * 8)]


class Hparams(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("eps", C.c_double), ("weight_decay", C.c_double),
                ("max_grad_norm", C.c_double), ("dynamic_loss_scale", C.c_int32),
                ("initial_scale_power", C.c_int32), ("loss_scale_window", C.c_int32),
                ("reserved", C.c_int32), ("static_loss_scale", C.c_double),
                ("min_loss_scale", C.c_double)]


class ScalerState(C.Structure):
    _fields_ = [("scale", C.c_float), ("good_steps", C.c_int32), ("step_t", C.c_int64),
                ("overflow_count", C.c_int64)]

    def as_tuple(self):
        return (self.scale, self.good_steps, self.step_t, self.overflow_count)


class StepResult(C.Structure):
    _fields_ = [("overflow", C.c_int32), ("skipped", C.c_int32), ("grad_norm", C.c_double),
                ("clip_coef", C.c_float), ("scale_used", C.c_float)]


class GroupMember(C.Structure):
    _fields_ = [("ranks", C.POINTER(C.c_int32)), ("n_ranks", C.c_int32), ("grads", C.c_void_p),
                ("grad_ld", C.c_int64), ("grad_rank_offset_mul", C.c_int64),
                ("master", C.POINTER(C.c_void_p)), ("m", C.POINTER(C.c_void_p)),
                ("v", C.POINTER(C.c_void_p)), ("flat_param_out", C.c_void_p),
                ("acc", C.POINTER(C.c_void_p)), ("flat_q8_out", C.c_void_p),
                ("q8_scales", C.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libzero_gb300.so is not built (expected at %s); run "
                          "fsdp_sharded_mixed_zero_gb300/build.py" % LIB_PATH)
    L = C.CDLL(LIB_PATH)
    vp, i32, i64, u64 = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64
    L.zero_flat_init.argtypes = [C.POINTER(ParamInfo), i32, i32, i32, i32, i32,
                                 C.POINTER(Hparams), C.POINTER(vp)]
    L.zero_flat_layout.argtypes = [vp, C.POINTER(i64), C.POINTER(i64), C.POINTER(i64)]
    L.zero_shard_step.argtypes = [vp, C.POINTER(i32), i32, vp, i64, i64, C.POINTER(vp),
                                  C.POINTER(vp), C.POINTER(vp), vp, C.c_double, vp,
                                  C.POINTER(StepResult)]
    L.zero_loss_scaler_state.argtypes = [vp, C.POINTER(ScalerState), vp]
    L.zero_set_loss_scaler_state.argtypes = [vp, C.POINTER(ScalerState), vp]
    L.zero_memory_bytes.argtypes = [i32, u64, i32] + [C.POINTER(u64)] * 4
    L.zero_flat_device_bytes.argtypes = [vp, C.POINTER(u64)]
    L.zero_flat_free.argtypes = [vp]
    L.zero_flat_profile_enable.argtypes = [vp, i32]
    L.zero_flat_profile_read.argtypes = [vp] + [C.POINTER(C.c_double)] * 3 + [C.POINTER(i64)]
    L.zero_flat_profile_reduce_form.argtypes = [vp, C.POINTER(i32)]
    L.zero_shard_step_noalloc.argtypes = [i64, i32, i32, i32, i32, C.POINTER(Hparams),
                                          C.POINTER(ScalerState), C.POINTER(i32), i32, vp, i64,
                                          i64, C.POINTER(vp), C.POINTER(vp), C.POINTER(vp), vp,
                                          C.c_double, vp, C.POINTER(StepResult)]
    L.zero_shard_step_q8.argtypes = [vp, C.POINTER(i32), i32, vp, i64, i64, C.POINTER(vp),
                                     C.POINTER(vp), C.POINTER(vp), vp, vp, vp, C.c_double, vp,
                                     C.POINTER(StepResult)]
    L.zero_grad_accumulate.argtypes = [vp, C.POINTER(i32), i32, vp, i64, i64, C.POINTER(vp), i32,
                                       vp]
    L.zero_shard_step_accumulated.argtypes = [vp, C.POINTER(i32), i32, C.POINTER(vp),
                                              C.POINTER(vp), C.POINTER(vp), C.POINTER(vp), vp,
                                              C.c_double, vp, C.POINTER(StepResult)]
    L.zero_flat_set_lr.argtypes = [vp, C.c_double]
    L.zero_debug_set_stage_tx_pad.argtypes = [C.c_uint32]
    L.zero_debug_reduce_form.argtypes = [i32, i32, i32, C.POINTER(u64), C.POINTER(i64),
                                         C.POINTER(i64), C.POINTER(u64), i32, C.POINTER(i32)]
    L.zero_shard_reduce.argtypes = [vp, C.POINTER(i32), i32, vp, i64, i64, vp, vp, vp]
    L.zero_group_init.argtypes = [C.POINTER(vp), i32, C.POINTER(vp)]
    L.zero_group_step.argtypes = [vp, C.POINTER(GroupMember), C.c_double, vp,
                                  C.POINTER(StepResult)]
    L.zero_group_step_q8.argtypes = [vp, C.POINTER(GroupMember), C.c_double, vp,
                                     C.POINTER(StepResult)]
    L.zero_group_step_offload.argtypes = [vp, C.POINTER(GroupMember), C.c_double, i32,
                                          C.c_double, vp, C.POINTER(StepResult)]
    L.zero_group_accumulate.argtypes = [vp, C.POINTER(GroupMember), i32, vp]
    L.zero_group_step_accumulated.argtypes = [vp, C.POINTER(GroupMember), C.c_double, vp,
                                              C.POINTER(StepResult)]
    L.zero_group_loss_scaler_state.argtypes = [vp, C.POINTER(ScalerState), vp]
    L.zero_group_set_loss_scaler_state.argtypes = [vp, C.POINTER(ScalerState), vp]
    L.zero_group_set_lr.argtypes = [vp, C.c_double]
    L.zero_group_free.argtypes = [vp]
    L.zero_shard_apply.argtypes = [vp, C.POINTER(i32), i32, C.POINTER(vp), C.POINTER(vp),
                                   C.POINTER(vp), vp, vp, vp, vp, C.POINTER(StepResult)]
    L.zero_shard_apply_partials.argtypes = [vp, C.POINTER(i32), i32, C.POINTER(vp),
                                            C.POINTER(vp), C.POINTER(vp), vp, vp, vp, i32, vp,
                                            C.POINTER(StepResult)]
    L.zero_shard_reduce_accumulated.argtypes = [vp, C.POINTER(i32), i32, C.POINTER(vp), vp, vp,
                                                vp]
    L.zero_shard_apply_partials_q8.argtypes = [vp, C.POINTER(i32), i32, C.POINTER(vp),
                                               C.POINTER(vp), C.POINTER(vp), vp, vp, vp, vp, vp,
                                               i32, vp, C.POINTER(StepResult)]
    L.zero_shard_step_offload.argtypes = [vp, C.POINTER(i32), i32, vp, i64, i64, C.POINTER(vp),
                                          C.POINTER(vp), C.POINTER(vp), vp, C.c_double, i32,
                                          C.c_double, vp, C.POINTER(StepResult)]
    L.zero_offload_adamw_host.argtypes = [C.POINTER(Hparams), i64, C.c_float, vp, vp, vp, vp,
                                          vp, i64, i32, i32]
    L.zero_status_string.argtypes = [i32]
    L.zero_status_string.restype = C.c_char_p
    L.zero_last_error.argtypes = []
    L.zero_last_error.restype = C.c_char_p
    for name in ("zero_flat_init", "zero_flat_layout", "zero_shard_step",
                 "zero_loss_scaler_state", "zero_set_loss_scaler_state", "zero_memory_bytes",
                 "zero_flat_device_bytes", "zero_flat_free", "zero_flat_profile_enable",
                 "zero_flat_profile_read", "zero_flat_profile_reduce_form",
                 "zero_shard_step_noalloc", "zero_grad_accumulate",
                 "zero_shard_step_q8", "zero_flat_set_lr", "zero_shard_step_offload",
                 "zero_offload_adamw_host", "zero_debug_set_stage_tx_pad",
                 "zero_debug_reduce_form",
                 "zero_shard_reduce", "zero_shard_apply", "zero_shard_apply_partials",
                 "zero_shard_apply_partials_q8", "zero_shard_reduce_accumulated",
                 "zero_group_init", "zero_group_step",
                 "zero_group_loss_scaler_state", "zero_group_set_loss_scaler_state",
                 "zero_group_set_lr", "zero_group_free", "zero_group_accumulate",
                 "zero_group_step_accumulated", "zero_group_step_q8",
                 "zero_group_step_offload",
                 "zero_shard_step_accumulated"):
        getattr(L, name).restype = i32
    return L


_lib = _load()


def _check(status, where):
    if status != ZERO_OK:
        raise ZeroError(status, where)


def hparams(lr=3e-5, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, max_grad_norm=1.0,
            dynamic=True, initial_scale_power=16, window=1000, static_scale=1.0,
            min_scale=1.0):
    """Settings named after the DeepSpeed config keys (defaults: the AdamW,
    fp16 dynamic loss-scale and gradient_clipping values of the config printed
    in the ZeRO paper reading, §5.1)."""
    return Hparams(lr, beta1, beta2, eps, weight_decay, max_grad_norm, 1 if dynamic else 0,
                   initial_scale_power, window, 0, static_scale, min_scale)


def param_infos(shapes, dtype=ZERO_F16):
    """The FlatParameter's parameter table for parameters of the given shapes,
    concatenated in order."""
    arr = (ParamInfo * len(shapes))()
    off = 0
    for k, shp in enumerate(shapes):
        shp = tuple(int(d) for d in shp)
        numel = 1
        for d in shp:
            numel *= d
        arr[k].offset = off
        arr[k].numel = numel
        arr[k].ndim = len(shp)
        arr[k].dtype = dtype
        for d, x in enumerate(shp):
            arr[k].shape[d] = x
        off += numel
    return arr


def zero_flat_init(infos, world_size, grad_dtype, param_dtype, op, hp):
    h = C.c_void_p()
    _check(_lib.zero_flat_init(infos, len(infos), world_size, grad_dtype, param_dtype, op,
                               C.byref(hp), C.byref(h)), "zero_flat_init")
    return h


def zero_flat_layout(h):
    out = [C.c_int64() for _ in range(3)]
    _check(_lib.zero_flat_layout(h, *[C.byref(o) for o in out]), "zero_flat_layout")
    return tuple(o.value for o in out)


def zero_shard_step(h, ranks, grads_ptr, grad_ld, grad_rank_offset_mul, master_ptrs,
                    m_ptrs, v_ptrs, out_ptr, extra_norm_sq=0.0, stream=0, want_result=True):
    """Raw pointers in, status checked.  Returns a StepResult (synchronizes
    the stream) when want_result, else None (fully asynchronous)."""
    n = len(ranks)
    r = (C.c_int32 * n)(*ranks)
    mp = (C.c_void_p * n)(*master_ptrs)
    mm = (C.c_void_p * n)(*m_ptrs)
    vv = (C.c_void_p * n)(*v_ptrs)
    res = StepResult() if want_result else None
    _check(_lib.zero_shard_step(h, r, n, C.c_void_p(grads_ptr), grad_ld, grad_rank_offset_mul,
                                mp, mm, vv, C.c_void_p(out_ptr), float(extra_norm_sq),
                                C.c_void_p(stream), C.byref(res) if res is not None else None),
           "zero_shard_step")
    return res


def zero_shard_step_noalloc(full_numel, world_size, grad_dtype, param_dtype, op, hp, state,
                            ranks, grads_ptr, grad_ld, grad_rank_offset_mul, master_ptrs,
                            m_ptrs, v_ptrs, out_ptr, extra_norm_sq=0.0, stream=0):
    """The shard step without a handle and without any allocation, for
    callers that must not allocate device memory (see include/zero.h).
    `state` is a ScalerState in host memory, updated in place; returns the
    StepResult.  Synchronous."""
    n = len(ranks)
    r = (C.c_int32 * n)(*ranks)
    mp = (C.c_void_p * n)(*master_ptrs)
    mm = (C.c_void_p * n)(*m_ptrs)
    vv = (C.c_void_p * n)(*v_ptrs)
    res = StepResult()
    _check(_lib.zero_shard_step_noalloc(full_numel, world_size, grad_dtype, param_dtype, op,
                                        C.byref(hp), C.byref(state), r, n, C.c_void_p(grads_ptr),
                                        grad_ld, grad_rank_offset_mul, mp, mm, vv,
                                        C.c_void_p(out_ptr), float(extra_norm_sq),
                                        C.c_void_p(stream), C.byref(res)),
           "zero_shard_step_noalloc")
    return res


def zero_shard_step_q8(h, ranks, grads_ptr, grad_ld, grad_rank_offset_mul, master_ptrs,
                       m_ptrs, v_ptrs, out_ptr, q8_ptr, scales_ptr, extra_norm_sq=0.0,
                       stream=0, want_result=True):
    """zero_shard_step that also writes the int8 all-gather payload (codes +
    one fp32 scale per 256 elements); out_ptr may be 0."""
    n = len(ranks)
    r = (C.c_int32 * n)(*ranks)
    arrs = [(C.c_void_p * n)(*p) for p in (master_ptrs, m_ptrs, v_ptrs)]
    res = StepResult() if want_result else None
    _check(_lib.zero_shard_step_q8(h, r, n, C.c_void_p(grads_ptr), grad_ld, grad_rank_offset_mul,
                                   *arrs, C.c_void_p(out_ptr or None), C.c_void_p(q8_ptr),
                                   C.c_void_p(scales_ptr), float(extra_norm_sq),
                                   C.c_void_p(stream), C.byref(res) if res is not None else None),
           "zero_shard_step_q8")
    return res


def zero_grad_accumulate(h, ranks, grads_ptr, grad_ld, grad_rank_offset_mul, acc_ptrs,
                         first_micro_step, stream=0):
    """acc[j] = reduce(contributions) on the first micro-step, else
    acc[j] + reduce(contributions).  Asynchronous."""
    n = len(ranks)
    r = (C.c_int32 * n)(*ranks)
    aa = (C.c_void_p * n)(*acc_ptrs)
    _check(_lib.zero_grad_accumulate(h, r, n, C.c_void_p(grads_ptr), grad_ld,
                                     grad_rank_offset_mul, aa, 1 if first_micro_step else 0,
                                     C.c_void_p(stream)), "zero_grad_accumulate")


def zero_shard_step_accumulated(h, ranks, acc_ptrs, master_ptrs, m_ptrs, v_ptrs, out_ptr,
                                extra_norm_sq=0.0, stream=0, want_result=True):
    """The optimizer step on accumulated fp32 shards (g = acc / loss scale)."""
    n = len(ranks)
    r = (C.c_int32 * n)(*ranks)
    arrs = [(C.c_void_p * n)(*p) for p in (acc_ptrs, master_ptrs, m_ptrs, v_ptrs)]
    res = StepResult() if want_result else None
    _check(_lib.zero_shard_step_accumulated(h, r, n, *arrs, C.c_void_p(out_ptr),
                                            float(extra_norm_sq), C.c_void_p(stream),
                                            C.byref(res) if res is not None else None),
           "zero_shard_step_accumulated")
    return res


def zero_shard_step_offload(h, ranks, grads_ptr, grad_ld, grad_rank_offset_mul, master_ptrs,
                            m_ptrs, v_ptrs, out_ptr, extra_norm_sq=0.0, n_threads=0,
                            gpu_share=0.0, stream=0, want_result=True):
    """The offload step: master/m/v pointers are HOST memory; the GPU updates
    the first gpu_share of each shard over the host link, the host threads the
    rest.  Returns a StepResult when want_result."""
    n = len(ranks)
    r = (C.c_int32 * n)(*ranks)
    arrs = [(C.c_void_p * n)(*p) for p in (master_ptrs, m_ptrs, v_ptrs)]
    res = StepResult() if want_result else None
    _check(_lib.zero_shard_step_offload(h, r, n, C.c_void_p(grads_ptr), grad_ld,
                                        grad_rank_offset_mul, *arrs, C.c_void_p(out_ptr),
                                        float(extra_norm_sq), int(n_threads), float(gpu_share),
                                        C.c_void_p(stream),
                                        C.byref(res) if res is not None else None),
           "zero_shard_step_offload")
    return res


def zero_offload_adamw_host(hp, step_t, clip_coef, g_ptr, master_ptr, m_ptr, v_ptr, out_ptr, n,
                            param_dtype=ZERO_F16, n_threads=0):
    """The host AdamW + 16-bit cast of the offload step on n elements of host
    arrays (no GPU involved)."""
    _check(_lib.zero_offload_adamw_host(C.byref(hp), int(step_t), C.c_float(clip_coef),
                                        C.c_void_p(g_ptr), C.c_void_p(master_ptr),
                                        C.c_void_p(m_ptr), C.c_void_p(v_ptr), C.c_void_p(out_ptr),
                                        int(n), int(param_dtype), int(n_threads)),
           "zero_offload_adamw_host")


def zero_shard_reduce(h, ranks, grads_ptr, grad_ld, grad_rank_offset_mul, norm_sq_ptr,
                      overflow_ptr, stream=0):
    """First half of a split step: device totals of this handle's norm^2 and
    overflow flag."""
    n = len(ranks)
    r = (C.c_int32 * n)(*ranks)
    _check(_lib.zero_shard_reduce(h, r, n, C.c_void_p(grads_ptr), grad_ld, grad_rank_offset_mul,
                                  C.c_void_p(norm_sq_ptr), C.c_void_p(overflow_ptr),
                                  C.c_void_p(stream)), "zero_shard_reduce")


def zero_shard_apply(h, ranks, master_ptrs, m_ptrs, v_ptrs, out_ptr, norm_sq_ptr, overflow_ptr,
                     stream=0, want_result=True):
    """Second half: the decision from the summed device totals, then AdamW."""
    n = len(ranks)
    r = (C.c_int32 * n)(*ranks)
    arrs = [(C.c_void_p * n)(*p) for p in (master_ptrs, m_ptrs, v_ptrs)]
    res = StepResult() if want_result else None
    _check(_lib.zero_shard_apply(h, r, n, *arrs, C.c_void_p(out_ptr), C.c_void_p(norm_sq_ptr),
                                 C.c_void_p(overflow_ptr), C.c_void_p(stream),
                                 C.byref(res) if res is not None else None), "zero_shard_apply")
    return res


def zero_shard_apply_partials(h, ranks, master_ptrs, m_ptrs, v_ptrs, out_ptr, norm_sq_parts_ptr,
                              overflow_parts_ptr, n_parts, stream=0, want_result=True):
    """Second half from n_parts per-rank partials (device fp64 norm^2 and
    int32 flags, e.g. all-gathered), totalled on the device; then AdamW."""
    n = len(ranks)
    r = (C.c_int32 * n)(*ranks)
    arrs = [(C.c_void_p * n)(*p) for p in (master_ptrs, m_ptrs, v_ptrs)]
    res = StepResult() if want_result else None
    _check(_lib.zero_shard_apply_partials(h, r, n, *arrs, C.c_void_p(out_ptr),
                                          C.c_void_p(norm_sq_parts_ptr),
                                          C.c_void_p(overflow_parts_ptr), n_parts,
                                          C.c_void_p(stream),
                                          C.byref(res) if res is not None else None),
           "zero_shard_apply_partials")
    return res


def zero_shard_reduce_accumulated(h, ranks, acc_ptrs, norm_sq_ptr, overflow_ptr, stream=0):
    """First half of a split step from micro-step accumulators: g = acc / scale
    into the handle's rows, this handle's norm^2 and overflow flag on the device."""
    n = len(ranks)
    r = (C.c_int32 * n)(*ranks)
    _check(_lib.zero_shard_reduce_accumulated(h, r, n, (C.c_void_p * n)(*acc_ptrs),
                                              C.c_void_p(norm_sq_ptr), C.c_void_p(overflow_ptr),
                                              C.c_void_p(stream)),
           "zero_shard_reduce_accumulated")


def zero_shard_apply_partials_q8(h, ranks, master_ptrs, m_ptrs, v_ptrs, out_ptr, q8_ptr,
                                 q8_scales_ptr, norm_sq_parts_ptr, overflow_parts_ptr, n_parts,
                                 stream=0, want_result=True):
    """zero_shard_apply_partials that also writes the int8 payload (out_ptr may be 0)."""
    n = len(ranks)
    r = (C.c_int32 * n)(*ranks)
    arrs = [(C.c_void_p * n)(*p) for p in (master_ptrs, m_ptrs, v_ptrs)]
    res = StepResult() if want_result else None
    _check(_lib.zero_shard_apply_partials_q8(h, r, n, *arrs, C.c_void_p(out_ptr or None),
                                             C.c_void_p(q8_ptr), C.c_void_p(q8_scales_ptr),
                                             C.c_void_p(norm_sq_parts_ptr),
                                             C.c_void_p(overflow_parts_ptr), n_parts,
                                             C.c_void_p(stream),
                                             C.byref(res) if res is not None else None),
           "zero_shard_apply_partials_q8")
    return res


def zero_group_init(handles):
    """A group over the given handles (raw zero_flat pointers)."""
    arr = (C.c_void_p * len(handles))(*handles)
    g = C.c_void_p()
    _check(_lib.zero_group_init(arr, len(handles), C.byref(g)), "zero_group_init")
    return g.value


def _group_call(name, g, members, *args, want_result=True):
    res = StepResult() if want_result else None
    _check(getattr(_lib, name)(g, members, *args, C.byref(res) if res is not None else None), name)
    return res


def zero_group_step(g, members, extra_norm_sq=0.0, stream=0, want_result=True):
    """members: a GroupMember array, one entry per member of the group."""
    return _group_call("zero_group_step", g, members, float(extra_norm_sq), C.c_void_p(stream),
                       want_result=want_result)


def zero_group_step_q8(g, members, extra_norm_sq=0.0, stream=0, want_result=True):
    return _group_call("zero_group_step_q8", g, members, float(extra_norm_sq),
                       C.c_void_p(stream), want_result=want_result)


def zero_group_step_accumulated(g, members, extra_norm_sq=0.0, stream=0, want_result=True):
    return _group_call("zero_group_step_accumulated", g, members, float(extra_norm_sq),
                       C.c_void_p(stream), want_result=want_result)


def zero_group_step_offload(g, members, extra_norm_sq=0.0, n_threads=0, gpu_share=0.0,
                            stream=0):
    return _group_call("zero_group_step_offload", g, members, float(extra_norm_sq),
                       int(n_threads), float(gpu_share), C.c_void_p(stream))


def zero_group_accumulate(g, members, first_micro_step, stream=0):
    _check(_lib.zero_group_accumulate(g, members, 1 if first_micro_step else 0,
                                      C.c_void_p(stream)), "zero_group_accumulate")


def zero_group_loss_scaler_state(g, stream=0):
    st = ScalerState()
    _check(_lib.zero_group_loss_scaler_state(g, C.byref(st), C.c_void_p(stream)),
           "zero_group_loss_scaler_state")
    return st


def zero_group_set_loss_scaler_state(g, state, stream=0):
    _check(_lib.zero_group_set_loss_scaler_state(g, C.byref(state), C.c_void_p(stream)),
           "zero_group_set_loss_scaler_state")


def zero_group_set_lr(g, lr):
    _check(_lib.zero_group_set_lr(g, float(lr)), "zero_group_set_lr")


def zero_group_free(g):
    _check(_lib.zero_group_free(g), "zero_group_free")


class ZeroGroup:
    """FlatParameters of one rank stepped together with one global decision.

    members: ZeroFlat objects sharing world size, dtypes, op and every
    hyper-parameter but lr and weight_decay (each member keeps its own).
    step(args): args[k] = dict(ranks, grads, master, m, v, out[, grad_rank_offset_mul])
    for member k, torch CUDA tensors as for ZeroFlat.step; accumulate() and
    step_accumulated() take acc (fp32 rows, one per stepped rank) as for
    ZeroFlat.accumulate and ZeroFlat.step_accumulated; step_q8() takes q8 and
    q8_scales as ZeroFlat.step_q8; step_offload() takes host master/m/v."""

    def __init__(self, members):
        self.members = list(members)
        self.handle = zero_group_init([f.handle for f in self.members])

    def _members(self, args, keep):
        """The GroupMember array of args (ctypes arrays appended to keep)."""
        ms = (GroupMember * len(args))()
        for k, (f, a) in enumerate(zip(self.members, args)):
            ranks = list(a["ranks"])
            r = (C.c_int32 * len(ranks))(*ranks)
            keep.append(r)
            x = GroupMember()
            x.ranks, x.n_ranks = r, len(ranks)
            g = a.get("grads")
            if g is not None:
                assert g.dim() == 2 and g.stride(1) == 1
                mul = a.get("grad_rank_offset_mul")
                if mul is None:
                    mul = f.shard_size if len(ranks) > 1 else 0
                x.grads, x.grad_ld, x.grad_rank_offset_mul = g.data_ptr(), g.stride(0), mul
            for name in ("master", "m", "v", "acc"):
                if a.get(name) is not None:
                    arr = (C.c_void_p * len(ranks))(*[t.data_ptr() for t in a[name]])
                    keep.append(arr)
                    setattr(x, name, arr)
            if a.get("out") is not None:
                x.flat_param_out = a["out"].data_ptr()
            if a.get("q8") is not None:
                x.flat_q8_out = a["q8"].data_ptr()
            if a.get("q8_scales") is not None:
                x.q8_scales = a["q8_scales"].data_ptr()
            ms[k] = x
        return ms

    @staticmethod
    def _stream(stream):
        import torch
        return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream

    def step(self, args, extra_norm_sq=0.0, stream=None, want_result=True):
        keep = []                                   # ctypes arrays alive for the call
        return zero_group_step(self.handle, self._members(args, keep), extra_norm_sq,
                               self._stream(stream), want_result)

    def step_q8(self, args, extra_norm_sq=0.0, stream=None, want_result=True):
        """The group step that also writes every member's int8 payload (out may
        be None)."""
        keep = []
        return zero_group_step_q8(self.handle, self._members(args, keep), extra_norm_sq,
                                  self._stream(stream), want_result)

    def step_offload(self, args, extra_norm_sq=0.0, n_threads=0, gpu_share=0.0, stream=None):
        """The ZeRO-Offload group step: master, m, v host (CPU, pinned for
        gpu_share > 0) fp32 tensors, updated when it returns."""
        keep = []
        return zero_group_step_offload(self.handle, self._members(args, keep), extra_norm_sq,
                                       n_threads, gpu_share, self._stream(stream))

    def accumulate(self, args, first_micro_step, stream=None):
        """One micro-step: args[k] = dict(ranks, grads, acc[, grad_rank_offset_mul]);
        each member's reduced micro-step gradient (loss scale not divided out)
        written (first) or added into its fp32 accumulator rows acc[j], one per
        stepped rank.  One launch per 64 rows of all members."""
        keep = []
        zero_group_accumulate(self.handle, self._members(args, keep), first_micro_step,
                              self._stream(stream))

    def step_accumulated(self, args, extra_norm_sq=0.0, stream=None, want_result=True):
        """The group step from accumulators: args[k] = dict(ranks, acc, master, m, v, out)."""
        keep = []
        return zero_group_step_accumulated(self.handle, self._members(args, keep),
                                           extra_norm_sq, self._stream(stream), want_result)

    def scaler_state(self, stream=None):
        return zero_group_loss_scaler_state(self.handle, self._stream(stream))

    def set_scaler_state(self, state, stream=None):
        """Restore the group's loss-scale state (scale, counter, step)."""
        zero_group_set_loss_scaler_state(self.handle, state, self._stream(stream))

    def set_lr(self, lr):
        """Set lr on every member (each keeps its weight decay)."""
        zero_group_set_lr(self.handle, lr)

    def close(self):
        if getattr(self, "handle", None):
            zero_group_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def zero_debug_set_stage_tx_pad(nbytes):
    """Test hook: the staged reduce's waits run out (see include/zero_debug.h)."""
    _check(_lib.zero_debug_set_stage_tx_pad(int(nbytes)), "zero_debug_set_stage_tx_pad")


def zero_debug_reduce_form(grad_dtype, n_contrib, rows, mode=0):
    """The planner's reduce for rows [(contribution address, row stride in
    elements, shard size[, accumulator address]), ...]: "staged" or "plain".
    Host logic only (no GPU, nothing dereferenced); mode 0 step, 1 first
    micro-step, 2 later micro-step."""
    n = len(rows)
    ins = (C.c_uint64 * n)(*[int(r[0]) for r in rows])
    lds = (C.c_int64 * n)(*[int(r[1]) for r in rows])
    ss = (C.c_int64 * n)(*[int(r[2]) for r in rows])
    accs = (C.c_uint64 * n)(*[int(r[3]) if len(r) > 3 else 0 for r in rows]) if mode else None
    out = C.c_int32()
    _check(_lib.zero_debug_reduce_form(grad_dtype, n_contrib, n, ins, lds, ss, accs, mode,
                                       C.byref(out)), "zero_debug_reduce_form")
    return "staged" if out.value else "plain"


def zero_flat_set_lr(h, lr):
    """Learning rate of the steps launched from now on."""
    _check(_lib.zero_flat_set_lr(h, float(lr)), "zero_flat_set_lr")


def zero_loss_scaler_state(h, stream=0):
    st = ScalerState()
    _check(_lib.zero_loss_scaler_state(h, C.byref(st), C.c_void_p(stream)),
           "zero_loss_scaler_state")
    return st


def zero_set_loss_scaler_state(h, state, stream=0):
    _check(_lib.zero_set_loss_scaler_state(h, C.byref(state), C.c_void_p(stream)),
           "zero_set_loss_scaler_state")


def zero_memory_bytes(stage, psi, world_size):
    """(total, params, grads, optimizer) bytes per GPU."""
    out = [C.c_uint64() for _ in range(4)]
    _check(_lib.zero_memory_bytes(stage, psi, world_size, *[C.byref(o) for o in out]),
           "zero_memory_bytes")
    return tuple(o.value for o in out)


def zero_flat_device_bytes(h):
    b = C.c_uint64()
    _check(_lib.zero_flat_device_bytes(h, C.byref(b)), "zero_flat_device_bytes")
    return b.value


def zero_flat_free(h):
    _check(_lib.zero_flat_free(h), "zero_flat_free")


def zero_flat_profile_enable(h, enable=True):
    _check(_lib.zero_flat_profile_enable(h, 1 if enable else 0), "zero_flat_profile_enable")


def zero_flat_profile_read(h):
    """(ms_reduce, ms_finalize, ms_adamw, steps) summed since the last read."""
    t = [C.c_double() for _ in range(3)]
    n = C.c_int64()
    _check(_lib.zero_flat_profile_read(h, *[C.byref(x) for x in t], C.byref(n)),
           "zero_flat_profile_read")
    return t[0].value, t[1].value, t[2].value, n.value


def zero_flat_profile_reduce_form(h):
    """The last contribution reduce's kernel: "staged", "plain", or None
    before the first."""
    v = C.c_int32()
    _check(_lib.zero_flat_profile_reduce_form(h, C.byref(v)), "zero_flat_profile_reduce_form")
    return {1: "staged", 0: "plain"}.get(v.value)


def zero_status_string(status):
    return _lib.zero_status_string(status).decode()


def zero_last_error():
    return _lib.zero_last_error().decode()


class ZeroFlat:
    """Owns a handle; steps torch CUDA tensors through the C ABI.

    grads: 2-D 16-bit CUDA tensor [world_size, ld] (row stride ld); master, m,
    v: lists of fp32 CUDA tensors, one per stepped rank; out: 1-D 16-bit CUDA
    tensor of padded_numel elements.
    """

    def __init__(self, shapes_or_infos, world_size, grad_dtype=ZERO_F16, param_dtype=None,
                 op=ZERO_AVG, hp=None):
        if param_dtype is None:
            param_dtype = grad_dtype if grad_dtype != ZERO_F32 else ZERO_F16
        infos = (shapes_or_infos if isinstance(shapes_or_infos, C.Array)
                 else param_infos(shapes_or_infos, param_dtype))
        self.hp = hp if hp is not None else hparams()
        self.world_size = world_size
        self.grad_dtype, self.param_dtype, self.op = grad_dtype, param_dtype, op
        self.handle = zero_flat_init(infos, world_size, grad_dtype, param_dtype, op, self.hp)
        self.full_numel, self.shard_size, self.padded_numel = zero_flat_layout(self.handle)

    def reduce_form(self):
        """The kernel of the last contribution reduce: "staged", "plain" or None."""
        return zero_flat_profile_reduce_form(self.handle)

    def step(self, ranks, grads, master, m, v, out, grad_rank_offset_mul=None,
             extra_norm_sq=0.0, stream=None, want_result=True):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        assert grads.dim() == 2 and grads.stride(1) == 1
        if grad_rank_offset_mul is None:
            grad_rank_offset_mul = self.shard_size if len(ranks) > 1 else 0
        return zero_shard_step(self.handle, list(ranks), grads.data_ptr(), grads.stride(0),
                               grad_rank_offset_mul, [t.data_ptr() for t in master],
                               [t.data_ptr() for t in m], [t.data_ptr() for t in v],
                               out.data_ptr(), extra_norm_sq, stream.cuda_stream, want_result)

    def step_q8(self, ranks, grads, master, m, v, out, q8, q8_scales, grad_rank_offset_mul=None,
                extra_norm_sq=0.0, stream=None, want_result=True):
        """Step and write the int8 payload: q8 int8 [padded_numel], q8_scales
        float32 [world_size * ceil(shard_size / 256)]; out may be None."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        if grad_rank_offset_mul is None:
            grad_rank_offset_mul = self.shard_size if len(ranks) > 1 else 0
        return zero_shard_step_q8(self.handle, list(ranks), grads.data_ptr(), grads.stride(0),
                                  grad_rank_offset_mul, [t.data_ptr() for t in master],
                                  [t.data_ptr() for t in m], [t.data_ptr() for t in v],
                                  out.data_ptr() if out is not None else 0, q8.data_ptr(),
                                  q8_scales.data_ptr(), extra_norm_sq, stream.cuda_stream,
                                  want_result)

    def accumulate(self, ranks, grads, acc, first_micro_step, grad_rank_offset_mul=None,
                   stream=None):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        assert grads.dim() == 2 and grads.stride(1) == 1
        if grad_rank_offset_mul is None:
            grad_rank_offset_mul = self.shard_size if len(ranks) > 1 else 0
        zero_grad_accumulate(self.handle, list(ranks), grads.data_ptr(), grads.stride(0),
                             grad_rank_offset_mul, [t.data_ptr() for t in acc],
                             first_micro_step, stream.cuda_stream)

    def step_accumulated(self, ranks, acc, master, m, v, out, extra_norm_sq=0.0, stream=None,
                         want_result=True):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        return zero_shard_step_accumulated(self.handle, list(ranks), [t.data_ptr() for t in acc],
                                           [t.data_ptr() for t in master],
                                           [t.data_ptr() for t in m], [t.data_ptr() for t in v],
                                           out.data_ptr(), extra_norm_sq, stream.cuda_stream,
                                           want_result)

    def step_offload(self, ranks, grads, master, m, v, out, grad_rank_offset_mul=None,
                     extra_norm_sq=0.0, n_threads=0, gpu_share=0.0, stream=None,
                     want_result=True):
        """The ZeRO-Offload step: master, m, v are fp32 CPU tensors (pinned,
        or pageable when gpu_share is 0 or the device reads pageable memory);
        grads and out are CUDA tensors as for step().  gpu_share: the fraction
        of each shard the GPU updates over the host link."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        assert grads.dim() == 2 and grads.stride(1) == 1
        for t in list(master) + list(m) + list(v):
            assert t.device.type == "cpu" and t.dtype == torch.float32 and t.is_contiguous()
        if grad_rank_offset_mul is None:
            grad_rank_offset_mul = self.shard_size if len(ranks) > 1 else 0
        return zero_shard_step_offload(self.handle, list(ranks), grads.data_ptr(),
                                       grads.stride(0), grad_rank_offset_mul,
                                       [t.data_ptr() for t in master], [t.data_ptr() for t in m],
                                       [t.data_ptr() for t in v], out.data_ptr(), extra_norm_sq,
                                       n_threads, gpu_share, stream.cuda_stream, want_result)

    def reduce(self, ranks, grads, norm_sq, overflow, grad_rank_offset_mul=None, stream=None):
        """First half of a split step; norm_sq: float64 CUDA scalar tensor,
        overflow: int32 CUDA scalar tensor (both written)."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        assert grads.dim() == 2 and grads.stride(1) == 1
        if grad_rank_offset_mul is None:
            grad_rank_offset_mul = self.shard_size if len(ranks) > 1 else 0
        zero_shard_reduce(self.handle, list(ranks), grads.data_ptr(), grads.stride(0),
                          grad_rank_offset_mul, norm_sq.data_ptr(), overflow.data_ptr(),
                          stream.cuda_stream)

    def reduce_accumulated(self, ranks, acc, norm_sq, overflow, stream=None):
        """First half of a split step from fp32 accumulators (one CUDA tensor
        of shard_size per stepped rank)."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        zero_shard_reduce_accumulated(self.handle, list(ranks), [t.data_ptr() for t in acc],
                                      norm_sq.data_ptr(), overflow.data_ptr(), stream.cuda_stream)

    def apply(self, ranks, master, m, v, out, norm_sq, overflow, stream=None, want_result=True):
        """Second half: the decision from the (summed) totals, then AdamW."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        return zero_shard_apply(self.handle, list(ranks), [t.data_ptr() for t in master],
                                [t.data_ptr() for t in m], [t.data_ptr() for t in v],
                                out.data_ptr(), norm_sq.data_ptr(), overflow.data_ptr(),
                                stream.cuda_stream, want_result)

    def apply_partials(self, ranks, master, m, v, out, norm_sq_parts, overflow_parts,
                       stream=None, want_result=True, q8=None, q8_scales=None):
        """Second half from per-rank partials: norm_sq_parts float64 and
        overflow_parts int32 CUDA tensors of equal length.  q8 / q8_scales:
        also write the int8 payload (out may then be None)."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        assert norm_sq_parts.numel() == overflow_parts.numel()
        assert norm_sq_parts.is_contiguous() and overflow_parts.is_contiguous()
        ptrs = ([t.data_ptr() for t in master], [t.data_ptr() for t in m],
                [t.data_ptr() for t in v])
        if q8 is not None:
            return zero_shard_apply_partials_q8(
                self.handle, list(ranks), *ptrs, out.data_ptr() if out is not None else 0,
                q8.data_ptr(), q8_scales.data_ptr(), norm_sq_parts.data_ptr(),
                overflow_parts.data_ptr(), norm_sq_parts.numel(), stream.cuda_stream,
                want_result)
        return zero_shard_apply_partials(self.handle, list(ranks), *ptrs, out.data_ptr(),
                                         norm_sq_parts.data_ptr(), overflow_parts.data_ptr(),
                                         norm_sq_parts.numel(), stream.cuda_stream, want_result)

    def set_lr(self, lr):
        zero_flat_set_lr(self.handle, lr)
        self.hp.lr = lr

    def scaler_state(self, stream=None):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        return zero_loss_scaler_state(self.handle, s.cuda_stream)

    def set_scaler_state(self, state, stream=None):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        zero_set_loss_scaler_state(self.handle, state, s.cuda_stream)

    def device_bytes(self):
        return zero_flat_device_bytes(self.handle)

    def close(self):
        if self.handle is not None:
            zero_flat_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
