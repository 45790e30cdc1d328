// zero_api.cu -- host side of the C ABI declared in include/zero.h: argument
// validation, the flat-parameter layout, device state, scratch management and
// the launches of a step (the reduce, whose last block makes the step's
// decision, and the AdamW), and the offload step's host half.  No arithmetic of the update happens here
// beyond forming the per-step fp32 scalars from the fp64 hyper-parameters.
#include "zero_handle.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <new>
#include <vector>

using namespace zi;

namespace zi {

thread_local char g_last_error[512] = "";

zero_status fail(zero_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return s;
}

zero_status cuda_fail(cudaError_t e, const char *what) {
    return fail(ZERO_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Bias-correction table: entry t = {(float)(1 - b1^t), (float)(1 - b2^t)} with
// pow in fp64, for t = 0 .. until both round to 1.0f (from there on they stay
// 1.0f, which the finalize kernel uses past the end of the table).
zero_status build_bc_table(zero_flat *h) {
    const int64_t kCap = int64_t(1) << 24;
    std::vector<float2> tab;
    tab.reserve(1 << 15);
    for (int64_t t = 0;; ++t) {
        if (t >= kCap)
            return fail(ZERO_ERR_INVALID_ARG,
                        "betas too close to 1: bias corrections do not reach 1.0f within 2^24 steps");
        const float c1 = (float)(1.0 - std::pow(h->hp.beta1, (double)t));
        const float c2 = (float)(1.0 - std::pow(h->hp.beta2, (double)t));
        tab.push_back(make_float2(c1, c2));
        if (t > 0 && c1 == 1.0f && c2 == 1.0f) break;
    }
    h->bc_len = (int64_t)tab.size();
    const size_t bytes = tab.size() * sizeof(float2);
    cudaError_t e = cudaMalloc(&h->d_bc, bytes);
    if (e) return cuda_fail(e, "cudaMalloc(bias-correction table)");
    h->device_bytes += bytes;
    e = cudaMemcpy(h->d_bc, tab.data(), bytes, cudaMemcpyHostToDevice);
    if (e) return cuda_fail(e, "cudaMemcpy(bias-correction table)");
    return ZERO_OK;
}

// The loss-scale state of a new handle (scale from the hyper-parameters), the
// block counter, the pinned read-back block and the bias-correction table.
zero_status init_device_state(zero_flat *h) {
    zg::DevState init{};
    init.scaler.scale = h->hp.dynamic_loss_scale ? (float)std::ldexp(1.0, h->hp.initial_scale_power)
                                                 : (float)h->hp.static_loss_scale;
    init.bc1 = init.bc2 = 1.0f;
    cudaError_t e = cudaMalloc(&h->d_state, sizeof(zg::DevState));
    if (e) { h->d_state = nullptr; return cuda_fail(e, "cudaMalloc(state)"); }
    h->device_bytes += sizeof(zg::DevState);
    e = cudaMemcpy(h->d_state, &init, sizeof(init), cudaMemcpyHostToDevice);
    if (e) return cuda_fail(e, "cudaMemcpy(state)");
    e = cudaMalloc(&h->d_done, sizeof(uint32_t));
    if (e) { h->d_done = nullptr; return cuda_fail(e, "cudaMalloc(block counter)"); }
    e = cudaMemset(h->d_done, 0, sizeof(uint32_t));
    if (e) return cuda_fail(e, "cudaMemset(block counter)");
    h->device_bytes += sizeof(uint32_t);
    e = cudaMallocHost(&h->h_state, sizeof(zg::DevState));
    if (e) { h->h_state = nullptr; return cuda_fail(e, "cudaMallocHost(state)"); }
    return build_bc_table(h);
}

zero_status validate_hparams(const zero_hparams *hp) {
    if (!hp) return fail(ZERO_ERR_INVALID_ARG, "hparams is NULL");
    auto finite = [](double x) { return std::isfinite(x); };
    if (!finite(hp->lr) || hp->lr < 0) return fail(ZERO_ERR_INVALID_ARG, "lr must be finite and >= 0");
    if (!finite(hp->beta1) || hp->beta1 < 0 || hp->beta1 >= 1)
        return fail(ZERO_ERR_INVALID_ARG, "beta1 must be in [0, 1)");
    if (!finite(hp->beta2) || hp->beta2 < 0 || hp->beta2 >= 1)
        return fail(ZERO_ERR_INVALID_ARG, "beta2 must be in [0, 1)");
    if (!finite(hp->eps) || hp->eps <= 0) return fail(ZERO_ERR_INVALID_ARG, "eps must be > 0");
    if (!finite(hp->weight_decay) || hp->weight_decay < 0)
        return fail(ZERO_ERR_INVALID_ARG, "weight_decay must be >= 0");
    if (!finite(hp->max_grad_norm)) return fail(ZERO_ERR_INVALID_ARG, "max_grad_norm must be finite");
    if (hp->dynamic_loss_scale != 0 && hp->dynamic_loss_scale != 1)
        return fail(ZERO_ERR_INVALID_ARG, "dynamic_loss_scale must be 0 or 1");
    if (hp->initial_scale_power < 0 || hp->initial_scale_power > 126)
        return fail(ZERO_ERR_INVALID_ARG, "initial_scale_power must be in [0, 126]");
    if (hp->loss_scale_window < 1) return fail(ZERO_ERR_INVALID_ARG, "loss_scale_window must be >= 1");
    if (hp->reserved != 0) return fail(ZERO_ERR_INVALID_ARG, "reserved must be 0");
    if (!hp->dynamic_loss_scale &&
        (!finite(hp->static_loss_scale) || hp->static_loss_scale <= 0 ||
         !std::isfinite((float)hp->static_loss_scale) || (float)hp->static_loss_scale <= 0))
        return fail(ZERO_ERR_INVALID_ARG, "static_loss_scale must be a positive fp32 value");
    if (!finite(hp->min_loss_scale) || hp->min_loss_scale <= 0 || (float)hp->min_loss_scale <= 0)
        return fail(ZERO_ERR_INVALID_ARG, "min_loss_scale must be > 0");
    return ZERO_OK;
}

zero_status ensure_scratch(zero_flat *h, int64_t rows, int64_t parts) {
    if (rows > h->g_rows) {
        int64_t bytes;
        if (!mul_ok(rows, h->g_stride, &bytes) || !mul_ok(bytes, 4, &bytes))
            return fail(ZERO_ERR_OVERFLOW_SIZE, "scratch size overflows");
        if (h->d_g) {
            cudaFree(h->d_g);
            h->device_bytes -= (uint64_t)(h->g_rows * h->g_stride * 4);
            h->d_g = nullptr;
            h->g_rows = 0;
        }
        if (bytes > 0) {
            cudaError_t e = cudaMalloc(&h->d_g, (size_t)bytes);
            if (e == cudaErrorMemoryAllocation) {
                cudaGetLastError();
                return fail(ZERO_ERR_NO_MEMORY, "cannot allocate %lld bytes of gradient scratch",
                            (long long)bytes);
            }
            if (e) return cuda_fail(e, "cudaMalloc(gradient scratch)");
        }
        h->g_rows = rows;
        h->device_bytes += (uint64_t)bytes;
    }
    if (parts > h->parts_cap) {
        if (h->d_part_ss) cudaFree(h->d_part_ss);
        if (h->d_part_of) cudaFree(h->d_part_of);
        h->device_bytes -= (uint64_t)(h->parts_cap * 12);
        h->d_part_ss = nullptr;
        h->d_part_of = nullptr;
        h->parts_cap = 0;
        cudaError_t e = cudaMalloc(&h->d_part_ss, (size_t)parts * sizeof(double));
        if (!e) e = cudaMalloc(&h->d_part_of, (size_t)parts * sizeof(int32_t));
        if (e) return cuda_fail(e, "cudaMalloc(norm partials)");
        h->parts_cap = parts;
        h->device_bytes += (uint64_t)(parts * 12);
    }
    return ZERO_OK;
}

// Next free event of the timing record (created on demand, reused).
cudaError_t next_event(zero_flat *h, cudaEvent_t *out) {
    if (h->ev_used == h->ev.size()) {
        cudaEvent_t e;
        cudaError_t err = cudaEventCreate(&e);
        if (err) return err;
        h->ev.push_back(e);
    }
    *out = h->ev[h->ev_used++];
    return cudaSuccess;
}

cudaError_t mark(zero_flat *h, cudaStream_t s) {
    if (!h->profile) return cudaSuccess;
    cudaEvent_t e;
    cudaError_t err = next_event(h, &e);
    if (err) return err;
    return cudaEventRecord(e, s);
}

void release(zero_flat *h) {
    if (!h) return;
    DeviceGuard g(h->device);
    h->pool.reset();
    if (h->out_done) {
        cudaEventSynchronize(h->out_done);        // copies may still read h_out
        cudaEventDestroy(h->out_done);
    }
    for (cudaStream_t sx : {h->copy_stream, h->up_stream})
        if (sx) {
            cudaStreamSynchronize(sx);
            cudaStreamDestroy(sx);
        }
    for (cudaEvent_t ex : {h->decided, h->gpu_part_done})
        if (ex) cudaEventDestroy(ex);
    for (cudaEvent_t e : h->seg_ev) cudaEventDestroy(e);
    if (h->h_g) cudaFreeHost(h->h_g);
    if (h->h_out) cudaFreeHost(h->h_out);
    for (cudaEvent_t e : h->ev) cudaEventDestroy(e);
    cudaFree(h->d_state);
    cudaFree(h->d_done);
    cudaFree(h->d_bc);
    cudaFree(h->d_g);
    cudaFree(h->d_part_ss);
    cudaFree(h->d_part_of);
    if (h->h_state) cudaFreeHost(h->h_state);
    delete h;
}

}  // namespace zi

// Lets the other translation units of the library set zero_last_error().
void zero_internal_set_error(const char *msg) {
    snprintf(g_last_error, sizeof(g_last_error), "%s", msg);
}

ZERO_API const char *zero_status_string(zero_status s) {
    switch (s) {
        case ZERO_OK: return "ok";
        case ZERO_ERR_INVALID_ARG: return "invalid argument";
        case ZERO_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
        case ZERO_ERR_ALIGNMENT: return "misaligned pointer";
        case ZERO_ERR_CUDA: return "CUDA error";
        case ZERO_ERR_OVERFLOW_SIZE: return "size overflows int64";
        case ZERO_ERR_TIMEOUT: return "timeout";
        case ZERO_ERR_NO_MEMORY: return "out of memory";
    }
    return "unknown status";
}

ZERO_API const char *zero_last_error(void) { return g_last_error; }

ZERO_API zero_status zero_memory_bytes(int32_t stage, uint64_t psi, int32_t world_size,
                                       uint64_t *total, uint64_t *params, uint64_t *grads,
                                       uint64_t *optim) {
    if (stage < 0 || stage > 3) return fail(ZERO_ERR_INVALID_ARG, "stage must be 0..3");
    if (world_size < 1) return fail(ZERO_ERR_INVALID_ARG, "world_size must be >= 1");
    // bytes/param of fp16 params, fp16 grads, fp32 master+m+v; which are split N ways
    static const unsigned kBytes[3] = {2, 2, 12};
    const bool split[3] = {stage >= 3, stage >= 2, stage >= 1};
    using u128 = unsigned __int128;
    const u128 n = (u128)(uint64_t)world_size;
    u128 num = 0;                               // total * n
    uint64_t part[3];
    for (int k = 0; k < 3; ++k) {
        const u128 b = (u128)kBytes[k] * psi;
        u128 p = split[k] ? (b + n - 1) / n : b;
        if (p > (u128)UINT64_MAX) return fail(ZERO_ERR_OVERFLOW_SIZE, "byte count overflows");
        part[k] = (uint64_t)p;
        num += split[k] ? b : b * n;
    }
    const u128 t = (num + n - 1) / n;
    if (t > (u128)UINT64_MAX) return fail(ZERO_ERR_OVERFLOW_SIZE, "byte count overflows");
    if (total) *total = (uint64_t)t;
    if (params) *params = part[0];
    if (grads) *grads = part[1];
    if (optim) *optim = part[2];
    return ZERO_OK;
}

ZERO_API zero_status zero_flat_init(const zero_param_info *infos, int32_t n_infos,
                                    int32_t world_size, zero_dtype grad_dtype,
                                    zero_dtype param_dtype, zero_reduce_op op,
                                    const zero_hparams *hp, zero_flat **out) {
    if (!out) return fail(ZERO_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!infos || n_infos < 1) return fail(ZERO_ERR_INVALID_ARG, "need at least one param_info");
    if (world_size < 1) return fail(ZERO_ERR_INVALID_ARG, "world_size must be >= 1");
    if ((grad_dtype != ZERO_F16 && grad_dtype != ZERO_BF16 && grad_dtype != ZERO_F32) ||
        (param_dtype != ZERO_F16 && param_dtype != ZERO_BF16))
        return fail(ZERO_ERR_UNSUPPORTED_DTYPE,
                    "grad dtype must be ZERO_F16, ZERO_BF16 or ZERO_F32; param dtype ZERO_F16 or ZERO_BF16");
    if (op != ZERO_SUM && op != ZERO_AVG) return fail(ZERO_ERR_INVALID_ARG, "op must be SUM or AVG");
    zero_status s = validate_hparams(hp);
    if (s) return s;

    int64_t total = 0;
    for (int32_t k = 0; k < n_infos; ++k) {
        const zero_param_info &p = infos[k];
        if (p.offset != total)
            return fail(ZERO_ERR_INVALID_ARG, "param_info %d: offset %lld, expected %lld", k,
                        (long long)p.offset, (long long)total);
        if (p.numel < 0) return fail(ZERO_ERR_INVALID_ARG, "param_info %d: negative numel", k);
        if (p.ndim < 0 || p.ndim > 8) return fail(ZERO_ERR_INVALID_ARG, "param_info %d: ndim", k);
        if (p.dtype != ZERO_F16 && p.dtype != ZERO_BF16)
            return fail(ZERO_ERR_UNSUPPORTED_DTYPE, "param_info %d: dtype", k);
        int64_t prod = 1;
        for (int d = 0; d < p.ndim; ++d)
            if (!mul_ok(prod, p.shape[d], &prod))
                return fail(ZERO_ERR_OVERFLOW_SIZE, "param_info %d: shape product", k);
        if (prod != p.numel)
            return fail(ZERO_ERR_INVALID_ARG, "param_info %d: numel %lld != prod(shape) %lld", k,
                        (long long)p.numel, (long long)prod);
        if (!add_ok(total, p.numel, &total))
            return fail(ZERO_ERR_OVERFLOW_SIZE, "total numel overflows int64");
    }
    const int64_t S = total / world_size + (total % world_size != 0);
    int64_t padded;
    if (!mul_ok(S, world_size, &padded)) return fail(ZERO_ERR_OVERFLOW_SIZE, "padded numel overflows");

    zero_flat *h = new (std::nothrow) zero_flat;
    if (!h) return fail(ZERO_ERR_NO_MEMORY, "host allocation failed");
    cudaError_t e = cudaGetDevice(&h->device);
    if (e) { delete h; return cuda_fail(e, "cudaGetDevice"); }
    e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device);
    if (e) { delete h; return cuda_fail(e, "cudaDeviceGetAttribute"); }
    {
        const int kind = grad_dtype == ZERO_F32 ? zg::kInF32
                       : (grad_dtype == ZERO_BF16 ? zg::kInBF16 : zg::kInF16);
        for (int mode = 0; mode < 4; ++mode) {
            e = zg::reduce_blocks_per_sm(kind, mode, false, &h->reduce_bps[mode]);
            if (!e && mode < 3) e = zg::reduce_blocks_per_sm(kind, mode, true, &h->staged_bps[mode]);
            if (e) { delete h; return cuda_fail(e, "occupancy query"); }
        }
    }
    {
        int pageable = 0;
        if (cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, h->device) == cudaSuccess)
            h->pageable_access = pageable != 0;
        cudaGetLastError();
    }
    h->world = world_size;
    h->grad_dtype = grad_dtype;
    h->param_dtype = param_dtype;
    h->op = op;
    h->hp = *hp;
    h->full_numel = total;
    h->shard = S;
    h->padded = padded;
    h->g_stride = (S + 3) / 4 * 4;
    h->b1 = (float)hp->beta1;
    h->b2 = (float)hp->beta2;
    h->omb1 = (float)(1.0 - hp->beta1);
    h->omb2 = (float)(1.0 - hp->beta2);
    h->lr = (float)hp->lr;
    h->eps = (float)hp->eps;
    h->decay = (float)(1.0 - hp->lr * hp->weight_decay);
    h->min_scale = (float)hp->min_loss_scale;

    s = init_device_state(h);
    if (s) { release(h); return s; }
    *out = h;
    return ZERO_OK;
}

ZERO_API zero_status zero_flat_layout(const zero_flat *h, int64_t *full_numel, int64_t *shard_size,
                                      int64_t *padded_numel) {
    if (!h) return fail(ZERO_ERR_INVALID_ARG, "handle is NULL");
    if (full_numel) *full_numel = h->full_numel;
    if (shard_size) *shard_size = h->shard;
    if (padded_numel) *padded_numel = h->padded;
    return ZERO_OK;
}

ZERO_API zero_status zero_flat_device_bytes(const zero_flat *h, uint64_t *bytes) {
    if (!h || !bytes) return fail(ZERO_ERR_INVALID_ARG, "NULL argument");
    *bytes = h->device_bytes;
    return ZERO_OK;
}

namespace zi {

// The stepped ranks: 1..world_size distinct ranks in range.
zero_status check_ranks(const zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                        int32_t *max_rank) {
    if (!ranks || n_ranks < 1 || n_ranks > h->world)
        return fail(ZERO_ERR_INVALID_ARG, "need 1..world_size stepped ranks");
    std::vector<int32_t> sorted(ranks, ranks + n_ranks);
    std::sort(sorted.begin(), sorted.end());
    for (int32_t j = 0; j < n_ranks; ++j) {
        if (sorted[j] < 0 || sorted[j] >= h->world)
            return fail(ZERO_ERR_INVALID_ARG, "rank %d out of range", sorted[j]);
        if (j && sorted[j] == sorted[j - 1])
            return fail(ZERO_ERR_INVALID_ARG, "rank %d listed twice", sorted[j]);
    }
    *max_rank = sorted.back();
    return ZERO_OK;
}

size_t grad_elem_size(const zero_flat *h) { return h->grad_dtype == ZERO_F32 ? 4 : 2; }

// The contributions of the stepped ranks (element (c, r, i) at
// grads[c*ld + r*mul + i]): present, aligned to their element size, and
// addressable in int64.
zero_status check_grads(const zero_flat *h, const void *grads, int64_t grad_ld,
                        int64_t grad_rank_offset_mul, int32_t max_rank) {
    const int64_t S = h->shard;
    if (grad_ld < 0 || grad_rank_offset_mul < 0)
        return fail(ZERO_ERR_INVALID_ARG, "grad_ld and grad_rank_offset_mul must be >= 0");
    if (S > 0 && !grads) return fail(ZERO_ERR_INVALID_ARG, "grads is NULL");
    if (h->world > 1 && grad_ld < S)
        return fail(ZERO_ERR_INVALID_ARG, "grad_ld must be >= shard_size");
    if ((uintptr_t)grads % grad_elem_size(h))
        return fail(ZERO_ERR_ALIGNMENT, "grads must be aligned to their element size");
    // the largest element index read, (N-1)*ld + r_max*mul + S - 1, must fit int64
    int64_t rows_span, rank_span, span;
    if (!mul_ok((int64_t)(h->world - 1), grad_ld, &rows_span) ||
        !mul_ok((int64_t)max_rank, grad_rank_offset_mul, &rank_span) ||
        !add_ok(rows_span, rank_span, &span) || !add_ok(span, S, &span) ||
        !mul_ok(span, (int64_t)grad_elem_size(h), &span))
        return fail(ZERO_ERR_OVERFLOW_SIZE, "gradient addressing overflows int64");
    return ZERO_OK;
}

// Per-rank fp32 arrays (master, m, v, accumulators): present and 4-byte aligned.
zero_status check_rows(const zero_flat *h, float *const *rows, int32_t n_ranks, const char *what) {
    if (!rows) return fail(ZERO_ERR_INVALID_ARG, "%s array is NULL", what);
    for (int32_t j = 0; j < n_ranks; ++j) {
        if (h->shard > 0 && !rows[j]) return fail(ZERO_ERR_INVALID_ARG, "%s pointer %d is NULL", what, j);
        if ((uintptr_t)rows[j] % 4) return fail(ZERO_ERR_ALIGNMENT, "%s must be 4-byte aligned", what);
    }
    return ZERO_OK;
}

zero_status check_update(const zero_flat *h, int32_t n_ranks, float *const *master,
                         float *const *m, float *const *v, void *flat_param_out,
                         double extra_norm_sq, bool out_optional) {
    zero_status s;
    if ((s = check_rows(h, master, n_ranks, "master"))) return s;
    if ((s = check_rows(h, m, n_ranks, "m"))) return s;
    if ((s = check_rows(h, v, n_ranks, "v"))) return s;
    if (!flat_param_out && !out_optional) return fail(ZERO_ERR_INVALID_ARG, "flat_param_out is NULL");
    if ((uintptr_t)flat_param_out % 2)
        return fail(ZERO_ERR_ALIGNMENT, "flat_param_out must be 2-byte aligned");
    if (!std::isfinite(extra_norm_sq) || extra_norm_sq < 0)
        return fail(ZERO_ERR_INVALID_ARG, "extra_norm_sq must be finite and >= 0");
    return ZERO_OK;
}

int in_kind_of(const zero_flat *h) {
    return h->grad_dtype == ZERO_F32 ? zg::kInF32 : (h->grad_dtype == ZERO_BF16 ? zg::kInBF16 : zg::kInF16);
}

// A kernel gave up a bounded wait (the step it belonged to was skipped):
// clear the device error word and report it.
zero_status take_device_error(zero_flat *h, cudaStream_t st) {
    cudaMemsetAsync(&h->d_state->error, 0, sizeof(int32_t), st);
    cudaStreamSynchronize(st);
    return fail(ZERO_ERR_TIMEOUT, "a kernel gave up waiting for its bulk copies; the step was skipped");
}

// K1 as planned (contributions -> scratch rows, or an accumulator norm pass),
// K2, K3 (from the scratch rows, or from the accumulators), with the timing
// marks and the optional result read-back.  With host_update (the offload
// step) K3 and the last timing mark are left to the caller.  Called on the
// handle's device.
// Geometry, scratch and the handle's buffers for a reduce plan whose mode,
// contributions and ranks the caller has set; *parts = norm partials.
zero_status plan_reduce(zero_flat *h, zg::ReducePlan &rp, int64_t *parts) {
    const int64_t S = h->shard;
    const int64_t batch = std::min<int64_t>(rp.n_ranks, zg::kMaxRanksPerLaunch);
    rp.S = S;
    rp.n_contrib = h->world;
    rp.staged = zg::reduce_wants_staging(rp);
    if (rp.grads) h->last_reduce_staged = rp.staged ? 1 : 0;
    rp.grid_x = zg::grid_x_for(S, batch, h->sm_count,
                               rp.staged ? h->staged_bps[rp.mode] : h->reduce_bps[rp.mode]);
    *parts = (int64_t)rp.grid_x * rp.n_ranks;
    const int64_t rows = rp.mode == zg::kModeStep ? rp.n_ranks : 0;
    zero_status s = ensure_scratch(h, rows, *parts);
    if (s) return s;
    rp.g = h->d_g;
    rp.g_stride = h->g_stride;
    rp.part_ss = h->d_part_ss;
    rp.part_of = h->d_part_of;
    rp.full_numel = h->full_numel;
    rp.avg = h->op == ZERO_AVG;
    rp.st = h->d_state;
    rp.done = h->d_done;
    return ZERO_OK;
}

// The handle's scalars, buffers and geometry for an AdamW plan whose state
// pointers (and accumulators, or int8 outputs) the caller has set.
void plan_adamw(zero_flat *h, zg::AdamPlan &ap, const int32_t *ranks, int32_t n_ranks) {
    const int64_t S = h->shard;
    const int64_t batch = std::min<int64_t>(n_ranks, zg::kMaxRanksPerLaunch);
    ap.grid_x = zg::grid_x_for(S, batch, h->sm_count,
                               ap.q8 ? zg::kAdamQ8BlocksPerSm : zg::kAdamBlocksPerSm);
    if (!ap.acc) {
        ap.g = h->d_g;
        ap.g_stride = h->g_stride;
    }
    ap.bf16_out = h->param_dtype == ZERO_BF16;
    ap.ranks = ranks;
    ap.n_ranks = n_ranks;
    ap.S = S;
    ap.full_numel = h->full_numel;
    ap.b1 = h->b1; ap.b2 = h->b2; ap.omb1 = h->omb1; ap.omb2 = h->omb2;
    ap.lr = h->lr; ap.eps = h->eps; ap.decay = h->decay;
    ap.st = h->d_state;
}

// The decision's arguments over n_parts partials (or one pair of totals).
zg::FinalizeArgs decision_args(zero_flat *h, const double *part_ss, const int32_t *part_of,
                               int32_t n_parts, double extra_norm_sq) {
    zg::FinalizeArgs f{};
    f.part_ss = part_ss;
    f.part_of = part_of;
    f.n_parts = n_parts;
    f.dynamic = h->hp.dynamic_loss_scale;
    f.window = h->hp.loss_scale_window;
    f.min_scale = h->min_scale;
    f.extra_norm_sq = extra_norm_sq;
    f.max_grad_norm = h->hp.max_grad_norm;
    f.bc_table = h->d_bc;
    f.bc_len = h->bc_len;
    f.st = h->d_state;
    return f;
}

// Copy the step's result to the host (synchronizes `st`).
zero_status read_result(zero_flat *h, cudaStream_t st, zero_step_result *res) {
    cudaError_t e = cudaMemcpyAsync(h->h_state, h->d_state, sizeof(zg::DevState),
                                    cudaMemcpyDeviceToHost, st);
    if (!e) e = cudaStreamSynchronize(st);
    if (e) return cuda_fail(e, "reading the step result");
    res->overflow = h->h_state->res.overflow;
    res->skipped = h->h_state->res.skipped;
    res->grad_norm = h->h_state->res.grad_norm;
    res->clip_coef = h->h_state->res.clip_coef;
    res->scale_used = h->h_state->res.scale_used;
    if (h->h_state->error) return take_device_error(h, st);
    return ZERO_OK;
}

zero_status launch_step(zero_flat *h, zg::ReducePlan rp, zg::AdamPlan ap, double extra_norm_sq,
                        cudaStream_t st, zero_step_result *res, bool host_update = false) {
    const int64_t S = h->shard;
    h->reduced_ranks.clear();             // this step overwrites a split step's gradient rows
    int64_t parts = 0;
    zero_status s = plan_reduce(h, rp, &parts);
    if (s) return s;
    plan_adamw(h, ap, rp.ranks, rp.n_ranks);
    const zg::FinalizeArgs f =
        decision_args(h, h->d_part_ss, h->d_part_of, S > 0 ? (int32_t)parts : 0, extra_norm_sq);
    // the last reduce block makes the decision (no K2 launch) whenever there
    // is a reduce to count in; an empty shard still needs K2
    rp.fuse_finalize = S > 0;
    rp.fin = f;

    cudaError_t e;
    if ((e = mark(h, st))) return cuda_fail(e, "timing event");
    if ((e = zg::run_reduce(rp, st))) return cuda_fail(e, "reduce kernel launch");
    if ((e = mark(h, st))) return cuda_fail(e, "timing event");
    if (!rp.fuse_finalize && (e = zg::launch_finalize(f, st)))
        return cuda_fail(e, "finalize kernel launch");
    if ((e = mark(h, st))) return cuda_fail(e, "timing event");
    if (host_update) return ZERO_OK;
    if ((e = zg::run_adamw(ap, st))) return cuda_fail(e, "adamw kernel launch");
    if ((e = mark(h, st))) return cuda_fail(e, "timing event");
    return res ? read_result(h, st, res) : ZERO_OK;
}

}  // namespace zi

ZERO_API zero_status zero_shard_step(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                                     const void *grads, int64_t grad_ld,
                                     int64_t grad_rank_offset_mul, float *const *master,
                                     float *const *m, float *const *v, void *flat_param_out,
                                     double extra_norm_sq, void *stream, zero_step_result *res) {
    if (!h) return fail(ZERO_ERR_INVALID_ARG, "handle is NULL");
    int32_t max_rank = 0;
    zero_status s;
    if ((s = check_ranks(h, ranks, n_ranks, &max_rank))) return s;
    if ((s = check_update(h, n_ranks, master, m, v, flat_param_out, extra_norm_sq))) return s;
    if ((s = check_grads(h, grads, grad_ld, grad_rank_offset_mul, max_rank))) return s;
    DeviceGuard guard(h->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the handle's device");
    zg::ReducePlan rp;
    rp.mode = zg::kModeStep;
    rp.grads = grads;
    rp.in_kind = in_kind_of(h);
    rp.ld = grad_ld;
    rp.rank_mul = grad_rank_offset_mul;
    rp.ranks = ranks;
    rp.n_ranks = n_ranks;
    zg::AdamPlan ap;
    ap.master = master;
    ap.m = m;
    ap.v = v;
    ap.out = flat_param_out;
    return launch_step(h, rp, ap, extra_norm_sq, (cudaStream_t)stream, res);
}

ZERO_API zero_status zero_shard_reduce(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                                       const void *grads, int64_t grad_ld,
                                       int64_t grad_rank_offset_mul, double *norm_sq_out,
                                       int32_t *overflow_out, void *stream) {
    if (!h) return fail(ZERO_ERR_INVALID_ARG, "handle is NULL");
    int32_t max_rank = 0;
    zero_status s;
    if ((s = check_ranks(h, ranks, n_ranks, &max_rank))) return s;
    if ((s = check_grads(h, grads, grad_ld, grad_rank_offset_mul, max_rank))) return s;
    if (!norm_sq_out || !overflow_out) return fail(ZERO_ERR_INVALID_ARG, "NULL output");
    if ((uintptr_t)norm_sq_out % 8 || (uintptr_t)overflow_out % 4)
        return fail(ZERO_ERR_ALIGNMENT, "norm_sq_out must be 8-byte, overflow_out 4-byte aligned");
    DeviceGuard guard(h->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the handle's device");
    const cudaStream_t st = (cudaStream_t)stream;
    zg::ReducePlan rp;
    rp.mode = zg::kModeStep;
    rp.grads = grads;
    rp.in_kind = in_kind_of(h);
    rp.ld = grad_ld;
    rp.rank_mul = grad_rank_offset_mul;
    rp.ranks = ranks;
    rp.n_ranks = n_ranks;
    int64_t parts = 0;
    if ((s = plan_reduce(h, rp, &parts))) return s;
    cudaError_t e;
    if (h->shard > 0) {                   // the last block totals the partials
        zg::FinalizeArgs f = decision_args(h, h->d_part_ss, h->d_part_of, (int32_t)parts, 0.0);
        f.sum_out = norm_sq_out;
        f.of_out = overflow_out;
        rp.fuse_finalize = true;
        rp.fin = f;
        e = zg::run_reduce(rp, st);
    } else {
        e = cudaMemsetAsync(norm_sq_out, 0, sizeof(double), st);
        if (!e) e = cudaMemsetAsync(overflow_out, 0, sizeof(int32_t), st);
    }
    if (e) return cuda_fail(e, "reduce kernel launch");
    h->reduced_ranks.assign(ranks, ranks + n_ranks);
    return ZERO_OK;
}

ZERO_API zero_status zero_shard_reduce_accumulated(zero_flat *h, const int32_t *ranks,
                                                   int32_t n_ranks, const float *const *acc,
                                                   double *norm_sq_out, int32_t *overflow_out,
                                                   void *stream) {
    if (!h) return fail(ZERO_ERR_INVALID_ARG, "handle is NULL");
    int32_t max_rank = 0;
    zero_status s;
    if ((s = check_ranks(h, ranks, n_ranks, &max_rank))) return s;
    if ((s = check_rows(h, const_cast<float *const *>(acc), n_ranks, "acc"))) return s;
    if (!norm_sq_out || !overflow_out) return fail(ZERO_ERR_INVALID_ARG, "NULL output");
    if ((uintptr_t)norm_sq_out % 8 || (uintptr_t)overflow_out % 4)
        return fail(ZERO_ERR_ALIGNMENT, "norm_sq_out must be 8-byte, overflow_out 4-byte aligned");
    DeviceGuard guard(h->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the handle's device");
    const cudaStream_t st = (cudaStream_t)stream;
    // the step's reduce with each accumulator as the one fp32 contribution of
    // its row: g = acc / scale (padding zero) into the handle's gradient rows,
    // the overflow check and the norm partials
    zg::ReducePlan rp;
    rp.mode = zg::kModeStep;
    rp.ranks = ranks;
    rp.n_ranks = n_ranks;
    int64_t parts = 0;
    if ((s = plan_reduce(h, rp, &parts))) return s;
    rp.in_kind = zg::kInF32;
    rp.n_contrib = 1;
    rp.avg = 0;
    rp.staged = false;
    int bps = 1;
    cudaError_t e = zg::reduce_blocks_per_sm(zg::kInF32, zg::kModeStep, false, &bps);
    if (e) return cuda_fail(e, "occupancy query");
    const int64_t batch = std::min<int64_t>(n_ranks, zg::kMaxRanksPerLaunch);
    rp.grid_x = std::min(rp.grid_x, zg::grid_x_for(h->shard, batch, h->sm_count, bps));
    parts = (int64_t)rp.grid_x * n_ranks;
    if (h->shard > 0) {
        std::vector<zg::ReduceRow> rows(n_ranks);
        for (int32_t j = 0; j < n_ranks; ++j) {
            zg::ReduceRow &w = rows[j];
            const int64_t first = (int64_t)ranks[j] * h->shard;
            w.in = acc[j];
            w.S = h->shard;
            w.valid = std::max<int64_t>(0, std::min<int64_t>(h->shard, h->full_numel - first));
            w.first = first;
            w.g = h->d_g + (int64_t)j * h->g_stride;
        }
        zg::FinalizeArgs f = decision_args(h, h->d_part_ss, h->d_part_of, (int32_t)parts, 0.0);
        f.sum_out = norm_sq_out;           // the last block totals the partials
        f.of_out = overflow_out;
        rp.fuse_finalize = true;
        rp.fin = f;
        e = zg::run_reduce_rows(rp, rows.data(), n_ranks, st, true);
    } else {
        e = cudaMemsetAsync(norm_sq_out, 0, sizeof(double), st);
        if (!e) e = cudaMemsetAsync(overflow_out, 0, sizeof(int32_t), st);
    }
    if (e) return cuda_fail(e, "reduce kernel launch");
    h->reduced_ranks.assign(ranks, ranks + n_ranks);
    return ZERO_OK;
}

// The second half of a split step: the decision over n_parts (norm_sq[k],
// overflow[k]) pairs in device memory, then AdamW and the cast (and, with
// q8, the int8 payload: flat_param_out may then be NULL).
static zero_status apply_parts(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                               float *const *master, float *const *m, float *const *v,
                               void *flat_param_out, const double *norm_sq,
                               const int32_t *overflow, int32_t n_parts, void *stream,
                               zero_step_result *res, bool q8 = false,
                               int8_t *flat_q8_out = nullptr, float *q8_scales = nullptr) {
    if (!h) return fail(ZERO_ERR_INVALID_ARG, "handle is NULL");
    int32_t max_rank = 0;
    zero_status s;
    if ((s = check_ranks(h, ranks, n_ranks, &max_rank))) return s;
    if ((s = check_update(h, n_ranks, master, m, v, flat_param_out, 0.0, q8))) return s;
    if (q8 && (!flat_q8_out || !q8_scales))
        return fail(ZERO_ERR_INVALID_ARG, "int8 outputs are NULL");
    if (q8 && (uintptr_t)q8_scales % 4)
        return fail(ZERO_ERR_ALIGNMENT, "q8_scales must be 4-byte aligned");
    if (!norm_sq || !overflow) return fail(ZERO_ERR_INVALID_ARG, "NULL total");
    if (n_parts < 1 || n_parts > (1 << 20))
        return fail(ZERO_ERR_INVALID_ARG, "n_parts must be in [1, 2^20]");
    if ((uintptr_t)norm_sq % 8 || (uintptr_t)overflow % 4)
        return fail(ZERO_ERR_ALIGNMENT, "norm_sq must be 8-byte, overflow 4-byte aligned");
    if (h->reduced_ranks.size() != (size_t)n_ranks ||
        !std::equal(ranks, ranks + n_ranks, h->reduced_ranks.begin()))
        return fail(ZERO_ERR_INVALID_ARG,
                    "zero_shard_apply needs the ranks of the preceding zero_shard_reduce");
    DeviceGuard guard(h->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the handle's device");
    const cudaStream_t st = (cudaStream_t)stream;
    zg::AdamPlan ap;
    ap.master = master;
    ap.m = m;
    ap.v = v;
    ap.out = flat_param_out;
    if (q8) {
        ap.q8 = flat_q8_out;
        ap.q8_scales = q8_scales;
    }
    plan_adamw(h, ap, ranks, n_ranks);
    // the decision from the caller's partials, totalled by the decision kernel
    // in its fixed order
    const zg::FinalizeArgs f = decision_args(h, norm_sq, overflow, n_parts, 0.0);
    cudaError_t e;
    if ((e = zg::launch_finalize(f, st))) return cuda_fail(e, "finalize kernel launch");
    if ((e = zg::run_adamw(ap, st))) return cuda_fail(e, "adamw kernel launch");
    h->reduced_ranks.clear();
    return res ? read_result(h, st, res) : ZERO_OK;
}

ZERO_API zero_status zero_shard_apply(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                                      float *const *master, float *const *m, float *const *v,
                                      void *flat_param_out, const double *norm_sq,
                                      const int32_t *overflow, void *stream,
                                      zero_step_result *res) {
    // one "partial" holding the caller's totals
    return apply_parts(h, ranks, n_ranks, master, m, v, flat_param_out, norm_sq, overflow, 1,
                       stream, res);
}

ZERO_API zero_status zero_shard_apply_partials_q8(
    zero_flat *h, const int32_t *ranks, int32_t n_ranks, float *const *master, float *const *m,
    float *const *v, void *flat_param_out, int8_t *flat_q8_out, float *q8_scales,
    const double *norm_sq_parts, const int32_t *overflow_parts, int32_t n_parts, void *stream,
    zero_step_result *res) {
    return apply_parts(h, ranks, n_ranks, master, m, v, flat_param_out, norm_sq_parts,
                       overflow_parts, n_parts, stream, res, true, flat_q8_out, q8_scales);
}

ZERO_API zero_status zero_shard_apply_partials(zero_flat *h, const int32_t *ranks,
                                               int32_t n_ranks, float *const *master,
                                               float *const *m, float *const *v,
                                               void *flat_param_out,
                                               const double *norm_sq_parts,
                                               const int32_t *overflow_parts, int32_t n_parts,
                                               void *stream, zero_step_result *res) {
    return apply_parts(h, ranks, n_ranks, master, m, v, flat_param_out, norm_sq_parts,
                       overflow_parts, n_parts, stream, res);
}

ZERO_API zero_status zero_shard_step_q8(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                                        const void *grads, int64_t grad_ld,
                                        int64_t grad_rank_offset_mul, float *const *master,
                                        float *const *m, float *const *v, void *flat_param_out,
                                        int8_t *flat_q8_out, float *q8_scales,
                                        double extra_norm_sq, void *stream,
                                        zero_step_result *res) {
    if (!h) return fail(ZERO_ERR_INVALID_ARG, "handle is NULL");
    int32_t max_rank = 0;
    zero_status s;
    if ((s = check_ranks(h, ranks, n_ranks, &max_rank))) return s;
    if ((s = check_update(h, n_ranks, master, m, v, flat_param_out, extra_norm_sq, true))) return s;
    if ((s = check_grads(h, grads, grad_ld, grad_rank_offset_mul, max_rank))) return s;
    if (!flat_q8_out || !q8_scales) return fail(ZERO_ERR_INVALID_ARG, "int8 outputs are NULL");
    if ((uintptr_t)q8_scales % 4) return fail(ZERO_ERR_ALIGNMENT, "q8_scales must be 4-byte aligned");
    DeviceGuard guard(h->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the handle's device");
    zg::ReducePlan rp;
    rp.mode = zg::kModeStep;
    rp.grads = grads;
    rp.in_kind = in_kind_of(h);
    rp.ld = grad_ld;
    rp.rank_mul = grad_rank_offset_mul;
    rp.ranks = ranks;
    rp.n_ranks = n_ranks;
    zg::AdamPlan ap;
    ap.master = master;
    ap.m = m;
    ap.v = v;
    ap.out = flat_param_out;
    ap.q8 = flat_q8_out;
    ap.q8_scales = q8_scales;
    return launch_step(h, rp, ap, extra_norm_sq, (cudaStream_t)stream, res);
}

ZERO_API zero_status zero_grad_accumulate(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                                          const void *grads, int64_t grad_ld,
                                          int64_t grad_rank_offset_mul, float *const *acc,
                                          int32_t first_micro_step, void *stream) {
    if (!h) return fail(ZERO_ERR_INVALID_ARG, "handle is NULL");
    int32_t max_rank = 0;
    zero_status s;
    if ((s = check_ranks(h, ranks, n_ranks, &max_rank))) return s;
    if ((s = check_rows(h, acc, n_ranks, "acc"))) return s;
    if ((s = check_grads(h, grads, grad_ld, grad_rank_offset_mul, max_rank))) return s;
    DeviceGuard guard(h->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the handle's device");
    zg::ReducePlan rp;
    rp.mode = first_micro_step ? zg::kModeAccFirst : zg::kModeAccAdd;
    rp.grads = grads;
    rp.in_kind = in_kind_of(h);
    rp.ld = grad_ld;
    rp.rank_mul = grad_rank_offset_mul;
    rp.acc_out = acc;
    rp.ranks = ranks;
    rp.n_ranks = n_ranks;
    rp.S = h->shard;
    rp.full_numel = h->full_numel;
    rp.n_contrib = h->world;
    rp.avg = h->op == ZERO_AVG;
    rp.st = h->d_state;
    rp.staged = zg::reduce_wants_staging(rp);
    h->last_reduce_staged = rp.staged ? 1 : 0;
    const int64_t batch = std::min<int64_t>(n_ranks, zg::kMaxRanksPerLaunch);
    rp.grid_x = zg::grid_x_for(h->shard, batch, h->sm_count,
                               rp.staged ? h->staged_bps[rp.mode] : h->reduce_bps[rp.mode]);
    const cudaError_t e = zg::run_reduce(rp, (cudaStream_t)stream);
    if (e) return cuda_fail(e, "accumulate kernel launch");
    return ZERO_OK;
}

ZERO_API zero_status zero_shard_step_accumulated(zero_flat *h, const int32_t *ranks,
                                                 int32_t n_ranks, const float *const *acc,
                                                 float *const *master, float *const *m,
                                                 float *const *v, void *flat_param_out,
                                                 double extra_norm_sq, void *stream,
                                                 zero_step_result *res) {
    if (!h) return fail(ZERO_ERR_INVALID_ARG, "handle is NULL");
    int32_t max_rank = 0;
    zero_status s;
    if ((s = check_ranks(h, ranks, n_ranks, &max_rank))) return s;
    if ((s = check_rows(h, const_cast<float *const *>(acc), n_ranks, "acc"))) return s;
    if ((s = check_update(h, n_ranks, master, m, v, flat_param_out, extra_norm_sq))) return s;
    DeviceGuard guard(h->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the handle's device");
    zg::ReducePlan rp;
    rp.mode = zg::kModeNormOnly;
    rp.in_kind = zg::kInF32;
    rp.acc_in = acc;
    rp.ranks = ranks;
    rp.n_ranks = n_ranks;
    zg::AdamPlan ap;
    ap.acc = acc;
    ap.master = master;
    ap.m = m;
    ap.v = v;
    ap.out = flat_param_out;
    return launch_step(h, rp, ap, extra_norm_sq, (cudaStream_t)stream, res);
}

namespace zi {

// Pinned host buffers and worker threads of the offload step, grown on demand.
// Pinned host rows of the handle's offload updates (reduced-gradient copies
// and 16-bit parameter staging) for n_ranks stepped ranks.  busy: an event
// whose copies may still read the staging (besides the handle's own), waited
// for before a buffer is replaced.
zero_status ensure_host_rows(zero_flat *h, int32_t n_ranks, cudaEvent_t busy) {
    const int64_t S = h->shard;
    if (n_ranks > h->h_g_rows || n_ranks > h->h_out_rows) {
        if (h->out_done) cudaEventSynchronize(h->out_done);
        if (busy) cudaEventSynchronize(busy);
    }
    if (n_ranks > h->h_g_rows) {
        if (h->h_g) cudaFreeHost(h->h_g);
        h->h_g = nullptr;
        h->h_g_rows = 0;
        int64_t bytes;
        if (!mul_ok((int64_t)n_ranks, h->g_stride, &bytes) || !mul_ok(bytes, 4, &bytes))
            return fail(ZERO_ERR_OVERFLOW_SIZE, "host gradient buffer size overflows");
        if (bytes > 0) {
            cudaError_t e = cudaHostAlloc((void **)&h->h_g, (size_t)bytes, cudaHostAllocPortable);
            if (e) {
                cudaGetLastError();
                h->h_g = nullptr;
                return fail(ZERO_ERR_NO_MEMORY, "cannot pin %lld bytes of host gradient rows: %s",
                            (long long)bytes, cudaGetErrorString(e));
            }
        }
        h->h_g_rows = n_ranks;
    }
    if (n_ranks > h->h_out_rows) {
        if (h->h_out) cudaFreeHost(h->h_out);
        h->h_out = nullptr;
        h->h_out_rows = 0;
        int64_t bytes;
        if (!mul_ok((int64_t)n_ranks, S, &bytes) || !mul_ok(bytes, 2, &bytes))
            return fail(ZERO_ERR_OVERFLOW_SIZE, "host parameter staging size overflows");
        if (bytes > 0) {
            cudaError_t e = cudaHostAlloc((void **)&h->h_out, (size_t)bytes, cudaHostAllocPortable);
            if (e) {
                cudaGetLastError();
                h->h_out = nullptr;
                return fail(ZERO_ERR_NO_MEMORY, "cannot pin %lld bytes of parameter staging: %s",
                            (long long)bytes, cudaGetErrorString(e));
            }
        }
        h->h_out_rows = n_ranks;
    }
    return ZERO_OK;
}

// The streams, events and worker threads that run offload updates.
zero_status ensure_host_runtime(zero_flat *h, int32_t n_threads) {
    if (!h->out_done) {
        cudaError_t e = cudaEventCreateWithFlags(&h->out_done, cudaEventDisableTiming);
        if (e) { h->out_done = nullptr; return cuda_fail(e, "cudaEventCreate"); }
    }
    for (cudaStream_t *sx : {&h->copy_stream, &h->up_stream})
        if (!*sx) {
            cudaError_t e = cudaStreamCreateWithFlags(sx, cudaStreamNonBlocking);
            if (e) { *sx = nullptr; return cuda_fail(e, "cudaStreamCreate"); }
        }
    for (cudaEvent_t *ex : {&h->decided, &h->gpu_part_done})
        if (!*ex) {
            cudaError_t e = cudaEventCreateWithFlags(ex, cudaEventDisableTiming);
            if (e) { *ex = nullptr; return cuda_fail(e, "cudaEventCreate"); }
        }
    const int want = n_threads > 0 ? n_threads : zh::available_cpus();
    if (!h->pool || h->pool->size() != want) {
        h->pool.reset();
        h->pool.reset(new (std::nothrow) zh::Pool(want));
        if (!h->pool) return fail(ZERO_ERR_NO_MEMORY, "host thread pool");
    }
    return ZERO_OK;
}

zero_status ensure_offload(zero_flat *h, int32_t n_ranks, int32_t n_threads) {
    zero_status s = ensure_host_runtime(h, n_threads);
    return s ? s : ensure_host_rows(h, n_ranks, nullptr);
}


// The host update of every row.  The reduced gradient rows come down from
// HBM segment by segment on rt's copy stream, and a host task waits only for
// the segment it works on, so the copies overlap the update; each segment's
// 16-bit parameters go back to the device on the up stream as soon as its
// last chunk is done.  rt supplies the streams, the pool, the segment events
// and the device.  Returns the first CUDA error, if any.
cudaError_t host_update_rows(zero_flat *rt, const HostRow *rows, int64_t n_rows, bool bf16) {
    const int64_t chunks_per_seg = kHostSegment / kHostChunk;
    // per row: its first segment and its first task, in row order
    std::vector<int64_t> seg0(n_rows + 1, 0), task0(n_rows + 1, 0);
    for (int64_t j = 0; j < n_rows; ++j) {
        const int64_t span = std::max<int64_t>(rows[j].S - rows[j].i_begin, 0);
        seg0[j + 1] = seg0[j] + (span + kHostSegment - 1) / kHostSegment;
        task0[j + 1] = task0[j] + (span + kHostChunk - 1) / kHostChunk;
    }
    const int64_t n_seg = seg0[n_rows], n_tasks = task0[n_rows];
    if (n_tasks == 0) return cudaSuccess;
    cudaError_t e;
    while ((int64_t)rt->seg_ev.size() < n_seg) {
        cudaEvent_t ev;
        if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming))) return e;
        rt->seg_ev.push_back(ev);
    }
    std::unique_ptr<std::atomic<int64_t>[]> left(new std::atomic<int64_t>[n_seg]);
    std::unique_ptr<std::atomic<int>[]> ready(new std::atomic<int>[n_seg]);
    for (int64_t j = 0; j < n_rows; ++j) {
        const HostRow &w = rows[j];
        const int64_t chunks = task0[j + 1] - task0[j];
        for (int64_t q = 0; q < seg0[j + 1] - seg0[j]; ++q) {
            const int64_t s0 = w.i_begin + q * kHostSegment, len = std::min(kHostSegment, w.S - s0);
            if ((e = cudaMemcpyAsync(w.h_g + s0, w.d_g + s0, (size_t)len * 4,
                                     cudaMemcpyDeviceToHost, rt->copy_stream)))
                return e;
            if ((e = cudaEventRecord(rt->seg_ev[seg0[j] + q], rt->copy_stream))) return e;
            left[seg0[j] + q].store(std::min(chunks_per_seg, chunks - q * chunks_per_seg));
            ready[seg0[j] + q].store(0);
        }
    }
    std::atomic<int> err{0};
    const int dev = rt->device;
    auto note = [&](cudaError_t x) {
        int none = 0;
        if (x) err.compare_exchange_strong(none, (int)x);
    };
    const std::function<void(int64_t)> task = [&](int64_t t) {
        const int64_t j = std::upper_bound(task0.begin(), task0.end(), t) - task0.begin() - 1;
        const HostRow &w = rows[j];
        const int64_t c = t - task0[j];
        const int64_t q = c / chunks_per_seg, sg = seg0[j] + q;
        if (!ready[sg].load(std::memory_order_acquire)) {
            const cudaError_t x = cudaEventSynchronize(rt->seg_ev[sg]);
            if (x) { note(x); return; }
            ready[sg].store(1, std::memory_order_release);
        }
        const int64_t i0 = w.i_begin + c * kHostChunk;
        const int64_t n = std::min(kHostChunk, w.S - i0);
        zh::adamw_cast_range(w.k, w.h_g + i0, w.master + i0, w.m + i0, w.v + i0, w.stage + i0, n,
                             bf16);
        if (left[sg].fetch_sub(1) == 1) {                      // segment complete
            const int64_t s0 = w.i_begin + q * kHostSegment;
            const int64_t len = std::min(kHostSegment, w.S - s0);
            cudaError_t x = cudaSetDevice(dev);
            if (!x) x = cudaMemcpyAsync(w.d_out + s0, w.stage + s0, (size_t)len * 2,
                                        cudaMemcpyHostToDevice, rt->up_stream);
            note(x);
        }
    };
    rt->pool->run(n_tasks, task);
    return (cudaError_t)err.load();
}

// The rows of one handle's offload update (its pinned buffers, its ranks).
void host_rows_of(zero_flat *h, const zh::AdamScalars &k, const int32_t *ranks, int32_t n_ranks,
                  float *const *master, float *const *m, float *const *v, void *flat_param_out,
                  int64_t i_begin, std::vector<HostRow> &rows) {
    const int64_t S = h->shard;
    uint16_t *out16 = static_cast<uint16_t *>(flat_param_out);
    for (int32_t j = 0; j < n_ranks; ++j)
        rows.push_back(HostRow{h->d_g + (int64_t)j * h->g_stride, h->h_g + (int64_t)j * h->g_stride,
                               master[j], m[j], v[j], h->h_out + (int64_t)j * S,
                               out16 + (int64_t)ranks[j] * S, S, i_begin, k});
}

// Whether the GPU can read and write every stepped rank's host arrays.
bool gpu_reaches(const zero_flat *h, int32_t n_ranks, float *const *const rows[3]) {
    if (h->pageable_access) return true;
    for (int a = 0; a < 3; ++a)
        for (int32_t j = 0; j < n_ranks; ++j) {
            cudaPointerAttributes at{};
            if (cudaPointerGetAttributes(&at, rows[a][j]) != cudaSuccess) {
                cudaGetLastError();
                return false;
            }
            if (at.type != cudaMemoryTypeHost) return false;   // pinned / registered only
        }
    return true;
}

}  // namespace zi

ZERO_API zero_status zero_shard_step_offload(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                                             const void *grads, int64_t grad_ld,
                                             int64_t grad_rank_offset_mul, float *const *master,
                                             float *const *m, float *const *v,
                                             void *flat_param_out, double extra_norm_sq,
                                             int32_t n_threads, double gpu_share, void *stream,
                                             zero_step_result *res) {
    if (!h) return fail(ZERO_ERR_INVALID_ARG, "handle is NULL");
    int32_t max_rank = 0;
    zero_status s;
    if ((s = check_ranks(h, ranks, n_ranks, &max_rank))) return s;
    if ((s = check_update(h, n_ranks, master, m, v, flat_param_out, extra_norm_sq))) return s;
    if ((s = check_grads(h, grads, grad_ld, grad_rank_offset_mul, max_rank))) return s;
    if (n_threads < 0) return fail(ZERO_ERR_INVALID_ARG, "n_threads must be >= 0");
    if (!(gpu_share >= 0.0 && gpu_share <= 1.0))
        return fail(ZERO_ERR_INVALID_ARG, "gpu_share must be in [0, 1]");
    const int64_t S = h->shard;
    // the GPU takes elements [0, split) of every rank, the host threads the rest
    int64_t split = gpu_share >= 1.0 ? S : (int64_t)(gpu_share * (double)S) / kHostChunk * kHostChunk;
    split = std::min(split, S);
    DeviceGuard guard(h->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the handle's device");
    float *const *const rows[3] = {master, m, v};
    if (split > 0 && !gpu_reaches(h, n_ranks, rows))
        return fail(ZERO_ERR_INVALID_ARG,
                    "gpu_share > 0 needs host arrays the GPU can access (pinned or registered)");
    if ((s = ensure_offload(h, n_ranks, n_threads))) return s;
    const cudaStream_t st = (cudaStream_t)stream;
    zg::ReducePlan rp;
    rp.mode = zg::kModeStep;
    rp.grads = grads;
    rp.in_kind = in_kind_of(h);
    rp.ld = grad_ld;
    rp.rank_mul = grad_rank_offset_mul;
    rp.ranks = ranks;
    rp.n_ranks = n_ranks;
    zg::AdamPlan none;
    if ((s = launch_step(h, rp, none, extra_norm_sq, st, nullptr, true))) return s;
    cudaError_t e = cudaMemcpyAsync(h->h_state, h->d_state, sizeof(zg::DevState),
                                    cudaMemcpyDeviceToHost, st);
    if (!e) e = cudaEventRecord(h->decided, st);
    if (e) return cuda_fail(e, "reading the step decision");
    if (split > 0) {                                  // the GPU's share, queued behind the decision
        zg::AdamPlan ap;
        ap.g = h->d_g;
        ap.g_stride = h->g_stride;
        ap.master = master;
        ap.m = m;
        ap.v = v;
        ap.out = flat_param_out;
        ap.bf16_out = h->param_dtype == ZERO_BF16;
        ap.ranks = ranks;
        ap.n_ranks = n_ranks;
        ap.S = S;
        ap.count = split;
        ap.full_numel = h->full_numel;
        ap.b1 = h->b1; ap.b2 = h->b2; ap.omb1 = h->omb1; ap.omb2 = h->omb2;
        ap.lr = h->lr; ap.eps = h->eps; ap.decay = h->decay;
        ap.st = h->d_state;
        ap.grid_x = zg::grid_x_for(split, std::min<int64_t>(n_ranks, zg::kMaxRanksPerLaunch),
                                   h->sm_count, zg::kAdamBlocksPerSm);
        if ((e = zg::run_adamw(ap, st))) return cuda_fail(e, "adamw kernel launch");
    }
    if ((e = cudaEventRecord(h->gpu_part_done, st))) return cuda_fail(e, "cudaEventRecord");
    if ((e = cudaEventSynchronize(h->decided))) return cuda_fail(e, "waiting for the step decision");
    const zg::DevState ds = *h->h_state;
    if (ds.error) return take_device_error(h, st);
    if (!ds.res.skipped && split < S) {
        // the previous call's parameter copies read h_out
        if ((e = cudaEventSynchronize(h->out_done))) return cuda_fail(e, "waiting for the last copies");
        const zh::AdamScalars k{h->b1, h->b2, h->omb1, h->omb2, h->lr, h->eps, h->decay,
                                ds.res.clip_coef, ds.bc1, ds.bc2};
        std::vector<HostRow> rows;
        host_rows_of(h, k, ranks, n_ranks, master, m, v, flat_param_out, split, rows);
        if ((e = host_update_rows(h, rows.data(), (int64_t)rows.size(),
                                  h->param_dtype == ZERO_BF16)))
            return cuda_fail(e, "copying parameters to the device");
        if ((e = cudaSetDevice(h->device))) return cuda_fail(e, "cudaSetDevice");
        if ((e = cudaEventRecord(h->out_done, h->up_stream))) return cuda_fail(e, "cudaEventRecord");
        if ((e = cudaStreamWaitEvent(st, h->out_done, 0))) return cuda_fail(e, "cudaStreamWaitEvent");
    }
    // the GPU's share of the host arrays is written when the call returns too
    if ((e = cudaEventSynchronize(h->gpu_part_done))) return cuda_fail(e, "waiting for the GPU share");
    if ((e = mark(h, st))) return cuda_fail(e, "timing event");
    if (res) {
        res->overflow = ds.res.overflow;
        res->skipped = ds.res.skipped;
        res->grad_norm = ds.res.grad_norm;
        res->clip_coef = ds.res.clip_coef;
        res->scale_used = ds.res.scale_used;
    }
    return ZERO_OK;
}

ZERO_API zero_status zero_offload_adamw_host(const zero_hparams *hp, int64_t step_t,
                                             float clip_coef, const float *g, float *master,
                                             float *m, float *v, void *param_out, int64_t n,
                                             zero_dtype param_dtype, int32_t n_threads) {
    zero_status s;
    if ((s = validate_hparams(hp))) return s;
    if (n < 0) return fail(ZERO_ERR_INVALID_ARG, "n must be >= 0");
    if (step_t < 1) return fail(ZERO_ERR_INVALID_ARG, "step_t must be >= 1");
    if (n_threads < 0) return fail(ZERO_ERR_INVALID_ARG, "n_threads must be >= 0");
    if (param_dtype != ZERO_F16 && param_dtype != ZERO_BF16)
        return fail(ZERO_ERR_UNSUPPORTED_DTYPE, "param dtype must be ZERO_F16 or ZERO_BF16");
    if (n > 0 && (!g || !master || !m || !v || !param_out))
        return fail(ZERO_ERR_INVALID_ARG, "NULL array");
    if ((uintptr_t)g % 4 || (uintptr_t)master % 4 || (uintptr_t)m % 4 || (uintptr_t)v % 4 ||
        (uintptr_t)param_out % 2)
        return fail(ZERO_ERR_ALIGNMENT, "fp32 arrays must be 4-byte and param_out 2-byte aligned");
    if (n == 0) return ZERO_OK;
    const zh::AdamScalars k{(float)hp->beta1, (float)hp->beta2, (float)(1.0 - hp->beta1),
                            (float)(1.0 - hp->beta2), (float)hp->lr, (float)hp->eps,
                            (float)(1.0 - hp->lr * hp->weight_decay), clip_coef,
                            (float)(1.0 - std::pow(hp->beta1, (double)step_t)),
                            (float)(1.0 - std::pow(hp->beta2, (double)step_t))};
    const bool bf16 = param_dtype == ZERO_BF16;
    uint16_t *out = static_cast<uint16_t *>(param_out);
    const int want = n_threads > 0 ? n_threads : zh::available_cpus();
    const int64_t chunks = (n + kHostChunk - 1) / kHostChunk;
    const std::function<void(int64_t)> task = [&](int64_t c) {
        const int64_t i0 = c * kHostChunk;
        zh::adamw_cast_range(k, g + i0, master + i0, m + i0, v + i0, out + i0,
                             std::min(kHostChunk, n - i0), bf16);
    };
    if (want <= 1 || chunks == 1) {
        for (int64_t c = 0; c < chunks; ++c) task(c);
        return ZERO_OK;
    }
    zh::Pool pool(std::min<int64_t>(want, chunks));
    pool.run(chunks, task);
    return ZERO_OK;
}

ZERO_API zero_status zero_debug_set_stage_tx_pad(uint32_t bytes) {
    zg::set_stage_tx_pad(bytes);
    return ZERO_OK;
}

ZERO_API zero_status zero_debug_reduce_form(zero_dtype grad_dtype, int32_t n_contrib,
                                            int32_t n_rows, const uint64_t *in_addr,
                                            const int64_t *ld, const int64_t *shard,
                                            const uint64_t *acc_addr, int32_t mode,
                                            int32_t *staged) {
    if (!staged || !in_addr || !ld || !shard || n_rows < 1 || n_contrib < 1)
        return fail(ZERO_ERR_INVALID_ARG, "NULL output or rows, or no rows or contributors");
    if (grad_dtype != ZERO_F16 && grad_dtype != ZERO_BF16 && grad_dtype != ZERO_F32)
        return fail(ZERO_ERR_INVALID_ARG, "unknown contribution dtype");
    if (mode < 0 || mode > 2) return fail(ZERO_ERR_INVALID_ARG, "mode must be 0, 1 or 2");
    if (mode != 0 && !acc_addr) return fail(ZERO_ERR_INVALID_ARG, "accumulator addresses missing");
    std::vector<zg::ReduceRow> rows((size_t)n_rows);
    for (int32_t j = 0; j < n_rows; ++j) {
        rows[j].in = reinterpret_cast<const void *>((uintptr_t)in_addr[j]);
        rows[j].ld = ld[j];
        rows[j].S = shard[j];
        rows[j].valid = shard[j];
        rows[j].acc = mode ? reinterpret_cast<float *>((uintptr_t)acc_addr[j]) : nullptr;
    }
    const int kind = grad_dtype == ZERO_F32 ? zg::kInF32
                                            : (grad_dtype == ZERO_BF16 ? zg::kInBF16 : zg::kInF16);
    const int m = mode == 0 ? zg::kModeStep : (mode == 1 ? zg::kModeAccFirst : zg::kModeAccAdd);
    *staged = zg::rows_want_staging(m, kind, n_contrib, rows.data(), n_rows) ? 1 : 0;
    return ZERO_OK;
}

ZERO_API zero_status zero_flat_set_lr(zero_flat *h, double lr) {
    if (!h) return fail(ZERO_ERR_INVALID_ARG, "handle is NULL");
    if (!std::isfinite(lr) || lr < 0) return fail(ZERO_ERR_INVALID_ARG, "lr must be finite and >= 0");
    h->hp.lr = lr;
    h->lr = (float)lr;
    h->decay = (float)(1.0 - lr * h->hp.weight_decay);
    return ZERO_OK;
}

ZERO_API zero_status zero_loss_scaler_state(zero_flat *h, zero_scaler_state *out, void *stream) {
    if (!h || !out) return fail(ZERO_ERR_INVALID_ARG, "NULL argument");
    DeviceGuard guard(h->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the handle's device");
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(h->h_state, h->d_state, sizeof(zg::DevState),
                                    cudaMemcpyDeviceToHost, st);
    if (!e) e = cudaStreamSynchronize(st);
    if (e) return cuda_fail(e, "reading the loss-scale state");
    out->scale = h->h_state->scaler.scale;
    out->good_steps = h->h_state->scaler.good_steps;
    out->step_t = h->h_state->scaler.step_t;
    out->overflow_count = h->h_state->scaler.overflow_count;
    return ZERO_OK;
}

ZERO_API zero_status zero_set_loss_scaler_state(zero_flat *h, const zero_scaler_state *in,
                                                void *stream) {
    if (!h || !in) return fail(ZERO_ERR_INVALID_ARG, "NULL argument");
    if (!(in->scale > 0.0f) || !std::isfinite(in->scale) || in->good_steps < 0 ||
        in->step_t < 0 || in->overflow_count < 0)
        return fail(ZERO_ERR_INVALID_ARG, "invalid loss-scale state");
    DeviceGuard guard(h->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the handle's device");
    cudaStream_t st = (cudaStream_t)stream;
    // stage through the pinned buffer after earlier work on the stream is done
    cudaError_t e = cudaStreamSynchronize(st);
    if (e) return cuda_fail(e, "cudaStreamSynchronize");
    zg::ScalerDev sc{in->scale, in->good_steps, in->step_t, in->overflow_count};
    memcpy(&h->h_state->scaler, &sc, sizeof(sc));
    e = cudaMemcpyAsync(&h->d_state->scaler, &h->h_state->scaler, sizeof(sc),
                        cudaMemcpyHostToDevice, st);
    if (!e) e = cudaStreamSynchronize(st);
    if (e) return cuda_fail(e, "writing the loss-scale state");
    return ZERO_OK;
}

// ------------------------------------------------------------------ groups
ZERO_API zero_status zero_flat_profile_enable(zero_flat *h, int32_t enable) {
    if (!h) return fail(ZERO_ERR_INVALID_ARG, "handle is NULL");
    if (h->ev_used % 4) return fail(ZERO_ERR_INVALID_ARG, "timing record is inconsistent");
    h->profile = enable != 0;
    return ZERO_OK;
}

ZERO_API zero_status zero_flat_profile_read(zero_flat *h, double *ms_reduce, double *ms_finalize,
                                            double *ms_adamw, int64_t *steps) {
    if (!h) return fail(ZERO_ERR_INVALID_ARG, "handle is NULL");
    DeviceGuard guard(h->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the handle's device");
    double t[3] = {0, 0, 0};
    const size_t n = h->ev_used / 4;
    for (size_t k = 0; k < n; ++k) {
        cudaError_t e = cudaEventSynchronize(h->ev[4 * k + 3]);
        if (e) return cuda_fail(e, "cudaEventSynchronize");
        for (int i = 0; i < 3; ++i) {
            float ms = 0;
            e = cudaEventElapsedTime(&ms, h->ev[4 * k + i], h->ev[4 * k + i + 1]);
            if (e) return cuda_fail(e, "cudaEventElapsedTime");
            t[i] += ms;
        }
    }
    h->ev_used = 0;
    if (ms_reduce) *ms_reduce = t[0];
    if (ms_finalize) *ms_finalize = t[1];
    if (ms_adamw) *ms_adamw = t[2];
    if (steps) *steps = (int64_t)n;
    return ZERO_OK;
}

ZERO_API zero_status zero_flat_profile_reduce_form(const zero_flat *h, int32_t *staged) {
    if (!h || !staged) return fail(ZERO_ERR_INVALID_ARG, "handle or output is NULL");
    *staged = h->last_reduce_staged;
    return ZERO_OK;
}

ZERO_API zero_status zero_flat_free(zero_flat *h) {
    if (!h) return ZERO_OK;
    {
        DeviceGuard guard(h->device);
        cudaDeviceSynchronize();
    }
    release(h);
    return ZERO_OK;
}
