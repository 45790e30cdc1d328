// zero_noalloc.cu -- zero_shard_step_noalloc: the shard step for callers that
// are not allowed to allocate device memory.
//
// Who needs it: code that runs while allocation is off limits -- inside a
// framework whose caching allocator owns all device memory and forbids side
// allocations, in runtimes that pre-plan every byte up front, or in callbacks
// and service loops where a cudaMalloc would synchronize the device or could
// fail at an unrecoverable moment.  Such callers cannot create a zero_flat
// handle (zero_flat_init allocates the loss-scale state, the bias-correction
// table and, on the first step, the reduced-gradient scratch).
//
// This entry point allocates nothing.  Its scratch -- the fp32 reduced-
// gradient rows, the per-block norm partials and the step's scalars -- lives
// in one file-scope __device__ array of ZERO_NOALLOC_SCRATCH_BYTES (32 MiB),
// which the CUDA runtime places on every device that loads this library and
// keeps until the process exits.  The loss-scale state stays with the caller
// in host memory and is passed in and returned on every call.
//
// Sharing: every call on a device uses the same array, which keeps whatever
// the last call left in it.  Each call therefore starts by overwriting the
// whole state block with the caller's loss-scale state and zeros -- among
// them the error word, which a staged reduce sets when one of its bounded
// waits gives up and which the decision reads (a set word skips the step).
// The reduce kernel then writes every gradient element and every partial
// that the later kernels read.  Calls whose GPU work overlaps (several host
// threads, or several streams without ordering) race on the array and give
// wrong results; callers must order them.
//
// Set-up: the first call on a device looks up the array's device address
// (cudaGetSymbolAddress, with that device current) and the launch geometry,
// and caches them; make that first call before any stream capture.
#include "zero.h"
#include "zero_plan.h"

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#define ZERO_API extern "C" __attribute__((visibility("default")))

// Sets the message zero_last_error() returns (defined in zero_api.cu).
void zero_internal_set_error(const char *msg);

namespace {

constexpr size_t kScratchBytes = ZERO_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxParts = 8192;                       // norm partials (blocks x ranks)
constexpr size_t kStateOff = 0;                       // zg::DevState
constexpr size_t kPartSsOff = 256;                    // kMaxParts doubles
constexpr size_t kPartOfOff = kPartSsOff + kMaxParts * sizeof(double);
constexpr size_t kGradOff = (kPartOfOff + kMaxParts * sizeof(int32_t) + 255) / 256 * 256;
constexpr int64_t kGradFloats = (int64_t)((kScratchBytes - kGradOff) / sizeof(float));
constexpr int kMaxDevices = 64;
static_assert(sizeof(zg::DevState) <= kPartSsOff, "state region too small");

// The scratch.  Host code must not use this name as an address: it refers to
// a host-side stand-in.  The device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceSetup {
    bool done;
    unsigned char *base;              // device address of g_noalloc_scratch
    int sm_count;
    int reduce_bps[3];                // per contribution encoding (InKind)
    int staged_bps[3];                // the staged reduce, per encoding
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mu;

zero_status fail(zero_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    zero_internal_set_error(buf);
    return s;
}

zero_status cuda_fail(cudaError_t e, const char *what) {
    return fail(ZERO_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

zero_status setup_device(int dev, const DeviceSetup **out) {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    DeviceSetup &d = g_setup[dev];
    if (!d.done) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        if (!p) return fail(ZERO_ERR_CUDA, "static scratch has no device address");
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        for (int kind = 0; kind < 3; ++kind) {
            e = zg::reduce_blocks_per_sm(kind, zg::kModeStep, false, &d.reduce_bps[kind]);
            if (e == cudaSuccess)
                e = zg::reduce_blocks_per_sm(kind, zg::kModeStep, true, &d.staged_bps[kind]);
            if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
        }
        d.base = static_cast<unsigned char *>(p);
        d.done = true;
    }
    *out = &d;
    return ZERO_OK;
}

bool hparams_ok(const zero_hparams *hp) {
    auto fin = [](double x) { return std::isfinite(x); };
    return hp && fin(hp->lr) && hp->lr >= 0 && fin(hp->beta1) && hp->beta1 >= 0 &&
           hp->beta1 < 1 && fin(hp->beta2) && hp->beta2 >= 0 && hp->beta2 < 1 &&
           fin(hp->eps) && hp->eps > 0 && fin(hp->weight_decay) && hp->weight_decay >= 0 &&
           fin(hp->max_grad_norm) && (hp->dynamic_loss_scale == 0 || hp->dynamic_loss_scale == 1) &&
           hp->initial_scale_power >= 0 && hp->initial_scale_power <= 126 &&
           hp->loss_scale_window >= 1 && hp->reserved == 0 && fin(hp->min_loss_scale) &&
           (float)hp->min_loss_scale > 0 &&
           (hp->dynamic_loss_scale || (fin(hp->static_loss_scale) &&
                                       (float)hp->static_loss_scale > 0 &&
                                       std::isfinite((float)hp->static_loss_scale)));
}

}  // namespace

ZERO_API zero_status zero_shard_step_noalloc(
    int64_t full_numel, int32_t world_size, zero_dtype grad_dtype, zero_dtype param_dtype,
    zero_reduce_op op, const zero_hparams *hp, zero_scaler_state *state, const int32_t *ranks,
    int32_t n_ranks, const void *grads, int64_t grad_ld, int64_t grad_rank_offset_mul,
    float *const *master, float *const *m, float *const *v, void *flat_param_out,
    double extra_norm_sq, void *stream, zero_step_result *res) {
    // ---- arguments (host only; nothing is launched on an error)
    if (full_numel < 0 || world_size < 1) return fail(ZERO_ERR_INVALID_ARG, "bad layout");
    if ((grad_dtype != ZERO_F16 && grad_dtype != ZERO_BF16 && grad_dtype != ZERO_F32) ||
        (param_dtype != ZERO_F16 && param_dtype != ZERO_BF16))
        return fail(ZERO_ERR_UNSUPPORTED_DTYPE,
                    "grad dtype must be ZERO_F16, ZERO_BF16 or ZERO_F32; param dtype ZERO_F16 or ZERO_BF16");
    if (op != ZERO_SUM && op != ZERO_AVG) return fail(ZERO_ERR_INVALID_ARG, "op must be SUM or AVG");
    if (!hparams_ok(hp)) return fail(ZERO_ERR_INVALID_ARG, "invalid hyper-parameters");
    if (!state || !(state->scale > 0.0f) || !std::isfinite(state->scale) ||
        state->good_steps < 0 || state->step_t < 0 || state->overflow_count < 0)
        return fail(ZERO_ERR_INVALID_ARG, "invalid loss-scale state");
    if (!ranks || n_ranks < 1 || n_ranks > world_size || n_ranks > zg::kMaxRanksPerLaunch)
        return fail(ZERO_ERR_INVALID_ARG, "need 1..min(world_size, %d) stepped ranks",
                    zg::kMaxRanksPerLaunch);
    for (int32_t j = 0; j < n_ranks; ++j) {
        if (ranks[j] < 0 || ranks[j] >= world_size)
            return fail(ZERO_ERR_INVALID_ARG, "rank %d out of range", ranks[j]);
        for (int32_t k = 0; k < j; ++k)
            if (ranks[k] == ranks[j]) return fail(ZERO_ERR_INVALID_ARG, "rank %d listed twice", ranks[j]);
    }
    if (!master || !m || !v || !flat_param_out)
        return fail(ZERO_ERR_INVALID_ARG, "NULL state or output pointer");
    if (!std::isfinite(extra_norm_sq) || extra_norm_sq < 0)
        return fail(ZERO_ERR_INVALID_ARG, "extra_norm_sq must be finite and >= 0");
    const int64_t S = full_numel / world_size + (full_numel % world_size != 0);
    if (grad_ld < 0 || grad_rank_offset_mul < 0 || (world_size > 1 && grad_ld < S))
        return fail(ZERO_ERR_INVALID_ARG, "grad_ld must be >= shard_size");
    if (S > 0 && !grads) return fail(ZERO_ERR_INVALID_ARG, "grads is NULL");
    const size_t esize = grad_dtype == ZERO_F32 ? 4 : 2;
    if ((uintptr_t)grads % esize || (uintptr_t)flat_param_out % 2)
        return fail(ZERO_ERR_ALIGNMENT,
                    "grads must be aligned to their element size, flat_param_out to 2 bytes");
    int32_t rmax = 0;
    for (int32_t j = 0; j < n_ranks; ++j) {
        if (ranks[j] > rmax) rmax = ranks[j];
        if (S > 0 && (!master[j] || !m[j] || !v[j]))
            return fail(ZERO_ERR_INVALID_ARG, "master/m/v pointer %d is NULL", j);
        if ((uintptr_t)master[j] % 4 || (uintptr_t)m[j] % 4 || (uintptr_t)v[j] % 4)
            return fail(ZERO_ERR_ALIGNMENT, "master/m/v must be 4-byte aligned");
    }
    const double span = (double)(world_size - 1) * (double)grad_ld +
                        (double)rmax * (double)grad_rank_offset_mul + (double)S;
    if (S > INT64_MAX / world_size || span >= 9.0e18)
        return fail(ZERO_ERR_OVERFLOW_SIZE, "sizes overflow int64");
    const int64_t g_stride = (S + 3) / 4 * 4;
    if (g_stride > kGradFloats / n_ranks)
        return fail(ZERO_ERR_INVALID_ARG,
                    "too large for the static scratch: %d shard(s) of %lld params need %lld "
                    "floats of reduced-gradient scratch, the %u-byte array holds %lld",
                    n_ranks, (long long)S, (long long)(g_stride * n_ranks),
                    (unsigned)kScratchBytes, (long long)kGradFloats);

    // ---- device set-up (first call on this device)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(ZERO_ERR_INVALID_ARG, "device index too large");
    const DeviceSetup *d = nullptr;
    zero_status s = setup_device(dev, &d);
    if (s != ZERO_OK) return s;

    // ---- launch geometry (as zero_shard_step computes it)
    const int in_kind = grad_dtype == ZERO_F32 ? zg::kInF32
                      : (grad_dtype == ZERO_BF16 ? zg::kInBF16 : zg::kInF16);
    zg::ReducePlan rp;
    rp.mode = zg::kModeStep;
    rp.grads = grads;
    rp.in_kind = in_kind;
    rp.ld = grad_ld;
    rp.rank_mul = grad_rank_offset_mul;
    rp.ranks = ranks;
    rp.n_ranks = n_ranks;
    rp.S = S;
    rp.n_contrib = world_size;
    rp.staged = zg::reduce_wants_staging(rp);
    const int gx1 = zg::grid_x_for(S, n_ranks, d->sm_count,
                                   rp.staged ? d->staged_bps[in_kind] : d->reduce_bps[in_kind]);
    const int gx3 = zg::grid_x_for(S, n_ranks, d->sm_count, zg::kAdamBlocksPerSm);
    const int64_t parts = (int64_t)gx1 * n_ranks;
    if (parts > kMaxParts) return fail(ZERO_ERR_INVALID_ARG, "too many norm partials");

    unsigned char *base = d->base;
    zg::DevState *dstate = reinterpret_cast<zg::DevState *>(base + kStateOff);
    double *part_ss = reinterpret_cast<double *>(base + kPartSsOff);
    int32_t *part_of = reinterpret_cast<int32_t *>(base + kPartOfOff);
    float *gbuf = reinterpret_cast<float *>(base + kGradOff);
    cudaStream_t st = (cudaStream_t)stream;

    // bias corrections of the step this call would apply (t + 1), in fp64 via
    // pow and rounded once to fp32, as the handle's table holds them
    const double t1 = (double)(state->step_t + 1);
    const float bc1 = (float)(1.0 - std::pow(hp->beta1, t1));
    const float bc2 = (float)(1.0 - std::pow(hp->beta2, t1));

    // the whole state block: the caller's loss-scale state, everything else
    // zero (the error word included, whatever an earlier call left there)
    zg::DevState init{};
    init.scaler = zg::ScalerDev{state->scale, state->good_steps, state->step_t,
                                state->overflow_count};
    e = cudaMemcpyAsync(dstate, &init, sizeof(init), cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "writing the loss-scale state");

    rp.g = gbuf;
    rp.g_stride = g_stride;
    rp.part_ss = part_ss;
    rp.part_of = part_of;
    rp.full_numel = full_numel;
    rp.avg = op == ZERO_AVG;
    rp.st = dstate;
    rp.grid_x = gx1;
    if ((e = zg::run_reduce(rp, st)) != cudaSuccess) return cuda_fail(e, "reduce kernel launch");
    // the decision kernel of zero_shard_step, with this step's bias
    // corrections by value instead of from a table
    zg::FinalizeArgs f{};
    f.part_ss = part_ss;
    f.part_of = part_of;
    f.n_parts = S > 0 ? (int32_t)parts : 0;
    f.dynamic = hp->dynamic_loss_scale;
    f.window = hp->loss_scale_window;
    f.min_scale = (float)hp->min_loss_scale;
    f.extra_norm_sq = extra_norm_sq;
    f.max_grad_norm = hp->max_grad_norm;
    f.bc_table = nullptr;
    f.bc_given = make_float2(bc1, bc2);
    f.st = dstate;
    if ((e = zg::launch_finalize(f, st)) != cudaSuccess) return cuda_fail(e, "finalize kernel launch");
    zg::AdamPlan ap;
    ap.g = gbuf;
    ap.g_stride = g_stride;
    ap.master = master;
    ap.m = m;
    ap.v = v;
    ap.out = flat_param_out;
    ap.bf16_out = param_dtype == ZERO_BF16;
    ap.ranks = ranks;
    ap.n_ranks = n_ranks;
    ap.S = S;
    ap.full_numel = full_numel;
    ap.b1 = (float)hp->beta1;
    ap.b2 = (float)hp->beta2;
    ap.omb1 = (float)(1.0 - hp->beta1);
    ap.omb2 = (float)(1.0 - hp->beta2);
    ap.lr = (float)hp->lr;
    ap.eps = (float)hp->eps;
    ap.decay = (float)(1.0 - hp->lr * hp->weight_decay);
    ap.st = dstate;
    ap.grid_x = gx3;
    if ((e = zg::run_adamw(ap, st)) != cudaSuccess) return cuda_fail(e, "adamw kernel launch");

    // ---- the new loss-scale state and the result back to the caller
    zg::DevState out_state;
    e = cudaMemcpyAsync(&out_state, dstate, sizeof(out_state), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "reading the step result");
    state->scale = out_state.scaler.scale;
    state->good_steps = out_state.scaler.good_steps;
    state->step_t = out_state.scaler.step_t;
    state->overflow_count = out_state.scaler.overflow_count;
    if (res) {
        res->overflow = out_state.res.overflow;
        res->skipped = out_state.res.skipped;
        res->grad_norm = out_state.res.grad_norm;
        res->clip_coef = out_state.res.clip_coef;
        res->scale_used = out_state.res.scale_used;
    }
    if (out_state.error)                 // a bounded wait gave up: the step was skipped
        return fail(ZERO_ERR_TIMEOUT, "a kernel gave up waiting for its bulk copies; the step was skipped");
    return ZERO_OK;
}
