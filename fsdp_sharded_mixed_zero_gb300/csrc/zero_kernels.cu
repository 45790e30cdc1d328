// zero_kernels.cu -- the kernels of one ZeRO shard step on sm_103a.
//
//   K1 reduce_kernel    N-way reduce of the fp16/bf16/fp32 gradient contributions of
//                       each stepped shard, AVG, loss-scale division, inf/NaN
//                       check and per-block partial sums of squares; writes
//                       the fp32 reduced gradient row (the reduce half of a
//                       reduce-scatter: "PyTorch FSDP ... 深度解析" §3.3;
//                       sum-then-split in the numpy demo of "DeepSpeed 与
//                       FSDP"; fp32 reduce per its MixedPrecision example).
//   K1 reduce_staged_kernel  the same for contributor rows that are not
//                       64-byte aligned, and for reduces that read at least
//                       1 GiB of contributions: a producer warp's TMA bulk
//                       copies of 64-byte-aligned spans into shared memory,
//                       re-aligned there by the consumer warps.
//   K2 the decision     fixed-order total of the partials, global norm, clip
//                       coefficient, overflow skip and the dynamic loss-scale
//                       state machine (ZeRO reading §5.1, §5.3): made by the
//                       K1 block that finishes last (finalize_block), or by
//                       finalize_kernel when there is no reduce to count in.
//   K3 adamw_kernel     AdamW with bias correction and decoupled weight decay
//                       on fp32 master/m/v ("DeepSpeed 与 FSDP" §ZeRO-Offload
//                       equations, §ZeRO-1 step 2) and the round-to-nearest
//                       cast into the rank's slot of the flat buffer (§ZeRO-1
//                       step 3: the slot the all-gather distributes).
//
// Everything is HBM-bound streaming (well under 1 flop per byte): no tensor
// cores.  Each 16-bit contribution and each fp32 state word crosses HBM once
// per step; the only extra traffic is the fp32 reduced gradient (written by
// K1, read by K3), forced by the global norm / skip decision that every
// update depends on.
//
// Arithmetic: every fp32 operation is an explicit round-to-nearest intrinsic
// (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn), so nothing is contracted
// into an FMA and each result is the IEEE-754 binary32 result of the written
// expression in the written order (the only FMAs are the explicit ones that
// give the exact rounding error of a square in the norm).  Division by a power of two is done as a
// multiplication by its exact reciprocal, which has the same exact value and
// therefore the same correctly rounded result.
#include "zero_kernels.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace zg {
namespace {

// ------------------------------------------------------------------ memory
// 16-byte loads of data that no thread writes during the kernel.
__device__ __forceinline__ uint4 ld_nc_u4(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}
__device__ __forceinline__ float4 ld_nc_f4(const float *p) {
    float4 r;
    asm("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
        : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
        : "l"(p));
    return r;
}
// 16-byte load of state this thread later overwrites (coherent path).
__device__ __forceinline__ float4 ld_f4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ void st_f4(float *p, float4 v) {
    *reinterpret_cast<float4 *>(p) = v;
}

// ------------------------------------------------------------------ formats
template <bool kBf16>
__device__ __forceinline__ float to_f32(uint16_t h) {
    if constexpr (kBf16) {
        return __uint_as_float((uint32_t)h << 16);
    } else {
        return __half2float(__ushort_as_half(h));
    }
}

// Eight 16-bit values (one 16-byte word) to fp32, element order preserved.
template <bool kBf16>
__device__ __forceinline__ void unpack8(const uint4 &w, float f[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if constexpr (kBf16) {
            f[2 * k] = __uint_as_float(u[k] << 16);
            f[2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
        } else {
            const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&u[k]));
            f[2 * k] = x.x;
            f[2 * k + 1] = x.y;
        }
    }
}

// Round-to-nearest-even casts (hardware cvt.rn).
template <bool kBf16>
__device__ __forceinline__ uint16_t from_f32(float x) {
    if constexpr (kBf16) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(x));
    } else {
        return __half_as_ushort(__float2half_rn(x));
    }
}
template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    return (uint32_t)from_f32<kBf16>(lo) | ((uint32_t)from_f32<kBf16>(hi) << 16);
}

// ------------------------------------------------------------------ division
// x / d for d > 0.  A normal power of two has an exact reciprocal, and
// x * (1/d) then equals x / d exactly before rounding.
struct Divisor {
    float d;
    float inv;
    bool pow2;
};
__device__ __forceinline__ Divisor make_divisor(float d) {
    const uint32_t u = __float_as_uint(d);
    const uint32_t e = (u >> 23) & 0xFFu;
    const bool pow2 = (u & 0x807FFFFFu) == 0u && e >= 1u && e <= 254u;
    return {d, pow2 ? __fdiv_rn(1.0f, d) : 0.0f, pow2};
}
__device__ __forceinline__ float divide(float x, const Divisor &q) {
    return q.pow2 ? __fmul_rn(x, q.inv) : __fdiv_rn(x, q.d);
}

// ------------------------------------------------------------------ norm
// The squared norm must be accurate to ~1e-14 so that the fp32 clip
// coefficient derived from it rounds like the exactly computed one.  Per
// 8-element chunk the squares are summed without error in fp32 pairs: the
// exact square of x is p + e with p = x*x and e = fma(x, x, -p), and Knuth's
// TwoSum gives the exact error of every addition; only the small correction
// term is rounded (relative error ~ eps^2).  A thread carries that pair over
// eight chunks before one fp64 addition, because GB300's fp64 rate is low
// enough that an fp64 add per chunk would bound a read-only pass.  Chunks
// whose sum lies outside [2^-100, 2^100] (where fp32 squares could overflow
// or lose their low bits), or that hold inf/NaN, are summed exactly in fp64.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &err) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

struct NormAcc {
    double ss = 0.0;                  // flushed total
    float hi = 0.0f, lo = 0.0f;       // carried pair
    int n = 0;                        // chunks in the pair

    __device__ __forceinline__ void flush() {
        ss += (double)hi + (double)lo;
        hi = 0.0f;
        lo = 0.0f;
        n = 0;
    }
    __device__ __forceinline__ void add_chunk(const float x[kVec]) {
        float ch = __fmul_rn(x[0], x[0]);
        float cl = __fmaf_rn(x[0], x[0], -ch);
#pragma unroll
        for (int k = 1; k < kVec; ++k) {
            const float p = __fmul_rn(x[k], x[k]);
            const float e = __fmaf_rn(x[k], x[k], -p);
            float t;
            two_sum(ch, p, ch, t);
            cl = __fadd_rn(cl, __fadd_rn(t, e));
        }
        if (ch >= 0x1p-100f && ch <= 0x1p100f) {
            float t;
            two_sum(hi, ch, hi, t);
            lo = __fadd_rn(lo, __fadd_rn(t, cl));
            if (++n == 8) flush();
        } else {
            // out of range, inf/NaN, or zero squares: zero squares may come
            // from nonzero values below 2^-75, so test the values themselves
            bool any = false;
#pragma unroll
            for (int k = 0; k < kVec; ++k) any |= x[k] != 0.0f;
            if (any) {
#pragma unroll
                for (int k = 0; k < kVec; ++k) ss += (double)x[k] * (double)x[k];
            }
        }
    }
    __device__ __forceinline__ void add_exact(float x) { ss += (double)x * (double)x; }
    __device__ __forceinline__ double total() {
        flush();
        return ss;
    }
};

// ------------------------------------------------------------------ reduction
// Block total of per-thread fp64 sums and flags, in a fixed order.
__device__ __forceinline__ void block_partial(double ss, int of, double *out_ss,
                                              int32_t *out_of) {
    __shared__ double warp_ss[32];
    of = __syncthreads_or(of);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_down_sync(0xFFFFFFFFu, ss, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) warp_ss[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += warp_ss[w];
        *out_ss = t;
        *out_of = of;
    }
}

// ------------------------------------------------------------------ decision
// The step's decision from the norm partials, by one block of up to 1024
// threads: fixed-order fp64 total of the partials (strided per thread, then
// a warp tree, then the warps in order), global norm, clip coefficient,
// overflow skip and the dynamic loss-scale state machine (ZeRO reading §5.1,
// §5.3); the bias corrections of an applied step come from the table, or by
// value when there is none.
// Partials are read through L2 (another block may have written them).
__device__ void finalize_block(const FinalizeArgs &a) {
    __shared__ double warp_ss[kFinalizeThreads / 32];
    DevState *st = a.st;
    ScalerDev sc{};
    float2 bc = make_float2(1.0f, 1.0f);
    if (threadIdx.x == 0) {               // independent of the partials: load early
        sc = st->scaler;
        const int64_t t1 = sc.step_t + 1;
        if (!a.bc_table) bc = a.bc_given;
        else if (t1 < a.bc_len) bc = a.bc_table[t1];
    }
    double s = 0.0;
    int of = 0;
    for (int i = threadIdx.x; i < a.n_parts; i += blockDim.x) {
        s += __ldcg(a.part_ss + i);
        of |= __ldcg(a.part_of + i);
    }
    of = __syncthreads_or(of);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xFFFFFFFFu, s, o);
    if ((threadIdx.x & 31) == 0) warp_ss[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x != 0) return;
    double total = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) total += warp_ss[w];
    // a kernel that gave up a bounded wait since the error word was last
    // read (e.g. an accumulation launch, which has no partials) voids the step
    if (__ldcg(&st->error)) of = 1;
    if (a.sum_out) {                       // first half of a split step
        *a.sum_out = total;
        *a.of_out = of;
        return;
    }

    ResultDev r;
    r.overflow = of;
    r.grad_norm = sqrt(total + a.extra_norm_sq);
    r.scale_used = sc.scale;
    if (of) {                              // skip the step, shrink the scale
        r.skipped = 1;
        r.clip_coef = 1.0f;
        sc.overflow_count += 1;
        if (a.dynamic) {
            const float h = __fdiv_rn(sc.scale, 2.0f);
            sc.scale = h < a.min_scale ? a.min_scale : h;
            sc.good_steps = 0;
        }
    } else {
        r.skipped = 0;
        sc.step_t += 1;
        float coef = 1.0f;
        if (a.max_grad_norm > 0.0) {
            const double q = a.max_grad_norm / (r.grad_norm + 1e-6);
            if (q < 1.0) coef = (float)q;
        }
        r.clip_coef = coef;
        if (a.dynamic) {                   // grow after `window` clean steps
            sc.good_steps += 1;
            if (sc.good_steps == a.window) {
                sc.scale = __fmul_rn(sc.scale, 2.0f);
                sc.good_steps = 0;
            }
        }
        st->bc1 = bc.x;                    // entry t of the table (t = the new step_t)
        st->bc2 = bc.y;
    }
    st->scaler = sc;
    st->res = r;
}

// After this block's partial is written: count the block; the block that
// completes the count (every block of every launch of the step has written
// its partial by then) makes the step's decision and re-arms the counter.
// No block waits for another.
__device__ __forceinline__ void count_and_finalize(const ReduceArgs &a) {
    __shared__ int last;
    if (threadIdx.x == 0) {
        __threadfence();                   // the partial before the count
        last = atomicAdd(a.done, 1u) == a.total_blocks - 1u;
    }
    __syncthreads();
    if (last) {
        __threadfence();                   // every counted block's partial is visible
        finalize_block(a.fin);
        if (threadIdx.x == 0) *a.done = 0u;
    }
}

// ------------------------------------------------------------------ K1
// Element traits of a contribution encoding: 16-byte words per 8 elements and
// contributor rows kept in flight per batch.
template <int kIn> struct InTraits {
    using T = uint16_t;
    static constexpr int kWords = 1;
    static constexpr int kBatch = 8;
};
template <> struct InTraits<kInF32> {
    using T = float;
    static constexpr int kWords = 2;
    static constexpr int kBatch = 4;
};

// Register budget: five resident blocks per SM (48 registers) except for the
// fp32-contribution reduce, whose four rows in flight need four (64).
template <int kIn, int kMode>
constexpr int reduce_min_blocks() {
    return (kIn == kInF32 && kMode != kModeNormOnly) ? 4 : 5;
}

template <int kIn>
__device__ __forceinline__ void load_words(const typename InTraits<kIn>::T *p, uint4 w[]) {
    w[0] = ld_nc_u4(p);
    if constexpr (InTraits<kIn>::kWords == 2) w[1] = ld_nc_u4(p + 4);
}

template <int kIn>
__device__ __forceinline__ void words_to_f32(const uint4 w[], float f[kVec]) {
    if constexpr (kIn == kInF32) {
        f[0] = __uint_as_float(w[0].x); f[1] = __uint_as_float(w[0].y);
        f[2] = __uint_as_float(w[0].z); f[3] = __uint_as_float(w[0].w);
        f[4] = __uint_as_float(w[1].x); f[5] = __uint_as_float(w[1].y);
        f[6] = __uint_as_float(w[1].z); f[7] = __uint_as_float(w[1].w);
    } else {
        unpack8<kIn == kInBF16>(w[0], f);
    }
}

template <int kIn>
__device__ __forceinline__ float elem_to_f32(const typename InTraits<kIn>::T *p) {
    if constexpr (kIn == kInF32) return *p;
    else return to_f32<kIn == kInBF16>(*p);
}

// kOneShape: the rows of the launch are one FlatParameter's -- the same
// contributor row stride and shard size, read as ld[0] and S[0], and evenly
// spaced gradient rows, g[0] + j * g_stride -- constant operands rather than
// registers held across the loops.
template <int kIn, int kMode, bool kOneShape = true>
__global__ void __launch_bounds__(kBlock, (reduce_min_blocks<kIn, kMode>()))
reduce_kernel(const __grid_constant__ ReduceArgs a) {
    using T = typename InTraits<kIn>::T;
    constexpr int kW = InTraits<kIn>::kWords;
    constexpr int kB = InTraits<kIn>::kBatch;
    constexpr bool kNorm = kMode == kModeStep || kMode == kModeNormOnly;
    const int j = blockIdx.y;
    const int64_t S = kOneShape ? a.S[0] : a.S[j];
    int64_t valid;                                // elements [valid, S) are padding
    if constexpr (kOneShape) {
        valid = a.full_numel - a.first[j];
        valid = valid < 0 ? 0 : (valid > S ? S : valid);
    } else {
        valid = a.valid[j];
    }
    const T *base = static_cast<const T *>(a.in[j]);
    float *g = kOneShape ? a.g[0] + (int64_t)j * a.g_stride : a.g[j];
    float *acc_out = a.acc[j];
    const int N = a.n_contrib;
    const int64_t ld = kOneShape ? a.ld[0] : a.ld[j];
    const bool avg = a.avg != 0;
    const Divisor dn = make_divisor((float)N);
    const Divisor ds = make_divisor(kNorm ? a.st->scaler.scale : 1.0f);

    // r of one element from its contributions, in contributor order from 0.
    auto finish = [&](float x) { return avg ? divide(x, dn) : x; };

    NormAcc na;
    int of = 0;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    int64_t done = 0;
    if constexpr (kMode == kModeNormOnly) {
        // A pure read stream of 4 bytes per element: keep two chunks (64
        // bytes) in flight per thread.  Chunks are still summed in the order
        // of the plain grid-stride loop: ch, ch + T, ch + 2T, ...
        if (a.vec[j]) {
            const float *acc_in = reinterpret_cast<const float *>(base);
            const int64_t nch = valid / kVec;
            int64_t ch = tid;
            for (; ch + nthreads < nch; ch += 2 * nthreads) {
                uint4 w[2][2];
#pragma unroll
                for (int u = 0; u < 2; ++u) load_words<kInF32>(acc_in + (ch + u * nthreads) * kVec, w[u]);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    float x[kVec];
                    words_to_f32<kInF32>(w[u], x);
#pragma unroll
                    for (int e = 0; e < kVec; ++e) {
                        x[e] = divide(x[e], ds);
                        of |= !isfinite(x[e]);
                    }
                    na.add_chunk(x);
                }
            }
            for (; ch < nch; ch += nthreads) {
                uint4 w[2];
                load_words<kInF32>(acc_in + ch * kVec, w);
                float x[kVec];
                words_to_f32<kInF32>(w, x);
#pragma unroll
                for (int e = 0; e < kVec; ++e) {
                    x[e] = divide(x[e], ds);
                    of |= !isfinite(x[e]);
                }
                na.add_chunk(x);
            }
            done = nch * kVec;
        }
    } else if (a.vec[j]) {
        const int64_t nch = valid / kVec;
        for (int64_t ch = tid; ch < nch; ch += nthreads) {
            const int64_t i0 = ch * kVec;
            float x[kVec];
            if constexpr (kMode == kModeNormOnly) {
                uint4 w[2];
                load_words<kInF32>(reinterpret_cast<const float *>(base) + i0, w);
                words_to_f32<kInF32>(w, x);
            } else {
                const T *p = base + i0;
#pragma unroll
                for (int e = 0; e < kVec; ++e) x[e] = 0.0f;
                int c = 0;
                for (; c + kB <= N; c += kB) {           // kB rows in flight
                    uint4 w[kB][kW];
#pragma unroll
                    for (int k = 0; k < kB; ++k) load_words<kIn>(p + (int64_t)(c + k) * ld, w[k]);
#pragma unroll
                    for (int k = 0; k < kB; ++k) {
                        float f[kVec];
                        words_to_f32<kIn>(w[k], f);
#pragma unroll
                        for (int e = 0; e < kVec; ++e) x[e] = __fadd_rn(x[e], f[e]);
                    }
                }
                for (; c < N; ++c) {
                    uint4 w[kW];
                    load_words<kIn>(p + (int64_t)c * ld, w);
                    float f[kVec];
                    words_to_f32<kIn>(w, f);
#pragma unroll
                    for (int e = 0; e < kVec; ++e) x[e] = __fadd_rn(x[e], f[e]);
                }
#pragma unroll
                for (int e = 0; e < kVec; ++e) x[e] = finish(x[e]);
            }
            if constexpr (kNorm) {
#pragma unroll
                for (int e = 0; e < kVec; ++e) {
                    x[e] = divide(x[e], ds);
                    of |= !isfinite(x[e]);
                }
                na.add_chunk(x);
            }
            if constexpr (kMode == kModeStep) {
                st_f4(g + i0, make_float4(x[0], x[1], x[2], x[3]));
                st_f4(g + i0 + 4, make_float4(x[4], x[5], x[6], x[7]));
            } else if constexpr (kMode == kModeAccFirst || kMode == kModeAccAdd) {
                if constexpr (kMode == kModeAccAdd) {
                    const float4 o0 = ld_f4(acc_out + i0), o1 = ld_f4(acc_out + i0 + 4);
                    const float o[kVec] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
#pragma unroll
                    for (int e = 0; e < kVec; ++e) x[e] = __fadd_rn(o[e], x[e]);
                }
                st_f4(acc_out + i0, make_float4(x[0], x[1], x[2], x[3]));
                st_f4(acc_out + i0 + 4, make_float4(x[4], x[5], x[6], x[7]));
            }
        }
        done = nch * kVec;
    }
    for (int64_t i = done + tid; i < valid; i += nthreads) {   // ragged tail / unaligned rows
        float x;
        if constexpr (kMode == kModeNormOnly) {
            x = reinterpret_cast<const float *>(base)[i];
        } else {
            x = 0.0f;
            for (int c = 0; c < N; ++c) x = __fadd_rn(x, elem_to_f32<kIn>(base + (int64_t)c * ld + i));
            x = finish(x);
        }
        if constexpr (kNorm) {
            x = divide(x, ds);
            of |= !isfinite(x);
            na.add_exact(x);                          // exact square in fp64
        }
        if constexpr (kMode == kModeStep) g[i] = x;
        if constexpr (kMode == kModeAccFirst) acc_out[i] = x;
        if constexpr (kMode == kModeAccAdd) acc_out[i] = __fadd_rn(acc_out[i], x);
    }
    for (int64_t i = valid + tid; i < S; i += nthreads) {     // padding: zero gradient
        if constexpr (kMode == kModeStep) g[i] = 0.0f;
        if constexpr (kMode == kModeAccFirst) acc_out[i] = 0.0f;
        if constexpr (kMode == kModeAccAdd) acc_out[i] = __fadd_rn(acc_out[i], 0.0f);
    }
    if constexpr (kNorm) {
        const int64_t pidx = a.part_base + (int64_t)j * gridDim.x + blockIdx.x;
        block_partial(na.total(), of, a.part_ss + pidx, a.part_of + pidx);
        if (a.fuse_finalize) count_and_finalize(a);
    }
}

// ------------------------------------------------------------------ K1, staged
// The reduce for contributor rows whose starts are not 64-byte aligned, and
// for launches large enough that its higher streaming rate outweighs its
// higher fixed cost.  For each block tile (kStageTile elements) and
// contributor row, one bulk copy
// (TMA, cp.async.bulk) brings the 64-byte-aligned span of global memory that
// covers the tile into a shared-memory slot, so DRAM sees only whole 64-byte
// units.  A thread then re-aligns its 8 elements from the slot (one 16-byte
// shared load when the row's offset is a multiple of 16 bytes, else two and a
// funnel shift).  Rows come in groups of kRows per stage, kStages stages in a
// ring.  One producer warp issues the copies -- one row per lane, after one
// lane has posted the stage's byte count on its `full` mbarrier -- and waits
// on the stage's `empty` mbarrier, on which each of the eight consumer warps
// arrives once it has read the stage; consumers wait on `full`.  No block-wide
// barrier sits inside the loop.  The arithmetic per element is that of
// reduce_kernel: contributions added in contributor order.
// Every wait is bounded (one second) and also ends when another warp has
// raised the block's abort flag; a block that gives up sets the error word,
// counts as an overflow (so the step is skipped) and waits, again bounded, for
// the copies it issued before it exits.
template <int kIn> struct StageTraits {
    static constexpr int kE = kIn == kInF32 ? 4 : 2;          // bytes per element
    // 4 KB-per-row tiles (8 KB for fp32), 4 rows (2 for fp32) per stage, 3
    // stages: 48 KB of copies in flight per block, 3 blocks per SM.  Measured
    // on GB300 against 8 rows x 2 stages: 10B reduce 3.68 -> 3.58 ms, GPT-2's
    // 0.391 -> 0.380, fp32 contributions 6.51 -> 6.39, the 64-contribution 1.5B
    // shard 0.508 -> 0.501, 2-byte-aligned rows at 1e8 params equal; 8 x 3
    // (2 blocks/SM), 4 x 4, 4 x 2, 2 x 4 and 2 x 6 slower.
    static constexpr int kRows = kIn == kInF32 ? 2 : 4;       // rows per stage
    static constexpr int kSlot = kStageTile * kE + 64;        // bytes per row slot
    static constexpr int kStages = 3;
    static constexpr int kHeader = 128;                       // mbarriers, abort flag
    static constexpr int kSmem = kHeader + kStages * kRows * kSlot;
    // full[kStages] and empty[kStages] (8 bytes each), then the abort flag:
    // all before the first slot
    static_assert(16 * kStages + 4 <= kHeader, "stage header overlaps the slots");
};
constexpr int kStagedThreads = kBlock + 32;                   // 8 consumer warps + 1 producer

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of `parity` to complete, for at most one second.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_test(bar, parity))
        if (global_ns() - t0 > 1000000000ull) return false;
    return true;
}
// The same, giving up early once *abort is set; a wait that runs out sets it.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity,
                                                   volatile int *abort) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_test(bar, parity)) {
        if (*abort) return false;
        if (global_ns() - t0 > 1000000000ull) {
            *abort = 1;
            return false;
        }
    }
    return true;
}
// Order this thread's earlier generic-proxy accesses of shared memory before
// later async-proxy (bulk copy) writes to it.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Bytes [o, o + 16) of the 32 bytes lo:hi (o a multiple of 2, below 16).
__device__ __forceinline__ uint4 bytes_at(const uint4 &lo, const uint4 &hi, uint32_t o) {
    const uint32_t u[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const uint32_t s = (o & 3u) * 8u;
    uint4 r;
    switch (o >> 2) {                  // uniform across the block for a given row
        case 0:
            r = make_uint4(__funnelshift_r(u[0], u[1], s), __funnelshift_r(u[1], u[2], s),
                           __funnelshift_r(u[2], u[3], s), __funnelshift_r(u[3], u[4], s));
            break;
        case 1:
            r = make_uint4(__funnelshift_r(u[1], u[2], s), __funnelshift_r(u[2], u[3], s),
                           __funnelshift_r(u[3], u[4], s), __funnelshift_r(u[4], u[5], s));
            break;
        case 2:
            r = make_uint4(__funnelshift_r(u[2], u[3], s), __funnelshift_r(u[3], u[4], s),
                           __funnelshift_r(u[4], u[5], s), __funnelshift_r(u[5], u[6], s));
            break;
        default:
            r = make_uint4(__funnelshift_r(u[3], u[4], s), __funnelshift_r(u[4], u[5], s),
                           __funnelshift_r(u[5], u[6], s), __funnelshift_r(u[6], u[7], s));
            break;
    }
    return r;
}

// This thread's 8 elements of one staged row, as fp32: the row's tile starts
// d bytes into its slot (d < 64, a multiple of the element size).
template <int kIn>
__device__ __forceinline__ void staged_elems(const unsigned char *slot, uint32_t d, float f[kVec]) {
    if constexpr (kIn == kInF32) {
        const uint32_t off = d + threadIdx.x * 32u;
        const uint32_t o = d & 15u;
        uint4 w0, w1;
        if (o == 0) {
            w0 = *reinterpret_cast<const uint4 *>(slot + off);
            w1 = *reinterpret_cast<const uint4 *>(slot + off + 16);
        } else {
            const unsigned char *p = slot + off - o;
            const uint4 a0 = *reinterpret_cast<const uint4 *>(p);
            const uint4 a1 = *reinterpret_cast<const uint4 *>(p + 16);
            const uint4 a2 = *reinterpret_cast<const uint4 *>(p + 32);
            w0 = bytes_at(a0, a1, o);
            w1 = bytes_at(a1, a2, o);
        }
        const uint4 w[2] = {w0, w1};
        words_to_f32<kInF32>(w, f);
    } else {
        const uint32_t off = d + threadIdx.x * 16u;
        const uint32_t o = d & 15u;
        uint4 w;
        if (o == 0) {
            w = *reinterpret_cast<const uint4 *>(slot + off);
        } else {
            const unsigned char *p = slot + off - o;
            w = bytes_at(*reinterpret_cast<const uint4 *>(p),
                         *reinterpret_cast<const uint4 *>(p + 16), o);
        }
        const uint4 ws[1] = {w};
        words_to_f32<kIn>(ws, f);
    }
}

template <int kIn, int kMode>
__global__ void __launch_bounds__(kStagedThreads, 3)
reduce_staged_kernel(const __grid_constant__ ReduceArgs a) {
    using T = typename InTraits<kIn>::T;
    using ST = StageTraits<kIn>;
    constexpr int kE = ST::kE, kR = ST::kRows, kSlot = ST::kSlot, kS = ST::kStages;
    constexpr bool kNorm = kMode == kModeStep;
    constexpr uint32_t kFull = 0xFFFFFFFFu;
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t full0 = smem_u32(smem);                    // full[s] at full0 + 8*s
    const uint32_t empty0 = full0 + 8u * kS;                  // empty[s] at empty0 + 8*s
    volatile int *abort = reinterpret_cast<volatile int *>(smem + 16 * kS);
    unsigned char *slots = smem + ST::kHeader;

    const int j = blockIdx.y;
    const int64_t S = a.S[j];
    const int64_t valid = a.valid[j];
    const T *base = static_cast<const T *>(a.in[j]);
    const unsigned char *bbase = static_cast<const unsigned char *>(a.in[j]);
    float *g = a.g[j];
    float *acc_out = a.acc[j];
    const int N = a.n_contrib;
    const int64_t ld = a.ld[j];
    const bool avg = a.avg != 0;
    const Divisor dn = make_divisor((float)N);
    const Divisor ds = make_divisor(kNorm ? a.st->scaler.scale : 1.0f);
    auto finish = [&](float x) { return avg ? divide(x, dn) : x; };

    const int groups = (N + kR - 1) / kR;
    const int64_t n_tiles = valid / kStageTile;
    const int64_t my_tiles =
        (int64_t)blockIdx.x < n_tiles ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t n_jobs = my_tiles * groups;           // job = (tile of this block, row group)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool producer = warp == kBlock / 32;

    // byte address of row c's element i (of this rank's slice)
    auto row_addr = [&](int c, int64_t i) {
        return bbase + ((int64_t)c * ld + i) * kE;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kS; ++s) {
            mbar_init(full0 + 8u * s, 1);                     // the producer's one arrive
            mbar_init(empty0 + 8u * s, kBlock / 32);          // one arrive per consumer warp
        }
        *abort = 0;
        mbar_init_fence();
    }
    __syncthreads();

    NormAcc na;
    int of = 0;
    int64_t issued = 0;                                       // producer: jobs issued
    if (producer) {
        for (int64_t job = 0; job < n_jobs; ++job) {
            const int stage = (int)(job % kS);
            if (job >= kS) {                                  // the stage's last readers are done
                const bool ok = mbar_wait_or_abort(empty0 + 8u * stage,
                                                   (uint32_t)((job / kS - 1) & 1), abort);
                if (!__all_sync(kFull, ok)) break;
            }
            const int64_t q = job / groups;
            const int gi = (int)(job - q * groups);
            const int64_t i0 = (blockIdx.x + q * gridDim.x) * (int64_t)kStageTile;
            const int c0 = gi * kR;
            const int nr = N - c0 < kR ? N - c0 : kR;
            uintptr_t lo = 0;
            uint32_t bytes = 0;
            if (lane < nr) {
                const uintptr_t A = (uintptr_t)row_addr(c0 + lane, i0);
                lo = A & ~(uintptr_t)63;
                bytes = (uint32_t)(((A + (uintptr_t)kStageTile * kE + 63) & ~(uintptr_t)63) - lo);
            }
            const uint32_t total = __reduce_add_sync(kFull, bytes);
            const uint32_t bar = full0 + 8u * stage;
            if (lane == 0) mbar_arrive_expect_tx(bar, total + a.tx_pad);
            __syncwarp();
            if (lane < nr) {
                fence_proxy_async();
                bulk_g2s(smem_u32(slots + (stage * kR + lane) * kSlot),
                         reinterpret_cast<const void *>(lo), bytes, bar);
            }
            issued = job + 1;
        }
    } else {
        float x[kVec];
        for (int64_t job = 0; job < n_jobs; ++job) {
            const int stage = (int)(job % kS);
            const bool ok = mbar_wait_or_abort(full0 + 8u * stage, (uint32_t)((job / kS) & 1),
                                               abort);
            if (!__all_sync(kFull, ok)) break;
            const int64_t q = job / groups;
            const int gi = (int)(job - q * groups);
            const int64_t t0 = (blockIdx.x + q * gridDim.x) * (int64_t)kStageTile;
            const int c0 = gi * kR;
            if (gi == 0) {
#pragma unroll
                for (int e = 0; e < kVec; ++e) x[e] = 0.0f;
            }
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                if (c0 + r < N) {                               // contributor order
                    const uint32_t d = (uint32_t)((uintptr_t)row_addr(c0 + r, t0) & 63u);
                    float f[kVec];
                    staged_elems<kIn>(slots + (stage * kR + r) * kSlot, d, f);
#pragma unroll
                    for (int e = 0; e < kVec; ++e) x[e] = __fadd_rn(x[e], f[e]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8u * stage);   // this warp is done reading
            if (gi == groups - 1) {                             // the tile's elements are reduced
                const int64_t i0 = t0 + (int64_t)threadIdx.x * kVec;
#pragma unroll
                for (int e = 0; e < kVec; ++e) x[e] = finish(x[e]);
                if constexpr (kNorm) {
#pragma unroll
                    for (int e = 0; e < kVec; ++e) {
                        x[e] = divide(x[e], ds);
                        of |= !isfinite(x[e]);
                    }
                    na.add_chunk(x);
                    st_f4(g + i0, make_float4(x[0], x[1], x[2], x[3]));
                    st_f4(g + i0 + 4, make_float4(x[4], x[5], x[6], x[7]));
                } else {
                    if constexpr (kMode == kModeAccAdd) {
                        const float4 o0 = ld_f4(acc_out + i0), o1 = ld_f4(acc_out + i0 + 4);
                        const float o[kVec] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
#pragma unroll
                        for (int e = 0; e < kVec; ++e) x[e] = __fadd_rn(o[e], x[e]);
                    }
                    st_f4(acc_out + i0, make_float4(x[0], x[1], x[2], x[3]));
                    st_f4(acc_out + i0 + 4, make_float4(x[4], x[5], x[6], x[7]));
                }
            }
        }
    }
    __syncthreads();                                            // every warp is out of its loop
    if (*abort) {
        // give the copies still in flight a bounded chance to land before the
        // block's shared memory goes away: the last job issued on each stage
        // (no later job was issued there, so its phase parity identifies it)
        if (producer && lane == 0) {
            for (int64_t k = issued > kS ? issued - kS : 0; k < issued; ++k)
                mbar_wait_bounded(full0 + 8u * (uint32_t)(k % kS), (uint32_t)((k / kS) & 1));
        }
        if (threadIdx.x == 0) atomicExch(a.err, 1);
        of = 1;
        __syncthreads();
    }

    // ragged tail (elements past the last full tile) and padding, as in reduce_kernel
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = n_tiles * kStageTile + tid; i < valid; i += nthreads) {
        float y = 0.0f;
        for (int c = 0; c < N; ++c) y = __fadd_rn(y, elem_to_f32<kIn>(base + (int64_t)c * ld + i));
        y = finish(y);
        if constexpr (kNorm) {
            y = divide(y, ds);
            of |= !isfinite(y);
            na.add_exact(y);
            g[i] = y;
        }
        if constexpr (kMode == kModeAccFirst) acc_out[i] = y;
        if constexpr (kMode == kModeAccAdd) acc_out[i] = __fadd_rn(acc_out[i], y);
    }
    for (int64_t i = valid + tid; i < S; i += nthreads) {
        if constexpr (kMode == kModeStep) g[i] = 0.0f;
        if constexpr (kMode == kModeAccFirst) acc_out[i] = 0.0f;
        if constexpr (kMode == kModeAccAdd) acc_out[i] = __fadd_rn(acc_out[i], 0.0f);
    }
    if constexpr (kNorm) {
        const int64_t pidx = a.part_base + (int64_t)j * gridDim.x + blockIdx.x;
        block_partial(na.total(), of, a.part_ss + pidx, a.part_of + pidx);
        if (a.fuse_finalize) count_and_finalize(a);
    }
}

// ------------------------------------------------------------------ K2
__global__ void __launch_bounds__(kFinalizeThreads) finalize_kernel(const __grid_constant__ FinalizeArgs a) {
    finalize_block(a);
}

// ------------------------------------------------------------------ K3
struct AdamConst {
    float b1, b2, omb1, omb2, lr, eps, decay, coef, bc1, bc2;
};

// a / b, correctly rounded, given y = RN(1/b) (the int8 quantizer divides a
// block's values by its scale), by Markstein's correction
// (P. Markstein, IBM J. Res. Dev. 34(1), 1990): when q is a faithful
// approximation of a/b and y approximates 1/b within a relative 2^-24, the
// remainder r = a - q*b is exact in one fma and RN(q + r*y) = RN(a/b).
// q0 = RN(a*y) can be up to ~1.5 ulp off (not always faithful), so one
// correction brings q1 within ~2e-7 ulp of a/b (faithful) and a second one
// gives the IEEE quotient.  Taken while a, the quotient and the remainders
// stay normal (2^-100 <= |a| <= 2^100, b and y in [2^-100, 2^100]);
// otherwise IEEE division.
__device__ __forceinline__ float div_known_recip(float a, float b, float y) {
    const float aa = fabsf(a);
    if (aa >= 0x1p-100f && aa <= 0x1p100f) {
        const float q0 = __fmul_rn(a, y);
        const float q1 = __fmaf_rn(__fmaf_rn(-q0, b, a), y, q0);
        return __fmaf_rn(__fmaf_rn(-q1, b, a), y, q1);
    }
    return __fdiv_rn(a, b);
}

// One element, in the order of the equations: clip, moments, bias
// correction, decoupled decay, Adam step (lr*mh)/(sqrt(vh)+eps).
__device__ __forceinline__ void adam_elem(float g, float &th, float &m, float &v,
                                          const AdamConst &k) {
    const float gc = __fmul_rn(g, k.coef);
    m = __fadd_rn(__fmul_rn(k.b1, m), __fmul_rn(k.omb1, gc));
    v = __fadd_rn(__fmul_rn(k.b2, v), __fmul_rn(k.omb2, __fmul_rn(gc, gc)));
    const float mh = __fdiv_rn(m, k.bc1);
    const float vh = __fdiv_rn(v, k.bc2);
    th = __fmul_rn(th, k.decay);
    th = __fsub_rn(th, __fdiv_rn(__fmul_rn(k.lr, mh), __fadd_rn(__fsqrt_rn(vh), k.eps)));
}

// One full warp stores its 32 x 16 consecutive output bytes (lane L's at
// o + 16 L, o = this lane's address) where o is 2-byte but not 16-byte
// aligned.  delta = o mod 16 is the same for every lane, and the aligned
// 16-byte word that starts delta bytes before lane L's span holds lane L-1's
// last delta bytes and lane L's first 16 - delta: lanes 1..31 write those
// words whole (one shuffle-up of the neighbour's data, four funnel shifts);
// lane 0 writes its first 16 - delta bytes and lane 31 its last delta bytes in
// 2-byte pieces.  Every lane of the warp must call this.
__device__ __forceinline__ void store_warp_realigned(uint16_t *o, const uint4 &w, int lane) {
    const uint32_t delta = (uint32_t)((uintptr_t)o & 15u);
    uint4 prev;
    prev.x = __shfl_up_sync(0xFFFFFFFFu, w.x, 1);
    prev.y = __shfl_up_sync(0xFFFFFFFFu, w.y, 1);
    prev.z = __shfl_up_sync(0xFFFFFFFFu, w.z, 1);
    prev.w = __shfl_up_sync(0xFFFFFFFFu, w.w, 1);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
    const int head = (int)(16u - delta) / 2;            // this lane's halves in the next word
    if (lane > 0)
        *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(o) - delta) =
            bytes_at(prev, w, 16u - delta);
    if (lane == 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e < head) o[e] = (uint16_t)(u[e >> 1] >> (16 * (e & 1)));
    }
    if (lane == 31) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e >= head) o[e] = (uint16_t)(u[e >> 1] >> (16 * (e & 1)));
    }
}

// kFromAcc: the gradient rows are micro-step accumulators that still carry
// the loss scale: g = acc / scale_used (the same division the reduce kernel
// applies), padding elements (flat index >= full_numel) are zero.
// kOneRate: every row of the launch has row 0's lr and decay (read as
// constant operands rather than per-row values held in registers).
template <bool kBf16, bool kFromAcc, bool kOneRate>
__global__ void __launch_bounds__(kBlock) adamw_kernel(const __grid_constant__ AdamArgs a) {
    const DevState *st = a.st;
    if (st->res.skipped) return;
    AdamConst k;
    k.b1 = a.b1; k.b2 = a.b2; k.omb1 = a.omb1; k.omb2 = a.omb2;
    const int j = blockIdx.y;
    k.lr = a.lr[kOneRate ? 0 : j]; k.eps = a.eps; k.decay = a.decay[kOneRate ? 0 : j];
    k.coef = st->res.clip_coef;
    k.bc1 = st->bc1;
    k.bc2 = st->bc2;

    float *th = a.master[j];
    float *mm = a.m[j];
    float *vv = a.v[j];
    const float *g = a.g[j];
    uint16_t *out = a.out[j];
    const int64_t S = a.S[j];
    const Divisor ds = make_divisor(kFromAcc ? st->res.scale_used : 1.0f);
    const int64_t valid = a.valid[j];
    auto grad = [&](float x, int64_t i) {
        if constexpr (kFromAcc) return i < valid ? divide(x, ds) : 0.0f;
        else return x;
    };
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    int64_t done = 0;
    if (a.vec[j]) {
        const int64_t nch = S / kVec;
        const int oal = a.out_align[j];
        for (int64_t ch = tid; ch < nch; ch += nthreads) {
            const int64_t i0 = ch * kVec;
            const float4 g0 = ld_nc_f4(g + i0), g1 = ld_nc_f4(g + i0 + 4);
            const float4 t0 = ld_f4(th + i0), t1 = ld_f4(th + i0 + 4);
            const float4 m0 = ld_f4(mm + i0), m1 = ld_f4(mm + i0 + 4);
            const float4 v0 = ld_f4(vv + i0), v1 = ld_f4(vv + i0 + 4);
            float G[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            float T[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
            float M[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
            float V[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) adam_elem(grad(G[e], i0 + e), T[e], M[e], V[e], k);
            st_f4(th + i0, make_float4(T[0], T[1], T[2], T[3]));
            st_f4(th + i0 + 4, make_float4(T[4], T[5], T[6], T[7]));
            st_f4(mm + i0, make_float4(M[0], M[1], M[2], M[3]));
            st_f4(mm + i0 + 4, make_float4(M[4], M[5], M[6], M[7]));
            st_f4(vv + i0, make_float4(V[0], V[1], V[2], V[3]));
            st_f4(vv + i0 + 4, make_float4(V[4], V[5], V[6], V[7]));
            const uint32_t w0 = pack2<kBf16>(T[0], T[1]), w1 = pack2<kBf16>(T[2], T[3]);
            const uint32_t w2 = pack2<kBf16>(T[4], T[5]), w3 = pack2<kBf16>(T[6], T[7]);
            uint16_t *o = out + i0;
            if (oal == 16) {
                *reinterpret_cast<uint4 *>(o) = make_uint4(w0, w1, w2, w3);
            } else if (ch - (threadIdx.x & 31) + 31 < nch) {   // a full warp: aligned stores
                store_warp_realigned(o, make_uint4(w0, w1, w2, w3), threadIdx.x & 31);
            } else if (oal == 4) {
                uint32_t *o32 = reinterpret_cast<uint32_t *>(o);
                o32[0] = w0; o32[1] = w1; o32[2] = w2; o32[3] = w3;
            } else {
                const uint32_t w[4] = {w0, w1, w2, w3};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    o[2 * e] = (uint16_t)(w[e] & 0xFFFFu);
                    o[2 * e + 1] = (uint16_t)(w[e] >> 16);
                }
            }
        }
        done = nch * kVec;
    }
    for (int64_t i = done + tid; i < S; i += nthreads) {   // ragged tail / unaligned shards
        float t = th[i], m = mm[i], v = vv[i];
        adam_elem(grad(g[i], i), t, m, v, k);
        th[i] = t;
        mm[i] = m;
        vv[i] = v;
        out[i] = from_f32<kBf16>(t);
    }
}

// ------------------------------------------------------------------ K3q
// AdamW + cast + the int8 all-gather payload (ZeRO++ quantized weights:
// "DeepSpeed 与 FSDP" §ZeRO++, ZeRO reading §4.2).  Each warp owns one
// kQ8Block-element block of the shard per iteration (lane L: elements
// 8L..8L+7), so the block's absmax is a warp reduction.  The quantized value
// is the 16-bit parameter as it would be gathered (decoded exactly to fp32):
// scale = amax / 127, q = clamp(rint(p / scale), -127, 127), NaN -> 0.
template <bool kBf16>
__device__ __forceinline__ float decode16(float x) {
    if constexpr (kBf16) return __bfloat162float(__float2bfloat16_rn(x));
    else return __half2float(__float2half_rn(x));
}

template <bool kBf16, bool kOneRate>
__global__ void __launch_bounds__(kBlock) adamw_q8_kernel(const __grid_constant__ AdamArgs a) {
    const DevState *st = a.st;
    if (st->res.skipped) return;
    AdamConst k;
    k.b1 = a.b1; k.b2 = a.b2; k.omb1 = a.omb1; k.omb2 = a.omb2;
    const int j = blockIdx.y;
    k.lr = a.lr[kOneRate ? 0 : j]; k.eps = a.eps; k.decay = a.decay[kOneRate ? 0 : j];
    k.coef = st->res.clip_coef;
    k.bc1 = st->bc1;
    k.bc2 = st->bc2;

    float *th = a.master[j];
    float *mm = a.m[j];
    float *vv = a.v[j];
    const float *g = a.g[j];
    uint16_t *out = a.out[j];
    int8_t *q8 = a.q8[j];
    float *scales = a.q8_scales[j];
    const int64_t S = a.S[j];
    const bool vec = a.vec[j] != 0;
    const int oal = a.out_align[j];
    const bool q8vec = a.q8_align[j] == 8;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t nblk = (S + kQ8Block - 1) / kQ8Block;

    for (int64_t b = warp; b < nblk; b += n_warps) {          // warp-uniform
        const int64_t i0 = b * kQ8Block + (int64_t)lane * kVec;
        const int64_t rem = S - i0;
        const int cnt = rem <= 0 ? 0 : (rem >= kVec ? kVec : (int)rem);
        const bool full_block = (b + 1) * kQ8Block <= S;          // warp-uniform
        float P[kVec];
        if (cnt == kVec && vec) {
            const float4 g0 = ld_nc_f4(g + i0), g1 = ld_nc_f4(g + i0 + 4);
            const float4 t0 = ld_f4(th + i0), t1 = ld_f4(th + i0 + 4);
            const float4 m0 = ld_f4(mm + i0), m1 = ld_f4(mm + i0 + 4);
            const float4 v0 = ld_f4(vv + i0), v1 = ld_f4(vv + i0 + 4);
            float G[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            float T[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
            float M[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
            float V[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) adam_elem(G[e], T[e], M[e], V[e], k);
            st_f4(th + i0, make_float4(T[0], T[1], T[2], T[3]));
            st_f4(th + i0 + 4, make_float4(T[4], T[5], T[6], T[7]));
            st_f4(mm + i0, make_float4(M[0], M[1], M[2], M[3]));
            st_f4(mm + i0 + 4, make_float4(M[4], M[5], M[6], M[7]));
            st_f4(vv + i0, make_float4(V[0], V[1], V[2], V[3]));
            st_f4(vv + i0 + 4, make_float4(V[4], V[5], V[6], V[7]));
            if (out) {
                const uint32_t w0 = pack2<kBf16>(T[0], T[1]), w1 = pack2<kBf16>(T[2], T[3]);
                const uint32_t w2 = pack2<kBf16>(T[4], T[5]), w3 = pack2<kBf16>(T[6], T[7]);
                uint16_t *o = out + i0;
                if (oal == 16) {
                    *reinterpret_cast<uint4 *>(o) = make_uint4(w0, w1, w2, w3);
                } else if (full_block) {                       // every lane is here
                    store_warp_realigned(o, make_uint4(w0, w1, w2, w3), lane);
                } else if (oal == 4) {
                    uint32_t *o32 = reinterpret_cast<uint32_t *>(o);
                    o32[0] = w0; o32[1] = w1; o32[2] = w2; o32[3] = w3;
                } else {
                    const uint32_t w[4] = {w0, w1, w2, w3};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        o[2 * e] = (uint16_t)(w[e] & 0xFFFFu);
                        o[2 * e + 1] = (uint16_t)(w[e] >> 16);
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < kVec; ++e) P[e] = decode16<kBf16>(T[e]);
        } else {
#pragma unroll
            for (int e = 0; e < kVec; ++e) {
                P[e] = 0.0f;
                if (e < cnt) {
                    const int64_t i = i0 + e;
                    float t = th[i], m = mm[i], v = vv[i];
                    adam_elem(g[i], t, m, v, k);
                    th[i] = t;
                    mm[i] = m;
                    vv[i] = v;
                    if (out) out[i] = from_f32<kBf16>(t);
                    P[e] = decode16<kBf16>(t);
                }
            }
        }
        float amax = 0.0f;                                     // NaN ignored (fmaxf)
#pragma unroll
        for (int e = 0; e < kVec; ++e) amax = fmaxf(amax, fabsf(P[e]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const float scale = __fdiv_rn(amax, 127.0f);
        // p / scale, correctly rounded: Markstein's correction from
        // y = RN(1/scale) (div_known_recip) while scale, 1/scale and the
        // quotients stay normal; IEEE division otherwise.
        const bool fast = scale >= 0x1p-100f && scale <= 0x1p100f;
        const float y = fast ? __frcp_rn(scale) : 0.0f;
        int8_t q[kVec];
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            int code = 0;
            if (scale != 0.0f) {
                const float pe = P[e];
                const float v = fast ? div_known_recip(pe, scale, y) : __fdiv_rn(pe, scale);
                if (!isnan(v)) {
                    code = __float2int_rn(v);                  // half to even; saturates
                    code = code > 127 ? 127 : (code < -127 ? -127 : code);
                }
            }
            q[e] = (int8_t)code;
        }
        if (cnt == kVec && q8vec) {
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                lo |= (uint32_t)(uint8_t)q[e] << (8 * e);
                hi |= (uint32_t)(uint8_t)q[e + 4] << (8 * e);
            }
            *reinterpret_cast<uint2 *>(q8 + i0) = make_uint2(lo, hi);
        } else {
#pragma unroll
            for (int e = 0; e < kVec; ++e)
                if (e < cnt) q8[i0 + e] = q[e];
        }
        if (lane == 0) scales[b] = scale;
    }
}

}  // namespace

template <int kIn, int kMode>
static cudaError_t launch_staged(const ReduceArgs &a, dim3 grid, cudaStream_t s) {
    constexpr int kSmem = StageTraits<kIn>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(reduce_staged_kernel<kIn, kMode>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    reduce_staged_kernel<kIn, kMode><<<grid, kStagedThreads, kSmem, s>>>(a);
    return cudaGetLastError();
}

template <int kIn, bool kOneShape>
static cudaError_t launch_plain(const ReduceArgs &a, dim3 grid, int mode, cudaStream_t s) {
    switch (mode) {
        case kModeStep: reduce_kernel<kIn, kModeStep, kOneShape><<<grid, kBlock, 0, s>>>(a); break;
        case kModeAccFirst: reduce_kernel<kIn, kModeAccFirst, kOneShape><<<grid, kBlock, 0, s>>>(a); break;
        case kModeAccAdd: reduce_kernel<kIn, kModeAccAdd, kOneShape><<<grid, kBlock, 0, s>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <int kIn>
static cudaError_t launch_reduce_in(const ReduceArgs &a, dim3 grid, int mode, bool staged,
                                    cudaStream_t s) {
    if (staged) {
        switch (mode) {
            case kModeStep: return launch_staged<kIn, kModeStep>(a, grid, s);
            case kModeAccFirst: return launch_staged<kIn, kModeAccFirst>(a, grid, s);
            case kModeAccAdd: return launch_staged<kIn, kModeAccAdd>(a, grid, s);
            default: return cudaErrorInvalidValue;
        }
    }
    bool one_shape = true;
    for (int32_t j = 1; j < a.n_ranks; ++j)
        one_shape = one_shape && a.ld[j] == a.ld[0] && a.S[j] == a.S[0] &&
                    (mode != kModeStep || a.g[j] == a.g[0] + (int64_t)j * a.g_stride);
    if (a.full_numel < 0) one_shape = false;      // rows of several FlatParameters
    return one_shape ? launch_plain<kIn, true>(a, grid, mode, s)
                     : launch_plain<kIn, false>(a, grid, mode, s);
}

cudaError_t launch_reduce(const ReduceArgs &a, int grid_x, int in_kind, int mode, bool staged,
                          cudaStream_t s) {
    const dim3 grid((unsigned)grid_x, (unsigned)a.n_ranks);
    if (mode == kModeNormOnly) {
        if (staged) return cudaErrorInvalidValue;
        if (a.full_numel >= 0)                    // the rows of one FlatParameter
            reduce_kernel<kInF32, kModeNormOnly, true><<<grid, kBlock, 0, s>>>(a);
        else
            reduce_kernel<kInF32, kModeNormOnly, false><<<grid, kBlock, 0, s>>>(a);
        return cudaGetLastError();
    }
    switch (in_kind) {
        case kInF16: return launch_reduce_in<kInF16>(a, grid, mode, staged, s);
        case kInBF16: return launch_reduce_in<kInBF16>(a, grid, mode, staged, s);
        case kInF32: return launch_reduce_in<kInF32>(a, grid, mode, staged, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_finalize(const FinalizeArgs &a, cudaStream_t s) {
    finalize_kernel<<<1, kFinalizeThreads, 0, s>>>(a);
    return cudaGetLastError();
}

static bool one_rate(const AdamArgs &a) {
    for (int32_t j = 1; j < a.n_ranks; ++j)
        if (a.lr[j] != a.lr[0] || a.decay[j] != a.decay[0]) return false;
    return true;
}

template <bool kOneRate>
static void launch_adamw_rate(const AdamArgs &a, dim3 grid, bool bf16_out, bool from_acc,
                              cudaStream_t s) {
    if (from_acc) {
        if (bf16_out) adamw_kernel<true, true, kOneRate><<<grid, kBlock, 0, s>>>(a);
        else adamw_kernel<false, true, kOneRate><<<grid, kBlock, 0, s>>>(a);
    } else {
        if (bf16_out) adamw_kernel<true, false, kOneRate><<<grid, kBlock, 0, s>>>(a);
        else adamw_kernel<false, false, kOneRate><<<grid, kBlock, 0, s>>>(a);
    }
}

cudaError_t launch_adamw(const AdamArgs &a, int grid_x, bool bf16_out, bool from_acc,
                         cudaStream_t s) {
    const dim3 grid((unsigned)grid_x, (unsigned)a.n_ranks);
    if (one_rate(a)) launch_adamw_rate<true>(a, grid, bf16_out, from_acc, s);
    else launch_adamw_rate<false>(a, grid, bf16_out, from_acc, s);
    return cudaGetLastError();
}

cudaError_t launch_adamw_q8(const AdamArgs &a, int grid_x, bool bf16_out, cudaStream_t s) {
    const dim3 grid((unsigned)grid_x, (unsigned)a.n_ranks);
    const bool one = one_rate(a);
    if (bf16_out) {
        if (one) adamw_q8_kernel<true, true><<<grid, kBlock, 0, s>>>(a);
        else adamw_q8_kernel<true, false><<<grid, kBlock, 0, s>>>(a);
    } else {
        if (one) adamw_q8_kernel<false, true><<<grid, kBlock, 0, s>>>(a);
        else adamw_q8_kernel<false, false><<<grid, kBlock, 0, s>>>(a);
    }
    return cudaGetLastError();
}

template <int kIn, int kMode>
static cudaError_t occ(bool staged, int *bps) {
    if (!staged)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(bps, reduce_kernel<kIn, kMode>, kBlock, 0);
    if constexpr (kMode == kModeNormOnly) {
        return cudaErrorInvalidValue;
    } else {
        constexpr int kSmem = StageTraits<kIn>::kSmem;
        cudaError_t e = cudaFuncSetAttribute(reduce_staged_kernel<kIn, kMode>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(bps, reduce_staged_kernel<kIn, kMode>,
                                                             kStagedThreads, kSmem);
    }
}

cudaError_t reduce_blocks_per_sm(int in_kind, int mode, bool staged, int *bps) {
    cudaError_t e = cudaErrorInvalidValue;
    *bps = 1;
    if (mode == kModeNormOnly) {
        e = occ<kInF32, kModeNormOnly>(staged, bps);
    } else {
#define ZG_OCC(K)                                                            \
        switch (mode) {                                                      \
            case kModeStep: e = occ<K, kModeStep>(staged, bps); break;       \
            case kModeAccFirst: e = occ<K, kModeAccFirst>(staged, bps); break; \
            case kModeAccAdd: e = occ<K, kModeAccAdd>(staged, bps); break;   \
        }
        if (in_kind == kInF16) { ZG_OCC(kInF16) }
        else if (in_kind == kInBF16) { ZG_OCC(kInBF16) }
        else if (in_kind == kInF32) { ZG_OCC(kInF32) }
#undef ZG_OCC
    }
    if (*bps < 1) *bps = 1;
    return e;
}

}  // namespace zg
