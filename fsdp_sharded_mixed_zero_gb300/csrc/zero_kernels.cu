// zero_kernels.cu -- the three kernels of one ZeRO shard step on sm_103a.
//
//   K1 reduce_kernel    N-way reduce of the 16-bit gradient contributions of
//                       each stepped shard, AVG, loss-scale division, inf/NaN
//                       check and per-block partial sums of squares; writes
//                       the fp32 reduced gradient row (the reduce half of a
//                       reduce-scatter: "PyTorch FSDP ... 深度解析" §3.3;
//                       sum-then-split in the numpy demo of "DeepSpeed 与
//                       FSDP"; fp32 reduce per its MixedPrecision example).
//   K2 finalize_kernel  one block: fixed-order total of the partials, global
//                       norm, clip coefficient, overflow skip and the dynamic
//                       loss-scale state machine (ZeRO reading §5.1, §5.3).
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
// exact square of x is p + e with p = x*x and e = fma(x, x, -p) (exact), and
// Knuth's TwoSum gives the exact error of every addition.  Only the small
// correction term `lo` is rounded (relative error ~ eps^2), and the chunk's
// hi + lo enters the thread's fp64 sum once.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &err) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ double chunk_sum_of_squares(const float x[kVec]) {
    float hi = __fmul_rn(x[0], x[0]);
    float lo = __fmaf_rn(x[0], x[0], -hi);
#pragma unroll
    for (int k = 1; k < kVec; ++k) {
        const float p = __fmul_rn(x[k], x[k]);
        const float e = __fmaf_rn(x[k], x[k], -p);
        float t;
        two_sum(hi, p, hi, t);
        lo = __fadd_rn(lo, __fadd_rn(t, e));
    }
    return (double)hi + (double)lo;
}

// ------------------------------------------------------------------ reduction
// Block total of per-thread fp64 sums and flags, in a fixed order.
__device__ __forceinline__ void block_partial(double ss, int of, double *out_ss,
                                              int32_t *out_of) {
    __shared__ double warp_ss[kBlock / 32];
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

// ------------------------------------------------------------------ K1
template <bool kBf16>
__global__ void __launch_bounds__(kBlock, 5) reduce_kernel(const __grid_constant__ ReduceArgs a) {
    const int j = blockIdx.y;
    const int64_t S = a.S;
    int64_t valid = a.full_numel - a.first[j];   // elements [valid, S) are padding
    valid = valid < 0 ? 0 : (valid > S ? S : valid);
    const uint16_t *base = a.grads + a.goff[j];
    float *g = a.g + (int64_t)j * a.g_stride;
    const int N = a.n_contrib;
    const int64_t ld = a.ld;
    const bool avg = a.avg != 0;
    const Divisor dn = make_divisor((float)N);
    const Divisor ds = make_divisor(a.st->scaler.scale);

    double ss = 0.0;
    int of = 0;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    int64_t done = 0;
    if (a.vec[j]) {
        const int64_t nch = valid / kVec;
        for (int64_t ch = tid; ch < nch; ch += nthreads) {
            const int64_t i0 = ch * kVec;
            const uint16_t *p = base + i0;
            float acc[kVec];
#pragma unroll
            for (int e = 0; e < kVec; ++e) acc[e] = 0.0f;
            int c = 0;
            for (; c + 8 <= N; c += 8) {          // eight rows in flight
                uint4 w[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) w[k] = ld_nc_u4(p + (int64_t)(c + k) * ld);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float f[kVec];
                    unpack8<kBf16>(w[k], f);
#pragma unroll
                    for (int e = 0; e < kVec; ++e) acc[e] = __fadd_rn(acc[e], f[e]);
                }
            }
            for (; c < N; ++c) {
                const uint4 w = ld_nc_u4(p + (int64_t)c * ld);
                float f[kVec];
                unpack8<kBf16>(w, f);
#pragma unroll
                for (int e = 0; e < kVec; ++e) acc[e] = __fadd_rn(acc[e], f[e]);
            }
#pragma unroll
            for (int e = 0; e < kVec; ++e) {
                float x = acc[e];
                if (avg) x = divide(x, dn);
                x = divide(x, ds);
                acc[e] = x;
                of |= !isfinite(x);
            }
            ss += chunk_sum_of_squares(acc);
            st_f4(g + i0, make_float4(acc[0], acc[1], acc[2], acc[3]));
            st_f4(g + i0 + 4, make_float4(acc[4], acc[5], acc[6], acc[7]));
        }
        done = nch * kVec;
    }
    for (int64_t i = done + tid; i < valid; i += nthreads) {   // ragged tail / unaligned rows
        float acc = 0.0f;
        for (int c = 0; c < N; ++c) acc = __fadd_rn(acc, to_f32<kBf16>(base[(int64_t)c * ld + i]));
        if (avg) acc = divide(acc, dn);
        acc = divide(acc, ds);
        of |= !isfinite(acc);
        ss += (double)acc * (double)acc;          // exact square in fp64
        g[i] = acc;
    }
    for (int64_t i = valid + tid; i < S; i += nthreads) g[i] = 0.0f;   // padding

    const int64_t pidx = a.part_base + (int64_t)j * gridDim.x + blockIdx.x;
    block_partial(ss, of, a.part_ss + pidx, a.part_of + pidx);
}

// ------------------------------------------------------------------ K2
__global__ void __launch_bounds__(kFinalizeThreads) finalize_kernel(const __grid_constant__ FinalizeArgs a) {
    __shared__ double warp_ss[kFinalizeThreads / 32];
    double s = 0.0;
    int of = 0;
    for (int i = threadIdx.x; i < a.n_parts; i += blockDim.x) {
        s += a.part_ss[i];
        of |= a.part_of[i];
    }
    of = __syncthreads_or(of);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xFFFFFFFFu, s, o);
    if ((threadIdx.x & 31) == 0) warp_ss[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x != 0) return;
    double total = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) total += warp_ss[w];

    DevState *st = a.st;
    ScalerDev sc = st->scaler;
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
        const float2 bc = sc.step_t < a.bc_len ? a.bc_table[sc.step_t] : make_float2(1.0f, 1.0f);
        st->bc1 = bc.x;
        st->bc2 = bc.y;
    }
    st->scaler = sc;
    st->res = r;
}

// ------------------------------------------------------------------ K3
struct AdamConst {
    float b1, b2, omb1, omb2, lr, eps, decay, coef, bc1, bc2;
};

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

template <bool kBf16>
__global__ void __launch_bounds__(kBlock) adamw_kernel(const __grid_constant__ AdamArgs a) {
    const DevState *st = a.st;
    if (st->res.skipped) return;
    AdamConst k;
    k.b1 = a.b1; k.b2 = a.b2; k.omb1 = a.omb1; k.omb2 = a.omb2;
    k.lr = a.lr; k.eps = a.eps; k.decay = a.decay;
    k.coef = st->res.clip_coef;
    k.bc1 = st->bc1;
    k.bc2 = st->bc2;

    const int j = blockIdx.y;
    float *th = a.master[j];
    float *mm = a.m[j];
    float *vv = a.v[j];
    const float *g = a.g + (int64_t)j * a.g_stride;
    uint16_t *out = reinterpret_cast<uint16_t *>(a.out) + a.out_off[j];
    const int64_t S = a.S;
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
            for (int e = 0; e < 8; ++e) adam_elem(G[e], T[e], M[e], V[e], k);
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
        adam_elem(g[i], t, m, v, k);
        th[i] = t;
        mm[i] = m;
        vv[i] = v;
        out[i] = from_f32<kBf16>(t);
    }
}

}  // namespace

cudaError_t launch_reduce(const ReduceArgs &a, int grid_x, bool bf16, cudaStream_t s) {
    const dim3 grid((unsigned)grid_x, (unsigned)a.n_ranks);
    if (bf16) reduce_kernel<true><<<grid, kBlock, 0, s>>>(a);
    else reduce_kernel<false><<<grid, kBlock, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_finalize(const FinalizeArgs &a, cudaStream_t s) {
    finalize_kernel<<<1, kFinalizeThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_adamw(const AdamArgs &a, int grid_x, bool bf16_out, cudaStream_t s) {
    const dim3 grid((unsigned)grid_x, (unsigned)a.n_ranks);
    if (bf16_out) adamw_kernel<true><<<grid, kBlock, 0, s>>>(a);
    else adamw_kernel<false><<<grid, kBlock, 0, s>>>(a);
    return cudaGetLastError();
}


cudaError_t reduce_blocks_per_sm(int *bps) {
    int r0 = 0, r1 = 0;
    cudaError_t e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r0, reduce_kernel<false>, kBlock, 0))) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r1, reduce_kernel<true>, kBlock, 0))) return e;
    *bps = r0 < r1 ? r0 : r1;
    if (*bps < 1) *bps = 1;
    return cudaSuccess;
}

}  // namespace zg
