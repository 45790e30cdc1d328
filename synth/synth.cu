// synth.cu -- seeded synthetic inputs for the ZeRO shard step, generated on
// the GPU (and, for host-side samples of the same workload, on host threads).
//
// This module holds none of the optimizer's arithmetic.  It draws:
//   * fp32 tensors ~ N(0, sigma) (optionally |N|) for master weights and
//     warm Adam moments;
//   * the N per-rank gradient contributions of a data-parallel step, each
//     element  grad[c][i] = cast16((g_i + n_{c,i}) * scale)  with a gradient
//     g ~ N(0, sigma_g) shared by every rank and per-rank noise
//     n_c ~ N(0, sigma_n), cast to fp16 (or bf16) by the platform's own
//     round-to-nearest conversion (CUDA cvt on the GPU, the compiler's
//     _Float16 conversion on the host; bf16 on the host is left to the caller
//     as fp32 values).
//
// Random bits: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11), counter = (element index lo, hi, 0, 0),
// key = (seed, stream id).  Every element is one Philox block, so any element
// can be regenerated on its own.
//
// Normal variates: Box-Muller (G. E. P. Box and M. E. Muller, "A Note on the
// Generation of Random Normal Deviates", Ann. Math. Statist. 29(2), 1958).
// Two words of the element's block give u1 = ((w0 >> 8) + 1) / 2^24 in
// (0, 1] and u2 = (w1 >> 8) / 2^24 in [0, 1), both exact in fp32, and
// z = sqrt(-2 ln u1) cos(2 pi u2) is N(0, 1) (|z| <= sqrt(2 ln 2^24) = 5.77).
// The logarithm, square root and cosine are the platform's own library
// functions (CUDA's logf, sqrtf and cospif on the GPU; the C library's on the
// host), so host and device values agree to a few ulp but not bit for bit;
// tests that compare the GPU with the oracle hand the oracle the GPU's bytes.
#include <cstdint>
#include <cstring>
#include <cmath>
#include <thread>
#include <vector>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#define SYNTH_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;   // golden ratio
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;   // sqrt(3) - 1

__host__ __device__ inline void mulhilo32(uint32_t a, uint32_t b, uint32_t &hi, uint32_t &lo) {
    const uint64_t p = (uint64_t)a * (uint64_t)b;
    hi = (uint32_t)(p >> 32);
    lo = (uint32_t)p;
}

// Ten rounds; the key is bumped by the Weyl constants between rounds.
__host__ __device__ inline void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round) { k0 += kPhiloxW0; k1 += kPhiloxW1; }
        uint32_t hi0, lo0, hi1, lo1;
        mulhilo32(kPhiloxM0, c[0], hi0, lo0);
        mulhilo32(kPhiloxM1, c[2], hi1, lo1);
        const uint32_t n0 = hi1 ^ c[1] ^ k0;
        const uint32_t n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
    }
}

__host__ __device__ inline float normal_at(uint32_t seed, uint32_t stream, uint64_t idx,
                                           double sigma) {
    uint32_t c[4] = {(uint32_t)idx, (uint32_t)(idx >> 32), 0u, 0u};
    philox4x32_10(c, seed, stream);
    const float u1 = (float)((c[0] >> 8) + 1u) * 0x1p-24f;
    const float u2 = (float)(c[1] >> 8) * 0x1p-24f;
#ifdef __CUDA_ARCH__
    const float r = sqrtf(__fmul_rn(-2.0f, logf(u1)));
    const float z = __fmul_rn(r, cospif(__fmul_rn(2.0f, u2)));
    return (float)__dmul_rn((double)z, sigma);
#else
    const float r = std::sqrt(-2.0f * std::log(u1));
    const float z = r * (float)std::cos(6.283185307179586 * (double)u2);
    return (float)((double)z * sigma);
#endif
}

// Stream ids: tensor kind in the top byte, step and contributor below.
enum : uint32_t { kMaster = 1, kMomentM = 2, kMomentV = 3, kGradShared = 4, kGradNoise = 5 };

__host__ __device__ inline uint32_t stream_id(uint32_t kind, uint32_t step, uint32_t contrib) {
    return (kind << 24) | ((step & 0xFFFu) << 12) | (contrib & 0xFFFu);
}

// Pre-cast gradient value of contributor c at flat index idx.
__host__ __device__ inline float grad_value(uint32_t seed, uint32_t step, uint32_t c,
                                            uint64_t idx, double sg, double sn, float scale) {
    const float g = normal_at(seed, stream_id(kGradShared, step, 0), idx, sg);
    const float n = normal_at(seed, stream_id(kGradNoise, step, c), idx, sn);
#ifdef __CUDA_ARCH__
    return __fmul_rn(__fadd_rn(g, n), scale);
#else
    return (g + n) * scale;                             // add, then multiply
#endif
}

// ---------------------------------------------------------------- device
__global__ void k_normal_f32(uint32_t seed, uint32_t stream, uint64_t first, int64_t n,
                             double sigma, int absval, float *out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        float x = normal_at(seed, stream, first + (uint64_t)i, sigma);
        out[i] = absval ? fabsf(x) : x;
    }
}

// dtype: 0 fp16, 1 bf16, 2 fp32 (the pre-cast value itself).
__global__ void k_grads(uint32_t seed, uint32_t step, int32_t c0, int32_t nc, double sg,
                        double sn, float scale, int dtype, uint64_t first, int64_t n,
                        uint64_t zero_from, void *out, int64_t ld) {
    const int64_t total = n * (int64_t)nc;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t c = e / n, i = e - c * n;
        const uint64_t idx = first + (uint64_t)i;
        float x = 0.0f;
        if (idx < zero_from) x = grad_value(seed, step, (uint32_t)(c0 + c), idx, sg, sn, scale);
        if (dtype == 2) {
            static_cast<float *>(out)[c * ld + i] = x;
            continue;
        }
        uint16_t h;
        if (dtype == 1) {
            __nv_bfloat16 b = __float2bfloat16_rn(x);
            memcpy(&h, &b, 2);
        } else {
            __half b = __float2half_rn(x);
            memcpy(&h, &b, 2);
        }
        static_cast<uint16_t *>(out)[c * ld + i] = h;
    }
}

inline int grid_for(int64_t n) {
    int64_t b = (n + 255) / 256;
    if (b > 152 * 32) b = 152 * 32;
    return (int)(b < 1 ? 1 : b);
}

// ---------------------------------------------------------------- host
template <class F>
void parallel_for(int64_t n, int threads, F f) {
    if (threads < 1) threads = 1;
    if (n < 65536 || threads == 1) { f(0, n); return; }
    std::vector<std::thread> pool;
    const int64_t per = (n + threads - 1) / threads;
    for (int t = 0; t < threads; ++t) {
        const int64_t a = t * per, b = a + per < n ? a + per : n;
        if (a >= b) break;
        pool.emplace_back([=] { f(a, b); });
    }
    for (auto &th : pool) th.join();
}

}  // namespace

// Raw Philox block, for known-answer tests.
SYNTH_API void synth_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    philox4x32_10(c, key[0], key[1]);
    memcpy(out, c, sizeof(c));
}

SYNTH_API uint32_t synth_stream_id(uint32_t kind, uint32_t step, uint32_t contrib) {
    return stream_id(kind, step, contrib);
}

// out[i] = N(0, sigma) (|.| if absval) at flat index first + i, i < n.
SYNTH_API int synth_normal_f32_host(uint32_t seed, uint32_t stream, uint64_t first, int64_t n,
                                    double sigma, int absval, float *out, int threads) {
    if (n < 0 || (n && !out)) return 1;
    parallel_for(n, threads, [&](int64_t a, int64_t b) {
        for (int64_t i = a; i < b; ++i) {
            float x = normal_at(seed, stream, first + (uint64_t)i, sigma);
            out[i] = absval ? std::fabs(x) : x;
        }
    });
    return 0;
}

// Gradient contributions c0 .. c0+nc-1 at flat indices first .. first+n-1.
// kind 0: fp16 encodings (uint16) via _Float16; kind 2: fp32 pre-cast values
// (the caller casts to bf16).  Row stride ld (elements).  Flat indices at or
// beyond zero_from give 0.
SYNTH_API int synth_grads_host(uint32_t seed, uint32_t step, int32_t c0, int32_t nc,
                               double sg, double sn, float scale, int kind, uint64_t first,
                               int64_t n, uint64_t zero_from, void *out, int64_t ld,
                               int threads) {
    if (n < 0 || nc < 0 || (n && nc && !out) || ld < n || (kind != 0 && kind != 2)) return 1;
    parallel_for(n, threads, [&](int64_t a, int64_t b) {
        for (int32_t c = 0; c < nc; ++c) {
            for (int64_t i = a; i < b; ++i) {
                const uint64_t idx = first + (uint64_t)i;
                float x = 0.0f;
                if (idx < zero_from) x = grad_value(seed, step, (uint32_t)(c0 + c), idx, sg, sn, scale);
                if (kind == 0) {
                    _Float16 h = (_Float16)x;
                    memcpy((uint16_t *)out + c * ld + i, &h, 2);
                } else {
                    ((float *)out)[c * ld + i] = x;
                }
            }
        }
    });
    return 0;
}

SYNTH_API int synth_normal_f32_device(uint32_t seed, uint32_t stream, uint64_t first, int64_t n,
                                      double sigma, int absval, float *out, void *cuda_stream) {
    if (n < 0 || (n && !out)) return 1;
    if (n == 0) return 0;
    k_normal_f32<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(seed, stream, first, n,
                                                                     sigma, absval, out);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

// dtype 0 = fp16, 1 = bf16 (out: uint16), 2 = fp32 (out: float); [nc rows, stride ld].
SYNTH_API int synth_grads_device(uint32_t seed, uint32_t step, int32_t c0, int32_t nc,
                                 double sg, double sn, float scale, int dtype, uint64_t first,
                                 int64_t n, uint64_t zero_from, void *out, int64_t ld,
                                 void *cuda_stream) {
    if (n < 0 || nc < 0 || (n && nc && !out) || ld < n || dtype < 0 || dtype > 2) return 1;
    if (n == 0 || nc == 0) return 0;
    k_grads<<<grid_for(n * (int64_t)nc), 256, 0, (cudaStream_t)cuda_stream>>>(
        seed, step, c0, nc, sg, sn, scale, dtype, first, n, zero_from, out, ld);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}
