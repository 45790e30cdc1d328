// host_adam.cc -- AdamW + 16-bit cast on the host CPU cores for the
// ZeRO-Offload shard step ("DeepSpeed 与 FSDP" §ZeRO-Offload; "ZeRO: Memory
// Optimizations Toward Training Trillion Parameter Models" §4.1 keeps the
// optimizer states in CPU memory), and the thread pool that runs it.
//
// Built with -ffp-contract=off and without fast-math: each expression below
// is one IEEE fp32 operation, evaluated in fp32, in the order of the update's
// equations.  -fno-math-errno only lets sqrt compile to the vector square
// root instruction (IEEE, correctly rounded).
#include "host_adam.h"
#include "zero.h"

#include <sched.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <memory>

void zero_internal_set_error(const char *msg);

namespace zh {
namespace {

inline uint16_t f16_rne(float f) {
    uint32_t x;
    std::memcpy(&x, &f, 4);
    const uint32_t sign = (x >> 16) & 0x8000u;
    const uint32_t a = x & 0x7FFFFFFFu;
    // half normals (|f| in [2^-14, 65520)): move the exponent bias from 127 to
    // 15 (subtract 112 << 23) and round the 23-bit mantissa at bit 13, ties to
    // the even neighbour (the +1 when bit 13 is set); a carry out of the
    // mantissa lands correctly in the exponent.
    const uint32_t normal = (a - 0x38000000u + 0x0FFFu + ((a >> 13) & 1u)) >> 13;
    // half subnormals (|f| < 2^-14): in [0.5, 1) fp32 spacing is 2^-24, the
    // half subnormal step, so the fp32 sum |f| + 0.5 is |f| rounded (to
    // nearest even) onto that grid; its mantissa bits are the half code.
    float af;
    std::memcpy(&af, &a, 4);
    const float t = af + 0.5f;
    uint32_t tb;
    std::memcpy(&tb, &t, 4);
    const uint32_t sub = tb - 0x3F000000u;
    // select with all-ones / all-zeros masks (branch-free, so it vectorises)
    const uint32_t is_sub = 0u - (uint32_t)(a < 0x38800000u);
    const uint32_t is_inf = 0u - (uint32_t)(a >= 0x477FF000u);   // 65520 and above, inf
    const uint32_t is_nan = 0u - (uint32_t)(a > 0x7F800000u);    // -> quiet NaN
    uint32_t r = (sub & is_sub) | (normal & ~is_sub);
    r = (0x7C00u & is_inf) | (r & ~is_inf);
    r = (0x7E00u & is_nan) | (r & ~is_nan);
    return (uint16_t)(sign | r);
}

inline uint16_t bf16_rne(float f) {
    uint32_t x;
    std::memcpy(&x, &f, 4);
    // drop the low 16 bits, rounding to nearest, ties to the even neighbour;
    // the largest finite values carry into the exponent and become inf
    const uint32_t r = (x + 0x7FFFu + ((x >> 16) & 1u)) >> 16;
    const bool nan = (x & 0x7FFFFFFFu) > 0x7F800000u;
    return (uint16_t)(nan ? ((x >> 16) | 0x0040u) : r);
}

// Elements per sub-block: the update pass leaves them in L1 for the cast pass.
constexpr int64_t kSub = 2048;

void update_block(const AdamScalars k, const float *__restrict g, float *__restrict th,
                  float *__restrict m, float *__restrict v, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        const float gc = g[i] * k.coef;
        const float mi = k.b1 * m[i] + k.omb1 * gc;
        const float vi = k.b2 * v[i] + k.omb2 * (gc * gc);
        const float mh = mi / k.bc1;
        const float vh = vi / k.bc2;
        const float t = th[i] * k.decay;
        th[i] = t - (k.lr * mh) / (std::sqrt(vh) + k.eps);
        m[i] = mi;
        v[i] = vi;
    }
}

void cast_block_f16(const float *__restrict th, uint16_t *__restrict out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = f16_rne(th[i]);
}

void cast_block_bf16(const float *__restrict th, uint16_t *__restrict out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_rne(th[i]);
}

}  // namespace

uint16_t f32_to_f16_rne(float f) { return f16_rne(f); }
uint16_t f32_to_bf16_rne(float f) { return bf16_rne(f); }

void adamw_cast_range(const AdamScalars &k, const float *g, float *th, float *m, float *v,
                      uint16_t *out, int64_t n, bool bf16) {
    for (int64_t i0 = 0; i0 < n; i0 += kSub) {
        const int64_t c = n - i0 < kSub ? n - i0 : kSub;
        update_block(k, g + i0, th + i0, m + i0, v + i0, c);
        if (bf16) cast_block_bf16(th + i0, out + i0, c);
        else cast_block_f16(th + i0, out + i0, c);
    }
}

int available_cpus() {
    cpu_set_t set;
    CPU_ZERO(&set);
    if (sched_getaffinity(0, sizeof(set), &set) == 0) {
        const int n = CPU_COUNT(&set);
        if (n > 0) return n;
    }
    const unsigned h = std::thread::hardware_concurrency();
    return h > 0 ? (int)h : 1;
}

Pool::Pool(int n_threads) {
    if (n_threads < 1) n_threads = 1;
    workers_.reserve(n_threads);
    for (int i = 0; i < n_threads; ++i) workers_.emplace_back([this] { loop(); });
}

Pool::~Pool() {
    {
        std::lock_guard<std::mutex> l(mu_);
        stop_ = true;
    }
    start_cv_.notify_all();
    for (auto &t : workers_) t.join();
}

void Pool::run(int64_t n_tasks, const std::function<void(int64_t)> &task) {
    if (n_tasks <= 0) return;
    std::unique_lock<std::mutex> l(mu_);
    task_ = &task;
    n_tasks_ = n_tasks;
    next_.store(0, std::memory_order_relaxed);
    busy_ = (int)workers_.size();
    ++generation_;
    start_cv_.notify_all();
    done_cv_.wait(l, [this] { return busy_ == 0; });
    task_ = nullptr;
}

void Pool::loop() {
    uint64_t seen = 0;
    std::unique_lock<std::mutex> l(mu_);
    for (;;) {
        start_cv_.wait(l, [&] { return stop_ || generation_ != seen; });
        if (stop_) return;
        seen = generation_;
        const std::function<void(int64_t)> *task = task_;
        const int64_t n = n_tasks_;
        l.unlock();
        for (int64_t t; (t = next_.fetch_add(1, std::memory_order_relaxed)) < n;) (*task)(t);
        l.lock();
        if (--busy_ == 0) done_cv_.notify_one();
    }
}

}  // namespace zh
