// host_adam.h -- the host-CPU half of the ZeRO-Offload shard step: AdamW and
// the 16-bit cast over fp32 state in host memory ("DeepSpeed 与 FSDP"
// §ZeRO-Offload: gradients go to the CPU, the CPU updates the fp32 master
// weights, and the 16-bit weights go back to the GPU), run by a persistent
// pool of worker threads.  Plain C++17, no intrinsics: the same source builds
// on x86-64 and on the Grace (aarch64) host, and the compiler vectorises the
// element loops.  Internal to the library; the C entry points are in zero.h.
#pragma once

#include <atomic>
#include <condition_variable>
#include <cstdint>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

namespace zh {

// The per-step fp32 scalars of the update, each rounded once (from the fp64
// hyper-parameters, the clip coefficient and the bias corrections).
struct AdamScalars {
    float b1, b2, omb1, omb2, lr, eps, decay, coef, bc1, bc2;
};

// n elements in place: the moments, bias correction, decoupled decay and the
// Adam step on th (fp32 master), then out[i] = RNE 16-bit of th[i].  Every
// operation is a single IEEE fp32 operation (no contraction), so the result is
// bit-identical to the device kernel given the same scalars.
void adamw_cast_range(const AdamScalars &k, const float *g, float *th, float *m, float *v,
                      uint16_t *out, int64_t n, bool bf16);

// Round-to-nearest-even encodings of one fp32 value (NaN stays NaN, overflow
// goes to infinity, fp16 subnormals are rounded, not flushed).
uint16_t f32_to_f16_rne(float f);
uint16_t f32_to_bf16_rne(float f);

// Threads this process may run on (its CPU affinity mask).
int available_cpus();

// A fixed set of worker threads.  run() hands out task indices 0..n_tasks-1
// dynamically and returns once every task has finished; tasks must not throw.
class Pool {
  public:
    explicit Pool(int n_threads);
    ~Pool();
    Pool(const Pool &) = delete;
    Pool &operator=(const Pool &) = delete;
    int size() const { return (int)workers_.size(); }
    void run(int64_t n_tasks, const std::function<void(int64_t)> &task);

  private:
    void loop();
    std::vector<std::thread> workers_;
    std::mutex mu_;
    std::condition_variable start_cv_, done_cv_;
    const std::function<void(int64_t)> *task_ = nullptr;
    int64_t n_tasks_ = 0;
    std::atomic<int64_t> next_{0};
    uint64_t generation_ = 0;
    int busy_ = 0;
    bool stop_ = false;
};

}  // namespace zh
