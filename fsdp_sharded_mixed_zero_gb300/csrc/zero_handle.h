// zero_handle.h -- internal to the library: the FlatParameter handle behind
// the C ABI's opaque zero_flat, and the helpers that zero_api.cu (single
// handles, the offload host update) shares with zero_group.cu (groups of
// handles).  Not installed; no caller outside this directory includes it.
#pragma once

#include "zero.h"
#include "zero_debug.h"
#include "zero_plan.h"
#include "host_adam.h"

#include <cstdint>
#include <memory>
#include <vector>

#define ZERO_API extern "C" __attribute__((visibility("default")))

namespace zi {

// The calling thread's last error message (zero_last_error).
extern thread_local char g_last_error[512];

// Record a formatted message for zero_last_error and return s.
zero_status fail(zero_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
zero_status cuda_fail(cudaError_t e, const char *what);

inline bool mul_ok(int64_t a, int64_t b, int64_t *out) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > INT64_MAX / a) return false;
    *out = a * b;
    return true;
}
inline bool add_ok(int64_t a, int64_t b, int64_t *out) {
    if (a < 0 || b < 0 || a > INT64_MAX - b) return false;
    *out = a + b;
    return true;
}

// Switch to the handle's device for the duration of a call.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace zi

struct zero_flat {
    int device = 0;
    int sm_count = 0;
    int reduce_bps[4] = {1, 1, 1, 1}; // resident reduce blocks per SM, per ReduceMode
    int staged_bps[3] = {1, 1, 1};    // the same for the staged reduce (no kModeNormOnly)
    int32_t last_reduce_staged = -1;  // the form of the last contribution reduce (-1: none yet)
    int32_t world = 1;
    zero_dtype grad_dtype = ZERO_F16, param_dtype = ZERO_F16;
    zero_reduce_op op = ZERO_AVG;
    zero_hparams hp{};
    int64_t full_numel = 0, shard = 0, padded = 0;
    // per-element fp32 scalars, each rounded once from fp64
    float b1 = 0, b2 = 0, omb1 = 0, omb2 = 0, lr = 0, eps = 0, decay = 0, min_scale = 0;
    zg::DevState *d_state = nullptr;
    uint32_t *d_done = nullptr;       // blocks of the current reduce that have counted in
    float2 *d_bc = nullptr;
    int64_t bc_len = 0;
    float *d_g = nullptr;             // reduced-gradient rows
    int64_t g_stride = 0;             // floats per row (multiple of 4)
    int64_t g_rows = 0;
    double *d_part_ss = nullptr;
    int32_t *d_part_of = nullptr;
    int64_t parts_cap = 0;
    zg::DevState *h_state = nullptr;  // pinned staging for state reads
    uint64_t device_bytes = 0;
    // offload step: pinned host gradient rows and 16-bit staging, the host
    // worker pool, the stream and per-segment events of the gradient copies
    // to the host, and an event after the last parameter copy
    float *h_g = nullptr;
    int64_t h_g_rows = 0;
    uint16_t *h_out = nullptr;
    int64_t h_out_rows = 0;
    std::unique_ptr<zh::Pool> pool;
    cudaStream_t copy_stream = nullptr;   // gradient rows HBM -> host
    cudaStream_t up_stream = nullptr;     // 16-bit parameters host -> HBM
    std::vector<cudaEvent_t> seg_ev;
    cudaEvent_t out_done = nullptr;       // after the last parameter copy (up_stream)
    cudaEvent_t decided = nullptr;        // the decision read back (caller's stream)
    cudaEvent_t gpu_part_done = nullptr;  // the GPU's share of the update
    bool pageable_access = false;         // the device reads pageable host memory
    // split step: the ranks whose gradient rows zero_shard_reduce left in the
    // scratch, waiting for zero_shard_apply
    std::vector<int32_t> reduced_ranks;
    // per-kernel timing (zero_flat_profile_enable)
    bool profile = false;
    std::vector<cudaEvent_t> ev;      // 4 events per recorded step
    size_t ev_used = 0;
};


namespace zi {

// Device state (loss scale, bias-correction table, counter) of a new handle,
// and the release of everything a handle owns.
zero_status init_device_state(zero_flat *h);
void release(zero_flat *h);

// Reduced-gradient rows and norm partials, grown on demand.
zero_status ensure_scratch(zero_flat *h, int64_t rows, int64_t parts);

// Argument checks shared by every step entry point (each records the message).
zero_status check_ranks(const zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                        int32_t *max_rank);
zero_status check_grads(const zero_flat *h, const void *grads, int64_t grad_ld,
                        int64_t grad_rank_offset_mul, int32_t max_rank);
zero_status check_rows(const zero_flat *h, float *const *rows, int32_t n_ranks, const char *what);
zero_status check_update(const zero_flat *h, int32_t n_ranks, float *const *master,
                         float *const *m, float *const *v, void *flat_param_out,
                         double extra_norm_sq, bool out_optional = false);

int in_kind_of(const zero_flat *h);

// The decision's arguments over n_parts block partials, the step result read
// back on st, and the report of a kernel that gave up a bounded wait.
zg::FinalizeArgs decision_args(zero_flat *h, const double *part_ss, const int32_t *part_of,
                               int32_t n_parts, double extra_norm_sq);
zero_status read_result(zero_flat *h, cudaStream_t st, zero_step_result *res);
zero_status take_device_error(zero_flat *h, cudaStream_t st);

// ---- the offload step's host update

// Elements per host task, and per gradient / parameter copy segment.
constexpr int64_t kHostChunk = int64_t(1) << 16;
constexpr int64_t kHostSegment = int64_t(1) << 24;

zero_status ensure_host_rows(zero_flat *h, int32_t n_ranks, cudaEvent_t busy);
zero_status ensure_host_runtime(zero_flat *h, int32_t n_threads);

// One row of a host update: a stepped rank's shard of one FlatParameter,
// updated on the host over elements [i_begin, S) (i_begin a multiple of
// kHostChunk).
struct HostRow {
    const float *d_g;                 // the reduced gradient row in HBM
    float *h_g;                       // its pinned host copy
    float *master, *m, *v;            // fp32 state in host memory
    uint16_t *stage;                  // pinned 16-bit staging of the row
    uint16_t *d_out;                  // the row's slot in the device flat buffer
    int64_t S, i_begin;
    zh::AdamScalars k;                // the row's scalars (its parameter group's lr, decay)
};

cudaError_t host_update_rows(zero_flat *rt, const HostRow *rows, int64_t n_rows, bool bf16);
void host_rows_of(zero_flat *h, const zh::AdamScalars &k, const int32_t *ranks, int32_t n_ranks,
                  float *const *master, float *const *m, float *const *v, void *flat_param_out,
                  int64_t i_begin, std::vector<HostRow> &rows);
bool gpu_reaches(const zero_flat *h, int32_t n_ranks, float *const *const rows[3]);

}  // namespace zi
