// zero_kernels.cuh -- device-side data structures and launch entry points of
// the ZeRO shard step (sm_103a).  See zero_kernels.cu for the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace zg {

// Stepped ranks handled by one launch (kernel-parameter tables stay < 4 KB;
// more ranks are processed in several launches).
constexpr int kMaxRanksPerLaunch = 64;
// Elements per thread-chunk: one 16-byte load of 16-bit gradients, two of fp32.
constexpr int kVec = 8;
constexpr int kBlock = 256;           // threads per block, reduce and AdamW kernels
constexpr int kFinalizeThreads = 1024;

// Device-resident state of a handle.  `scaler` persists across steps; `res`
// and the fields after it are written by the finalize kernel of each step and
// read by the AdamW kernel of the same step.  The first two members have the
// layout of zero_scaler_state and zero_step_result.
struct ScalerDev {
    float scale;
    int32_t good_steps;
    int64_t step_t;
    int64_t overflow_count;
};
struct ResultDev {
    int32_t overflow;
    int32_t skipped;
    double grad_norm;
    float clip_coef;
    float scale_used;
};
struct DevState {
    ScalerDev scaler;
    ResultDev res;
    float bc1, bc2;                   // bias corrections of this step (1 - beta^t)
    int32_t bc_saturated;             // t ran past the table: both corrections are 1
    int32_t error;                    // nonzero: a kernel gave up a bounded wait (the
                                      // step is then skipped as if it had overflowed)
};

// Elements per int8 quantization block of the all-gather payload (one warp's
// 32 x 8 elements in the quantizing AdamW kernel).
constexpr int kQ8Block = 256;

// Contribution encodings of the reduce kernel.
enum InKind : int { kInF16 = 0, kInBF16 = 1, kInF32 = 2 };

// What the reduce kernel does with the reduced value r of each element
// (r = sum of the N contributions in contributor order, / N for AVG):
//   kModeStep:     g = r / scale -> the fp32 gradient rows, overflow, norm
//   kModeAccFirst: acc = r                      (first micro-step)
//   kModeAccAdd:   acc = acc + r                (later micro-steps)
//   kModeNormOnly: g = acc / scale read from the accumulator: overflow and
//                  norm only (the AdamW kernel re-derives g from acc)
enum ReduceMode : int { kModeStep = 0, kModeAccFirst = 1, kModeAccAdd = 2, kModeNormOnly = 3 };

// K2: one block; deterministic total of the partials, norm, clip, loss scale.
struct FinalizeArgs {
    const double *part_ss;
    const int32_t *part_of;
    int32_t n_parts;
    int32_t dynamic;
    int32_t window;
    float min_scale;
    double extra_norm_sq;
    double max_grad_norm;
    const float2 *bc_table;           // bc_table[t] = {1 - b1^t, 1 - b2^t} as fp32
    int64_t bc_len;                   // entries t >= bc_len are {1, 1}
    float2 bc_given;                  // bc_table == NULL: the bias corrections of the
                                      // step this decision would apply, by value
    DevState *st;
    // non-NULL: only total the partials into *sum_out and *of_out (the first
    // half of a split step); no decision, no state change
    double *sum_out;
    int32_t *of_out;
};

// K1: reduce of the N contributions + AVG + unscale + overflow + norm partials.
// Row j of a launch (blockIdx.y) is one stepped rank's shard of one
// FlatParameter; rows may come from different FlatParameters that share the
// contributor count, the op and the contribution encoding.
struct ReduceArgs {
    double *part_ss;                  // per-block partial sums of squares
    int32_t *part_of;                 // per-block overflow flags
    int32_t part_base;                // partial index = part_base + j*gridDim.x + blockIdx.x
    int32_t n_contrib;
    int32_t avg;
    int32_t n_ranks;                  // rows in this launch
    const DevState *st;
    const void *in[kMaxRanksPerLaunch];   // contributor 0's element 0 of row j's slice
                                          // (kModeNormOnly: the row's accumulator)
    float *g[kMaxRanksPerLaunch];         // kModeStep: row j's reduced-gradient output
    int64_t g_stride;                     // g[j] == g[0] + j * g_stride when the rows are
                                          // one FlatParameter's (0: not evenly spaced)
    float *acc[kMaxRanksPerLaunch];       // kModeAccFirst / kModeAccAdd: row j's accumulator
    int64_t S[kMaxRanksPerLaunch];        // row j's shard size
    int64_t valid[kMaxRanksPerLaunch];    // elements [valid, S) are padding
    int64_t full_numel;                   // one-FlatParameter launches: valid is
    int64_t first[kMaxRanksPerLaunch];    // clamp(full_numel - first[j], 0, S)
    int64_t ld[kMaxRanksPerLaunch];       // contributor row stride of row j, elements
    uint8_t vec[kMaxRanksPerLaunch];      // 16-byte-aligned rows: vector path
    int32_t *err;                         // staged kernel: set on a timed-out wait
    uint32_t tx_pad;                      // staged kernel: bytes added to every stage's
                                          // expected transaction count (0; a test hook
                                          // that makes the waits run out)
    // The step's decision made by the block that finishes last (norm modes):
    // each block counts itself in *done after writing its partial; the one
    // that brings the count to total_blocks (over every launch of the step)
    // runs the finalize on all partials and resets the count.
    int32_t fuse_finalize;
    uint32_t total_blocks;
    uint32_t *done;
    FinalizeArgs fin;
};

// Elements per block tile of the staged reduce (one 8-element chunk per thread).
constexpr int kStageTile = kBlock * kVec;

// K3: AdamW + cast into the flat buffer; row j (blockIdx.y) as for K1.
struct AdamArgs {
    float b1, b2, omb1, omb2, eps;
    int32_t n_ranks;                  // rows in this launch
    const DevState *st;
    const float *g[kMaxRanksPerLaunch];   // reduced gradient row j (or its accumulator)
    float *master[kMaxRanksPerLaunch];
    float *m[kMaxRanksPerLaunch];
    float *v[kMaxRanksPerLaunch];
    uint16_t *out[kMaxRanksPerLaunch];    // row j's slot in its flat 16-bit buffer
                                          // (adamw_q8_kernel: may be NULL)
    int64_t S[kMaxRanksPerLaunch];        // elements updated in row j
    int64_t valid[kMaxRanksPerLaunch];    // from accumulators: [valid, S) is padding
    uint8_t vec[kMaxRanksPerLaunch];      // g/master/m/v 16-byte aligned
    uint8_t out_align[kMaxRanksPerLaunch];// byte alignment of the output slot: 16, 4 or 2
    // int8 all-gather payload (adamw_q8_kernel only): row j's codes and its
    // one fp32 scale per kQ8Block elements
    int8_t *q8[kMaxRanksPerLaunch];
    float *q8_scales[kMaxRanksPerLaunch];
    uint8_t q8_align[kMaxRanksPerLaunch];      // 8: 8-byte code stores, else byte stores
    // row j's learning rate and decay factor (float)(1 - lr*wd): the rows of a
    // group may belong to parameter groups with their own rates
    float lr[kMaxRanksPerLaunch];
    float decay[kMaxRanksPerLaunch];
};

// in_kind: InKind; mode: ReduceMode.  from_acc: g = acc / scale_used, with
// padding elements (flat index >= full_numel) taken as zero.  staged: the
// TMA-staged reduce for rows that are not 64-byte aligned (modes Step,
// AccFirst and AccAdd).
cudaError_t launch_reduce(const ReduceArgs &a, int grid_x, int in_kind, int mode, bool staged,
                          cudaStream_t s);
cudaError_t launch_finalize(const FinalizeArgs &a, cudaStream_t s);
cudaError_t launch_adamw(const AdamArgs &a, int grid_x, bool bf16_out, bool from_acc,
                         cudaStream_t s);
// AdamW + cast + int8 block quantization of the cast values (a.out may be NULL).
cudaError_t launch_adamw_q8(const AdamArgs &a, int grid_x, bool bf16_out, cudaStream_t s);


// Resident blocks per SM of one reduce-kernel instance (occupancy API).
cudaError_t reduce_blocks_per_sm(int in_kind, int mode, bool staged, int *bps);

}  // namespace zg
