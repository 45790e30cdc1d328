// zero_plan.h -- host-side planning of the step's kernels over any number of
// stepped ranks (one launch per kMaxRanksPerLaunch ranks), shared by every
// entry point: which reduce kernel a plan takes, the launch geometry, and the
// per-launch argument blocks.
#pragma once

#include "zero_kernels.cuh"

#include <vector>

namespace zg {

// Host-side planning of one kernel class over any number of stepped ranks
// (one launch per kMaxRanksPerLaunch ranks), shared by every entry point.
struct ReducePlan {
    int mode = kModeStep;             // ReduceMode
    const void *grads = nullptr;      // contributions: rank r, contributor c, element i at
    int in_kind = kInF16;             //   grads[c*ld + r*rank_mul + i] (InKind encoding)
    int64_t ld = 0;
    int64_t rank_mul = 0;
    const float *const *acc_in = nullptr;  // kModeNormOnly: per-rank accumulators
    float *const *acc_out = nullptr;       // kModeAccFirst / kModeAccAdd
    float *g = nullptr;               // kModeStep: rows of g_stride floats per stepped rank
    int64_t g_stride = 0;
    double *part_ss = nullptr;        // kModeStep / kModeNormOnly: grid_x partials per rank
    int32_t *part_of = nullptr;
    const int32_t *ranks = nullptr;
    int32_t n_ranks = 0;
    int64_t S = 0, full_numel = 0;
    int32_t n_contrib = 1;
    int32_t avg = 0;
    const DevState *st = nullptr;
    int grid_x = 1;
    bool staged = false;              // reduce_wants_staging(*this), decided before grid_x
    // kModeStep / kModeNormOnly: finalize in the last block (done: a zeroed
    // device counter owned by the caller), else the caller launches K2
    bool fuse_finalize = false;
    uint32_t *done = nullptr;
    FinalizeArgs fin{};
};
cudaError_t run_reduce(const ReducePlan &p, cudaStream_t s);

// One row of a reduce launch: a stepped rank's shard of one FlatParameter.
struct ReduceRow {
    const void *in = nullptr;         // contributor 0's element 0 of the slice
                                      // (kModeNormOnly: the accumulator)
    int64_t ld = 0;                   // contributor row stride, elements
    int64_t S = 0;                    // shard size
    int64_t valid = 0;                // elements [valid, S) are padding
    float *g = nullptr;               // kModeStep: reduced-gradient output row
    float *acc = nullptr;             // kModeAccFirst / kModeAccAdd: accumulator
    int64_t first = 0;                // flat index of the shard's element 0
};
// The rows of a single-FlatParameter plan (its ranks, in order).
void reduce_rows_of(const ReducePlan &p, std::vector<ReduceRow> &rows);
// A reduce whose rows (over all its launches) hold at least this many
// contribution bytes takes the staged kernel even when every row is 64-byte
// aligned.  Measured on GB300 (same box, three alternations, 8 rows x 2
// stages): the bulk-copy reduce streams 6.8-6.9 TB/s whatever the contributor
// rows' stride, the plain one 5.97-6.67 TB/s depending on it (10B shard
// 3.78 -> 3.66 ms, 7B 2.53 -> 2.48, GPT-2's eight shards 0.417 -> 0.391, fp32
// contributions at 10B 7.05 -> 6.49, a 10B accumulation launch
// 4.15 -> 3.98), but the staged launch costs more fixed time: slower for the
// 1-MB tiny step (15.9 -> 17.5 us) and, by 1-3 %, for 1e8-param shards or
// groups of a few M-param members.  With 4 rows x 3 stages the staged reduce
// is still 1-6 % slower for reduces of 16 MB-512 MB and equal at 768 MB.
constexpr size_t kStageAlignedBytes = size_t(1) << 30;
// Whether rows should take the staged reduce: a row with a full tile, every
// accumulator 16-byte aligned, and either a row start off a 64-byte boundary
// or at least kStageAlignedBytes of contributions over all the rows.
bool rows_want_staging(int mode, int in_kind, int32_t n_contrib, const ReduceRow *rows,
                       int32_t n_rows);
// The launches of a reduce over any rows: p supplies the launch-wide settings
// (mode, encoding, contributor count, op, state, partials, grid, staging,
// decision); total_blocks of the decision counts every row.
cudaError_t run_reduce_rows(const ReducePlan &p, const ReduceRow *rows, int32_t n_rows,
                            cudaStream_t s, bool one_flat_parameter = false);
// (p.g_stride: the spacing of the rows' gradient outputs when they are one
// FlatParameter's scratch rows, else 0.)

// Test hook (zero_debug.h): bytes added to the staged reduce's expected
// transaction count per stage, 0 in normal operation.
void set_stage_tx_pad(uint32_t bytes);

// Whether a plan's contributions should go through the staged reduce: the
// shard holds at least one full tile, and some stepped rank has a contributor
// row whose start is not 64-byte aligned or the rows hold at least
// kStageAlignedBytes.  (A 16-byte vector load that starts inside a 64-byte
// DRAM access unit makes the unit's other half a separate request, which is
// fetched again: 7 % extra traffic with 32-byte aligned rows; 2-byte aligned
// rows cannot use vector loads at all.)  Plans whose accumulators are not
// 16-byte aligned stay on the plain kernel.
bool reduce_wants_staging(const ReducePlan &p);

struct AdamPlan {
    const float *g = nullptr;         // scratch rows (g_stride floats per stepped rank), or
    int64_t g_stride = 0;
    const float *const *acc = nullptr;    // per-rank accumulators (then g = acc / scale)
    float *const *master = nullptr, *const *m = nullptr, *const *v = nullptr;
    void *out = nullptr;
    bool bf16_out = false;
    const int32_t *ranks = nullptr;
    int32_t n_ranks = 0;
    int64_t S = 0, full_numel = 0;
    float b1 = 0, b2 = 0, omb1 = 0, omb2 = 0, lr = 0, eps = 0, decay = 0;
    const DevState *st = nullptr;
    int8_t *q8 = nullptr;             // non-NULL: also write the int8 payload and its scales
    float *q8_scales = nullptr;
    int grid_x = 1;
    int64_t count = -1;               // elements updated per rank from element 0 (< 0: S);
                                      // the output slot of rank r still starts at r * S
};
cudaError_t run_adamw(const AdamPlan &p, cudaStream_t s);

// One row of an AdamW launch.
struct AdamRow {
    const float *g = nullptr;         // reduced gradient (or accumulator) row
    float *master = nullptr, *m = nullptr, *v = nullptr;
    uint16_t *out = nullptr;          // the row's slot in its flat 16-bit buffer
    int64_t S = 0;                    // elements updated
    int64_t valid = 0;                // from accumulators: [valid, S) is padding
    int8_t *q8 = nullptr;             // int8 payload of the slot, and its scales
    float *q8_scales = nullptr;
    float lr = 0, decay = 0;          // the row's learning rate and (float)(1 - lr*wd)
};
// The launches of AdamW over any rows: p supplies the shared scalars (betas,
// eps), state, output encoding, accumulator mode (p.acc non-NULL), int8 mode
// (p.q8 non-NULL) and grid; each row its own lr and decay.
cudaError_t run_adamw_rows(const AdamPlan &p, const AdamRow *rows, int32_t n_rows,
                           cudaStream_t s);

// Launch geometry, measured on GB300 (152 SMs) on the 10B rank-7 step.  The
// AdamW kernel streams four arrays in and four out and is fastest with exactly
// two 256-thread blocks per SM (5.67 ms; 6.50 ms with four, 6.3 ms with three,
// and grids between whole multiples of the SM count are worse).  The
// read-dominated reduce is fastest with one full wave of resident blocks (its
// 48 registers allow five per SM; a partial second wave costs ~15 %).  A
// launch's blocks are split across the stepped ranks it handles and never
// exceed the work there is.
constexpr int kAdamBlocksPerSm = 2;
constexpr int kAdamQ8BlocksPerSm = 3;    // AdamW + int8 payload (72 registers): 6.10 ms vs 6.90 at two

inline int grid_x_for(int64_t S, int64_t ranks_in_launch, int sm_count, int blocks_per_sm) {
    const int64_t chunks = (S + kVec - 1) / kVec;
    const int64_t want = (chunks + kBlock - 1) / kBlock;
    int64_t cap = (int64_t)sm_count * blocks_per_sm / (ranks_in_launch > 0 ? ranks_in_launch : 1);
    if (cap < 1) cap = 1;
    const int64_t g = want < cap ? want : cap;
    return (int)(g < 1 ? 1 : g);
}

}  // namespace zg
