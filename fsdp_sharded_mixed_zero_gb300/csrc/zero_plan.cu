// zero_plan.cu -- host-side planning: the staging decision and the launches
// of the reduce and AdamW kernels over any number of stepped ranks.
#include "zero_plan.h"

#include <atomic>

namespace zg {

namespace {
std::atomic<uint32_t> g_stage_tx_pad{0};
}  // namespace

void set_stage_tx_pad(uint32_t bytes) { g_stage_tx_pad.store(bytes); }

void reduce_rows_of(const ReducePlan &p, std::vector<ReduceRow> &rows) {
    const size_t esize = p.in_kind == kInF32 ? 4 : 2;
    rows.resize(p.n_ranks);
    for (int32_t j = 0; j < p.n_ranks; ++j) {
        const int64_t r = p.ranks[j];
        ReduceRow &w = rows[j];
        if (p.mode == kModeNormOnly) {
            w.in = p.acc_in[j];
            w.ld = 0;
        } else {
            w.in = static_cast<const char *>(p.grads) + (size_t)(r * p.rank_mul) * esize;
            w.ld = p.ld;
        }
        w.S = p.S;
        int64_t valid = p.full_numel - r * p.S;
        w.valid = valid < 0 ? 0 : (valid > p.S ? p.S : valid);
        w.first = r * p.S;
        w.g = p.g ? p.g + (int64_t)j * p.g_stride : nullptr;
        w.acc = (p.mode == kModeAccFirst || p.mode == kModeAccAdd) ? p.acc_out[j] : nullptr;
    }
}

bool rows_want_staging(int mode, int in_kind, int32_t n_contrib, const ReduceRow *rows,
                       int32_t n_rows) {
    if (mode == kModeNormOnly) return false;
    const size_t esize = in_kind == kInF32 ? 4 : 2;
    bool any = false, tile = false;
    size_t bytes = 0;
    for (int32_t j = 0; j < n_rows; ++j) {
        const ReduceRow &w = rows[j];
        if (!w.in) return false;
        if ((mode == kModeAccFirst || mode == kModeAccAdd) && (uintptr_t)w.acc % 16) return false;
        const bool rows_vary = n_contrib > 1 && ((size_t)w.ld * esize) % 64 != 0;
        any = any || rows_vary || (uintptr_t)w.in % 64 != 0;
        tile = tile || w.S >= kStageTile;
        bytes += (size_t)(n_contrib > 0 ? n_contrib : 0) * (size_t)(w.S > 0 ? w.S : 0) * esize;
    }
    return tile && (any || bytes >= kStageAlignedBytes);
}

bool reduce_wants_staging(const ReducePlan &p) {
    if (p.mode == kModeNormOnly || !p.grads) return false;
    std::vector<ReduceRow> rows;
    reduce_rows_of(p, rows);
    return rows_want_staging(p.mode, p.in_kind, p.n_contrib, rows.data(), p.n_ranks);
}

cudaError_t run_reduce_rows(const ReducePlan &p, const ReduceRow *rows, int32_t n_rows,
                            cudaStream_t s, bool one_flat_parameter) {
    const size_t esize = p.in_kind == kInF32 ? 4 : 2;
    int64_t max_s = 0;
    for (int32_t j = 0; j < n_rows; ++j) max_s = rows[j].S > max_s ? rows[j].S : max_s;
    if (max_s <= 0) return cudaSuccess;
    for (int32_t b0 = 0; b0 < n_rows; b0 += kMaxRanksPerLaunch) {
        const int32_t nb = n_rows - b0 < kMaxRanksPerLaunch ? n_rows - b0 : kMaxRanksPerLaunch;
        ReduceArgs a{};
        a.part_ss = p.part_ss;
        a.part_of = p.part_of;
        a.part_base = b0 * p.grid_x;
        a.g_stride = p.g_stride;
        a.full_numel = one_flat_parameter ? p.full_numel : -1;
        a.n_contrib = p.mode == kModeNormOnly ? 1 : p.n_contrib;
        a.avg = p.mode == kModeNormOnly ? 0 : p.avg;
        a.n_ranks = nb;
        a.st = p.st;
        a.err = p.st ? const_cast<int32_t *>(&p.st->error) : nullptr;
        a.tx_pad = g_stage_tx_pad.load();
        a.fuse_finalize = p.fuse_finalize;
        a.total_blocks = (uint32_t)((int64_t)p.grid_x * n_rows);
        a.done = p.done;
        a.fin = p.fin;
        for (int32_t j = 0; j < nb; ++j) {
            const ReduceRow &w = rows[b0 + j];
            a.in[j] = w.in;
            a.g[j] = w.g;
            a.acc[j] = w.acc;
            a.S[j] = w.S;
            a.valid[j] = w.valid;
            a.first[j] = w.first;
            a.ld[j] = w.ld;
            bool vec = (uintptr_t)w.in % 16 == 0;
            if (p.mode != kModeNormOnly) vec = vec && ((size_t)w.ld * esize) % 16 == 0;
            if (p.mode == kModeAccFirst || p.mode == kModeAccAdd)
                vec = vec && (uintptr_t)w.acc % 16 == 0;
            a.vec[j] = vec;
        }
        const cudaError_t e = launch_reduce(a, p.grid_x, p.in_kind, p.mode, p.staged, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t run_reduce(const ReducePlan &p, cudaStream_t s) {
    if (p.S <= 0) return cudaSuccess;
    std::vector<ReduceRow> rows;
    reduce_rows_of(p, rows);
    return run_reduce_rows(p, rows.data(), p.n_ranks, s, true);
}

cudaError_t run_adamw_rows(const AdamPlan &p, const AdamRow *rows, int32_t n_rows,
                           cudaStream_t s) {
    int64_t max_s = 0;
    for (int32_t j = 0; j < n_rows; ++j) max_s = rows[j].S > max_s ? rows[j].S : max_s;
    if (max_s <= 0) return cudaSuccess;
    for (int32_t b0 = 0; b0 < n_rows; b0 += kMaxRanksPerLaunch) {
        const int32_t nb = n_rows - b0 < kMaxRanksPerLaunch ? n_rows - b0 : kMaxRanksPerLaunch;
        AdamArgs a{};
        a.b1 = p.b1; a.b2 = p.b2; a.omb1 = p.omb1; a.omb2 = p.omb2;
        a.eps = p.eps;
        a.n_ranks = nb;
        a.st = p.st;
        for (int32_t j = 0; j < nb; ++j) {
            const AdamRow &w = rows[b0 + j];
            a.g[j] = w.g;
            a.master[j] = w.master;
            a.m[j] = w.m;
            a.v[j] = w.v;
            a.out[j] = w.out;
            a.S[j] = w.S;
            a.valid[j] = w.valid;
            a.vec[j] = (uintptr_t)w.g % 16 == 0 && (uintptr_t)w.master % 16 == 0 &&
                       (uintptr_t)w.m % 16 == 0 && (uintptr_t)w.v % 16 == 0;
            const uintptr_t addr = (uintptr_t)w.out;
            a.out_align[j] = addr % 16 == 0 ? 16 : (addr % 4 == 0 ? 4 : 2);
            a.q8[j] = w.q8;
            a.q8_scales[j] = w.q8_scales;
            a.q8_align[j] = (uintptr_t)w.q8 % 8 == 0 ? 8 : 1;
            a.lr[j] = w.lr;
            a.decay[j] = w.decay;
        }
        const cudaError_t e = p.q8 ? launch_adamw_q8(a, p.grid_x, p.bf16_out, s)
                                   : launch_adamw(a, p.grid_x, p.bf16_out, p.acc != nullptr, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t run_adamw(const AdamPlan &p, cudaStream_t s) {
    const int64_t count = p.count < 0 ? p.S : p.count;
    if (count <= 0) return cudaSuccess;
    if (count > p.S) return cudaErrorInvalidValue;
    if (p.q8 && (p.acc || count != p.S)) return cudaErrorInvalidValue;  // whole shards only
    std::vector<AdamRow> rows(p.n_ranks);
    for (int32_t j = 0; j < p.n_ranks; ++j) {
        const int64_t r = p.ranks[j];
        AdamRow &w = rows[j];
        w.g = p.acc ? p.acc[j] : p.g + (int64_t)j * p.g_stride;
        w.master = p.master[j];
        w.m = p.m[j];
        w.v = p.v[j];
        w.out = p.out ? static_cast<uint16_t *>(p.out) + r * p.S : nullptr;
        w.S = count;                                   // the kernels' element range per rank
        int64_t valid = p.full_numel - r * p.S;
        w.valid = valid < 0 ? 0 : (valid > count ? count : valid);
        w.lr = p.lr;
        w.decay = p.decay;
        if (p.q8) {
            w.q8 = p.q8 + r * p.S;
            w.q8_scales = p.q8_scales + r * ((p.S + kQ8Block - 1) / kQ8Block);
        }
    }
    return run_adamw_rows(p, rows.data(), p.n_ranks, s);
}

}  // namespace zg
