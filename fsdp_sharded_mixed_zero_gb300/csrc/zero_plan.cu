// zero_plan.cu -- host-side planning: the staging decision and the launches
// of the reduce and AdamW kernels over any number of stepped ranks.
#include "zero_plan.h"

#include <atomic>

namespace zg {

namespace {
std::atomic<uint32_t> g_stage_tx_pad{0};
}  // namespace

void set_stage_tx_pad(uint32_t bytes) { g_stage_tx_pad.store(bytes); }

bool reduce_wants_staging(const ReducePlan &p) {
    if (p.mode == kModeNormOnly || p.S < kStageTile || !p.grads) return false;
    const size_t esize = p.in_kind == kInF32 ? 4 : 2;
    const bool rows_vary = p.n_contrib > 1 && ((size_t)p.ld * esize) % 64 != 0;
    bool any = false;
    for (int32_t j = 0; j < p.n_ranks; ++j) {
        const uintptr_t base = (uintptr_t)p.grads + (uintptr_t)(p.ranks[j] * p.rank_mul) * esize;
        any = any || rows_vary || base % 64 != 0;
        if ((p.mode == kModeAccFirst || p.mode == kModeAccAdd) && (uintptr_t)p.acc_out[j] % 16)
            return false;
    }
    return any;
}

cudaError_t run_reduce(const ReducePlan &p, cudaStream_t s) {
    if (p.S <= 0) return cudaSuccess;
    const size_t esize = p.in_kind == kInF32 ? 4 : 2;
    for (int32_t b0 = 0; b0 < p.n_ranks; b0 += kMaxRanksPerLaunch) {
        const int32_t nb = p.n_ranks - b0 < kMaxRanksPerLaunch ? p.n_ranks - b0 : kMaxRanksPerLaunch;
        ReduceArgs a{};
        a.ld = p.ld;
        a.S = p.S;
        a.full_numel = p.full_numel;
        a.g = p.g ? p.g + (int64_t)b0 * p.g_stride : nullptr;
        a.g_stride = p.g_stride;
        a.part_ss = p.part_ss;
        a.part_of = p.part_of;
        a.part_base = b0 * p.grid_x;
        a.n_contrib = p.mode == kModeNormOnly ? 1 : p.n_contrib;
        a.avg = p.mode == kModeNormOnly ? 0 : p.avg;
        a.n_ranks = nb;
        a.st = p.st;
        a.err = p.st ? const_cast<int32_t *>(&p.st->error) : nullptr;
        a.tx_pad = g_stage_tx_pad.load();
        a.fuse_finalize = p.fuse_finalize;
        a.total_blocks = (uint32_t)((int64_t)p.grid_x * p.n_ranks);
        a.done = p.done;
        a.fin = p.fin;
        for (int32_t j = 0; j < nb; ++j) {
            const int64_t r = p.ranks[b0 + j];
            bool vec;
            if (p.mode == kModeNormOnly) {
                a.in[j] = p.acc_in[b0 + j];
                vec = (uintptr_t)a.in[j] % 16 == 0;
            } else {
                a.in[j] = static_cast<const char *>(p.grads) + (size_t)(r * p.rank_mul) * esize;
                vec = (uintptr_t)a.in[j] % 16 == 0 && ((size_t)p.ld * esize) % 16 == 0;
            }
            if (p.mode == kModeAccFirst || p.mode == kModeAccAdd) {
                a.acc[j] = p.acc_out[b0 + j];
                vec = vec && (uintptr_t)a.acc[j] % 16 == 0;
            }
            a.first[j] = r * p.S;
            a.vec[j] = vec;
        }
        const cudaError_t e = launch_reduce(a, p.grid_x, p.in_kind, p.mode, p.staged, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t run_adamw(const AdamPlan &p, cudaStream_t s) {
    const int64_t count = p.count < 0 ? p.S : p.count;
    if (count <= 0) return cudaSuccess;
    if (count > p.S) return cudaErrorInvalidValue;
    if (p.q8 && (p.acc || count != p.S)) return cudaErrorInvalidValue;  // whole shards only
    for (int32_t b0 = 0; b0 < p.n_ranks; b0 += kMaxRanksPerLaunch) {
        const int32_t nb = p.n_ranks - b0 < kMaxRanksPerLaunch ? p.n_ranks - b0 : kMaxRanksPerLaunch;
        AdamArgs a{};
        a.S = count;                                   // the kernels' element range per rank
        a.full_numel = p.full_numel;
        a.b1 = p.b1; a.b2 = p.b2; a.omb1 = p.omb1; a.omb2 = p.omb2;
        a.lr = p.lr; a.eps = p.eps; a.decay = p.decay;
        a.n_ranks = nb;
        a.st = p.st;
        a.out = p.out;
        for (int32_t j = 0; j < nb; ++j) {
            const int64_t r = p.ranks[b0 + j];
            a.g[j] = p.acc ? p.acc[b0 + j] : p.g + (int64_t)(b0 + j) * p.g_stride;
            a.master[j] = p.master[b0 + j];
            a.m[j] = p.m[b0 + j];
            a.v[j] = p.v[b0 + j];
            a.out_off[j] = r * p.S;
            a.vec[j] = (uintptr_t)a.g[j] % 16 == 0 && (uintptr_t)a.master[j] % 16 == 0 &&
                       (uintptr_t)a.m[j] % 16 == 0 && (uintptr_t)a.v[j] % 16 == 0;
            const uintptr_t addr = (uintptr_t)p.out + (uintptr_t)(r * p.S) * 2;
            a.out_align[j] = addr % 16 == 0 ? 16 : (addr % 4 == 0 ? 4 : 2);
            if (p.q8) {
                a.q8_scale_off[j] = r * ((p.S + kQ8Block - 1) / kQ8Block);
                a.q8_align[j] = ((uintptr_t)(p.q8 + r * p.S)) % 8 == 0 ? 8 : 1;
            }
        }
        a.q8 = p.q8;
        a.q8_scales = p.q8_scales;
        const cudaError_t e = p.q8 ? launch_adamw_q8(a, p.grid_x, p.bf16_out, s)
                                   : launch_adamw(a, p.grid_x, p.bf16_out, p.acc != nullptr, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace zg
