// zero_group.cu -- groups of FlatParameter handles (include/zero.h,
// zero_group_*): the FlatParameters one rank steps together with one clip
// norm and one loss-scale decision, in one reduce launch and one update per
// 64 (member, stepped rank) rows, in every step form (plain, int8 payload,
// accumulation, offload).  Host side only: rows and launch plans; the
// kernels are the single-handle ones.
#include "zero_handle.h"

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <new>
#include <vector>

using namespace zi;

struct zero_group {
    zero_flat *core = nullptr;            // the group's state, table, counter and partials
    std::vector<zero_flat *> members;
};

namespace {

// Every field but lr and weight_decay, which each member keeps as its own
// parameter group's.
bool same_hparams(const zero_hparams &a, const zero_hparams &b) {
    return a.beta1 == b.beta1 && a.beta2 == b.beta2 && a.eps == b.eps &&
           a.max_grad_norm == b.max_grad_norm &&
           a.dynamic_loss_scale == b.dynamic_loss_scale &&
           a.initial_scale_power == b.initial_scale_power &&
           a.loss_scale_window == b.loss_scale_window && a.reserved == b.reserved &&
           a.static_loss_scale == b.static_loss_scale && a.min_loss_scale == b.min_loss_scale;
}

}  // namespace

ZERO_API zero_status zero_group_init(zero_flat *const *members, int32_t n_members,
                                     zero_group **out) {
    if (!out) return fail(ZERO_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!members || n_members < 1) return fail(ZERO_ERR_INVALID_ARG, "need at least one member");
    const zero_flat *a = members[0];
    for (int32_t k = 0; k < n_members; ++k) {
        const zero_flat *b = members[k];
        if (!b) return fail(ZERO_ERR_INVALID_ARG, "member %d is NULL", k);
        for (int32_t q = 0; q < k; ++q)
            if (members[q] == b) return fail(ZERO_ERR_INVALID_ARG, "member %d listed twice", k);
        if (b->device != a->device || b->world != a->world || b->grad_dtype != a->grad_dtype ||
            b->param_dtype != a->param_dtype || b->op != a->op || !same_hparams(b->hp, a->hp))
            return fail(ZERO_ERR_INVALID_ARG,
                        "member %d differs from member 0 (device, world size, dtypes, op or "
                        "hyper-parameters other than lr and weight_decay)", k);
    }
    DeviceGuard guard(a->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the members' device");
    zero_group *g = new (std::nothrow) zero_group;
    zero_flat *c = g ? new (std::nothrow) zero_flat : nullptr;
    if (!c) { delete g; return fail(ZERO_ERR_NO_MEMORY, "host allocation failed"); }
    g->core = c;
    c->device = a->device;
    c->sm_count = a->sm_count;
    for (int k = 0; k < 4; ++k) c->reduce_bps[k] = a->reduce_bps[k];
    for (int k = 0; k < 3; ++k) c->staged_bps[k] = a->staged_bps[k];
    c->world = a->world;
    c->grad_dtype = a->grad_dtype;
    c->param_dtype = a->param_dtype;
    c->op = a->op;
    c->hp = a->hp;
    c->b1 = a->b1; c->b2 = a->b2; c->omb1 = a->omb1; c->omb2 = a->omb2;
    c->lr = a->lr; c->eps = a->eps; c->decay = a->decay; c->min_scale = a->min_scale;
    zero_status s = init_device_state(c);
    if (s) { release(c); delete g; return s; }
    g->members.assign(members, members + n_members);
    *out = g;
    return ZERO_OK;
}

namespace {

enum GroupCall { kGroupStep, kGroupAccumulate, kGroupStepAccumulated, kGroupStepQ8 };

// Validate every member's arguments for `call`; on an error the message names
// the member.
zero_status check_group_args(const zero_group *g, const zero_group_member *args, GroupCall call) {
    for (size_t k = 0; k < g->members.size(); ++k) {
        const zero_flat *mk = g->members[k];
        const zero_group_member &x = args[k];
        int32_t max_rank = 0;
        zero_status s = check_ranks(mk, x.ranks, x.n_ranks, &max_rank);
        if (!s && (call == kGroupAccumulate || call == kGroupStepAccumulated))
            s = check_rows(mk, x.acc, x.n_ranks, "acc");
        if (!s && call != kGroupAccumulate)
            s = check_update(mk, x.n_ranks, x.master, x.m, x.v, x.flat_param_out, 0.0,
                             call == kGroupStepQ8);
        if (!s && call == kGroupStepQ8) {
            if (!x.flat_q8_out || !x.q8_scales)
                s = fail(ZERO_ERR_INVALID_ARG, "int8 outputs are NULL");
            else if ((uintptr_t)x.q8_scales % 4)
                s = fail(ZERO_ERR_ALIGNMENT, "q8_scales must be 4-byte aligned");
        }
        if (!s && call != kGroupStepAccumulated)
            s = check_grads(mk, x.grads, x.grad_ld, x.grad_rank_offset_mul, max_rank);
        if (s) {
            char msg[512];
            snprintf(msg, sizeof(msg), "member %zu: %.480s", k, g_last_error);
            return fail(s, "%s", msg);
        }
    }
    return ZERO_OK;
}

// The reduce rows (and, for the steps, the AdamW rows) of every member, in
// member order; *max_s = the largest shard.
zero_status group_rows(zero_group *g, const zero_group_member *args, int mode, bool q8,
                       std::vector<zg::ReduceRow> &rrows, std::vector<zg::AdamRow> *arows,
                       int64_t *max_s) {
    std::vector<zg::ReduceRow> part;
    *max_s = 0;
    for (size_t k = 0; k < g->members.size(); ++k) {
        zero_flat *mk = g->members[k];
        const zero_group_member &x = args[k];
        zg::ReducePlan p;
        p.mode = mode;
        p.ranks = x.ranks;
        p.n_ranks = x.n_ranks;
        p.S = mk->shard;
        p.full_numel = mk->full_numel;
        if (mode == zg::kModeNormOnly) {
            p.in_kind = zg::kInF32;
            p.acc_in = const_cast<const float *const *>(x.acc);
        } else {
            p.grads = x.grads;
            p.in_kind = in_kind_of(mk);
            p.ld = x.grad_ld;
            p.rank_mul = x.grad_rank_offset_mul;
            p.acc_out = x.acc;
        }
        if (mode == zg::kModeStep) {
            zero_status s = ensure_scratch(mk, x.n_ranks, 0);
            if (s) return s;
            mk->reduced_ranks.clear();    // this step overwrites the member's scratch
            p.g = mk->d_g;
            p.g_stride = mk->g_stride;
        }
        zg::reduce_rows_of(p, part);
        rrows.insert(rrows.end(), part.begin(), part.end());
        if (arows) {
            for (int32_t j = 0; j < x.n_ranks; ++j) {
                const int64_t r = x.ranks[j];
                zg::AdamRow w;
                w.g = mode == zg::kModeNormOnly ? x.acc[j] : mk->d_g + (int64_t)j * mk->g_stride;
                w.master = x.master[j];
                w.m = x.m[j];
                w.v = x.v[j];
                w.out = x.flat_param_out ? static_cast<uint16_t *>(x.flat_param_out) + r * mk->shard
                                         : nullptr;
                if (q8) {
                    w.q8 = x.flat_q8_out + r * mk->shard;
                    w.q8_scales = x.q8_scales + r * ((mk->shard + zg::kQ8Block - 1) / zg::kQ8Block);
                }
                w.S = mk->shard;
                w.valid = part[j].valid;
                w.lr = mk->lr;                // the member's parameter-group rates
                w.decay = mk->decay;
                arows->push_back(w);
            }
        }
        *max_s = std::max(*max_s, mk->shard);
    }
    return ZERO_OK;
}

// The plain or accumulated group step: the reduce (or norm pass) over every
// row with the decision in its last block, then one AdamW over every row.
// The reduce (or the norm pass) of a group step over every row, with the
// decision in its last block, queued on st; *arows: the rows of the update
// that follows, *max_s: the largest shard.
zero_status group_reduce(zero_group *g, const zero_group_member *args, double extra_norm_sq,
                         cudaStream_t st, GroupCall call, std::vector<zg::AdamRow> *arows,
                         int64_t *max_s) {
    const bool from_acc = call == kGroupStepAccumulated, q8 = call == kGroupStepQ8;
    zero_flat *c = g->core;
    const int mode = from_acc ? zg::kModeNormOnly : zg::kModeStep;
    std::vector<zg::ReduceRow> rrows;
    zero_status s = group_rows(g, args, mode, q8, rrows, arows, max_s);
    if (s) return s;
    const int32_t n_rows = (int32_t)rrows.size();
    zg::ReducePlan rp;
    rp.mode = mode;
    rp.in_kind = from_acc ? zg::kInF32 : in_kind_of(c);
    rp.n_contrib = c->world;
    rp.avg = c->op == ZERO_AVG;
    rp.st = c->d_state;
    rp.done = c->d_done;
    rp.staged = zg::rows_want_staging(rp.mode, rp.in_kind, rp.n_contrib, rrows.data(), n_rows);
    rp.grid_x = zg::grid_x_for(*max_s, std::min<int64_t>(n_rows, zg::kMaxRanksPerLaunch),
                               c->sm_count,
                               rp.staged ? c->staged_bps[rp.mode] : c->reduce_bps[rp.mode]);
    const int64_t parts = (int64_t)rp.grid_x * n_rows;
    if ((s = ensure_scratch(c, 0, parts))) return s;
    rp.part_ss = c->d_part_ss;
    rp.part_of = c->d_part_of;
    const zg::FinalizeArgs f = decision_args(c, c->d_part_ss, c->d_part_of,
                                             *max_s > 0 ? (int32_t)parts : 0, extra_norm_sq);
    rp.fuse_finalize = *max_s > 0;
    rp.fin = f;
    cudaError_t e;
    if ((e = zg::run_reduce_rows(rp, rrows.data(), n_rows, st))) return cuda_fail(e, "reduce kernel launch");
    if (!rp.fuse_finalize && (e = zg::launch_finalize(f, st)))
        return cuda_fail(e, "finalize kernel launch");
    return ZERO_OK;
}

// The group's AdamW plan (shared scalars, state, output encoding, grid).
zg::AdamPlan group_adam_plan(const zero_flat *c, int64_t max_s, int32_t n_rows, bool q8) {
    zg::AdamPlan ap;
    ap.bf16_out = c->param_dtype == ZERO_BF16;
    ap.b1 = c->b1; ap.b2 = c->b2; ap.omb1 = c->omb1; ap.omb2 = c->omb2;
    ap.eps = c->eps;
    ap.st = c->d_state;
    ap.grid_x = zg::grid_x_for(max_s, std::min<int32_t>(n_rows, zg::kMaxRanksPerLaunch),
                               c->sm_count, q8 ? zg::kAdamQ8BlocksPerSm : zg::kAdamBlocksPerSm);
    return ap;
}

// The plain, int8-payload or accumulated group step: the reduce (or norm
// pass) over every row with the decision in its last block, then one AdamW
// over every row.
zero_status group_step(zero_group *g, const zero_group_member *args, double extra_norm_sq,
                       void *stream, zero_step_result *res, GroupCall call) {
    if (!g || !args) return fail(ZERO_ERR_INVALID_ARG, "NULL argument");
    if (!std::isfinite(extra_norm_sq) || extra_norm_sq < 0)
        return fail(ZERO_ERR_INVALID_ARG, "extra_norm_sq must be finite and >= 0");
    zero_status s = check_group_args(g, args, call);
    if (s) return s;
    zero_flat *c = g->core;
    DeviceGuard guard(c->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the group's device");
    const cudaStream_t st = (cudaStream_t)stream;
    std::vector<zg::AdamRow> arows;
    int64_t max_s = 0;
    if ((s = group_reduce(g, args, extra_norm_sq, st, call, &arows, &max_s))) return s;
    const bool q8 = call == kGroupStepQ8;
    zg::AdamPlan ap = group_adam_plan(c, max_s, (int32_t)arows.size(), q8);
    if (call == kGroupStepAccumulated) ap.acc = args[0].acc;   // the rows' g are accumulators
    if (q8) ap.q8 = args[0].flat_q8_out;                       // the int8-payload kernel
    const cudaError_t e = zg::run_adamw_rows(ap, arows.data(), (int32_t)arows.size(), st);
    if (e) return cuda_fail(e, "adamw kernel launch");
    return res ? read_result(c, st, res) : ZERO_OK;
}

}  // namespace

ZERO_API zero_status zero_group_step(zero_group *g, const zero_group_member *args,
                                     double extra_norm_sq, void *stream, zero_step_result *res) {
    return group_step(g, args, extra_norm_sq, stream, res, kGroupStep);
}

ZERO_API zero_status zero_group_step_q8(zero_group *g, const zero_group_member *args,
                                        double extra_norm_sq, void *stream,
                                        zero_step_result *res) {
    return group_step(g, args, extra_norm_sq, stream, res, kGroupStepQ8);
}

ZERO_API zero_status zero_group_step_accumulated(zero_group *g, const zero_group_member *args,
                                                 double extra_norm_sq, void *stream,
                                                 zero_step_result *res) {
    return group_step(g, args, extra_norm_sq, stream, res, kGroupStepAccumulated);
}

ZERO_API zero_status zero_group_step_offload(zero_group *g, const zero_group_member *args,
                                             double extra_norm_sq, int32_t n_threads,
                                             double gpu_share, void *stream,
                                             zero_step_result *res) {
    if (!g || !args) return fail(ZERO_ERR_INVALID_ARG, "NULL argument");
    if (!std::isfinite(extra_norm_sq) || extra_norm_sq < 0)
        return fail(ZERO_ERR_INVALID_ARG, "extra_norm_sq must be finite and >= 0");
    if (n_threads < 0) return fail(ZERO_ERR_INVALID_ARG, "n_threads must be >= 0");
    if (!(gpu_share >= 0.0 && gpu_share <= 1.0))
        return fail(ZERO_ERR_INVALID_ARG, "gpu_share must be in [0, 1]");
    zero_status s = check_group_args(g, args, kGroupStep);
    if (s) return s;
    zero_flat *c = g->core;
    DeviceGuard guard(c->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the group's device");
    const size_t n_members = g->members.size();
    // member k's GPU share: elements [0, split[k]) of each of its rows
    std::vector<int64_t> split(n_members);
    for (size_t k = 0; k < n_members; ++k) {
        const zero_flat *mk = g->members[k];
        const int64_t S = mk->shard;
        split[k] = std::min(S, gpu_share >= 1.0
                                   ? S
                                   : (int64_t)(gpu_share * (double)S) / kHostChunk * kHostChunk);
        float *const *const rows[3] = {args[k].master, args[k].m, args[k].v};
        if (split[k] > 0 && !gpu_reaches(mk, args[k].n_ranks, rows))
            return fail(ZERO_ERR_INVALID_ARG, "member %zu: gpu_share > 0 needs host arrays the "
                        "GPU can access (pinned or registered)", k);
    }
    if ((s = ensure_host_runtime(c, n_threads))) return s;
    for (size_t k = 0; k < n_members; ++k)
        if ((s = ensure_host_rows(g->members[k], args[k].n_ranks, c->out_done))) return s;
    const cudaStream_t st = (cudaStream_t)stream;
    std::vector<zg::AdamRow> arows;
    int64_t max_s = 0;
    if ((s = group_reduce(g, args, extra_norm_sq, st, kGroupStep, &arows, &max_s))) return s;
    cudaError_t e = cudaMemcpyAsync(c->h_state, c->d_state, sizeof(zg::DevState),
                                    cudaMemcpyDeviceToHost, st);
    if (!e) e = cudaEventRecord(c->decided, st);
    if (e) return cuda_fail(e, "reading the step decision");
    // the GPU's share of every row, queued behind the decision
    std::vector<zg::AdamRow> gpu_rows;
    int64_t max_split = 0;
    for (size_t k = 0, i = 0; k < n_members; ++k)
        for (int32_t j = 0; j < args[k].n_ranks; ++j, ++i)
            if (split[k] > 0) {
                gpu_rows.push_back(arows[i]);
                gpu_rows.back().S = split[k];
                max_split = std::max(max_split, split[k]);
            }
    if (!gpu_rows.empty()) {
        const zg::AdamPlan ap = group_adam_plan(c, max_split, (int32_t)gpu_rows.size(), false);
        if ((e = zg::run_adamw_rows(ap, gpu_rows.data(), (int32_t)gpu_rows.size(), st)))
            return cuda_fail(e, "adamw kernel launch");
    }
    if ((e = cudaEventRecord(c->gpu_part_done, st))) return cuda_fail(e, "cudaEventRecord");
    if ((e = cudaEventSynchronize(c->decided))) return cuda_fail(e, "waiting for the step decision");
    const zg::DevState ds = *c->h_state;
    if (ds.error) return take_device_error(c, st);
    if (!ds.res.skipped) {
        // the previous call's parameter copies read the members' staging
        if ((e = cudaEventSynchronize(c->out_done))) return cuda_fail(e, "waiting for the last copies");
        std::vector<HostRow> rows;
        for (size_t k = 0; k < n_members; ++k) {
            zero_flat *mk = g->members[k];
            const zh::AdamScalars sk{c->b1, c->b2, c->omb1, c->omb2, mk->lr, c->eps, mk->decay,
                                     ds.res.clip_coef, ds.bc1, ds.bc2};
            host_rows_of(mk, sk, args[k].ranks, args[k].n_ranks, args[k].master, args[k].m,
                         args[k].v, args[k].flat_param_out, split[k], rows);
        }
        if ((e = host_update_rows(c, rows.data(), (int64_t)rows.size(),
                                  c->param_dtype == ZERO_BF16)))
            return cuda_fail(e, "copying parameters to the device");
        if ((e = cudaSetDevice(c->device))) return cuda_fail(e, "cudaSetDevice");
        if ((e = cudaEventRecord(c->out_done, c->up_stream))) return cuda_fail(e, "cudaEventRecord");
        if ((e = cudaStreamWaitEvent(st, c->out_done, 0))) return cuda_fail(e, "cudaStreamWaitEvent");
    }
    // the GPU's share of the host arrays is written when the call returns too
    if ((e = cudaEventSynchronize(c->gpu_part_done))) return cuda_fail(e, "waiting for the GPU share");
    if (res) {
        res->overflow = ds.res.overflow;
        res->skipped = ds.res.skipped;
        res->grad_norm = ds.res.grad_norm;
        res->clip_coef = ds.res.clip_coef;
        res->scale_used = ds.res.scale_used;
    }
    return ZERO_OK;
}

ZERO_API zero_status zero_group_accumulate(zero_group *g, const zero_group_member *args,
                                          int32_t first_micro_step, void *stream) {
    if (!g || !args) return fail(ZERO_ERR_INVALID_ARG, "NULL argument");
    zero_status s = check_group_args(g, args, kGroupAccumulate);
    if (s) return s;
    zero_flat *c = g->core;
    DeviceGuard guard(c->device);
    if (!guard.ok) return fail(ZERO_ERR_CUDA, "cannot select the group's device");
    const int mode = first_micro_step ? zg::kModeAccFirst : zg::kModeAccAdd;
    std::vector<zg::ReduceRow> rrows;
    int64_t max_s = 0;
    if ((s = group_rows(g, args, mode, false, rrows, nullptr, &max_s))) return s;
    const int32_t n_rows = (int32_t)rrows.size();
    zg::ReducePlan rp;
    rp.mode = mode;
    rp.in_kind = in_kind_of(c);
    rp.n_contrib = c->world;
    rp.avg = c->op == ZERO_AVG;
    rp.st = c->d_state;
    rp.staged = zg::rows_want_staging(rp.mode, rp.in_kind, rp.n_contrib, rrows.data(), n_rows);
    rp.grid_x = zg::grid_x_for(max_s, std::min<int64_t>(n_rows, zg::kMaxRanksPerLaunch),
                               c->sm_count,
                               rp.staged ? c->staged_bps[rp.mode] : c->reduce_bps[rp.mode]);
    const cudaError_t e = zg::run_reduce_rows(rp, rrows.data(), n_rows, (cudaStream_t)stream);
    if (e) return cuda_fail(e, "accumulate kernel launch");
    return ZERO_OK;
}

ZERO_API zero_status zero_group_loss_scaler_state(zero_group *g, zero_scaler_state *out,
                                                  void *stream) {
    if (!g) return fail(ZERO_ERR_INVALID_ARG, "group is NULL");
    return zero_loss_scaler_state(g->core, out, stream);
}

ZERO_API zero_status zero_group_set_loss_scaler_state(zero_group *g, const zero_scaler_state *in,
                                                      void *stream) {
    if (!g) return fail(ZERO_ERR_INVALID_ARG, "group is NULL");
    return zero_set_loss_scaler_state(g->core, in, stream);
}

ZERO_API zero_status zero_group_set_lr(zero_group *g, double lr) {
    if (!g) return fail(ZERO_ERR_INVALID_ARG, "group is NULL");
    zero_status s = zero_flat_set_lr(g->core, lr);
    for (size_t k = 0; k < g->members.size() && !s; ++k) s = zero_flat_set_lr(g->members[k], lr);
    return s;
}

ZERO_API zero_status zero_group_free(zero_group *g) {
    if (!g) return ZERO_OK;
    {
        DeviceGuard guard(g->core->device);
        cudaDeviceSynchronize();          // no group launch may still use the core's buffers
    }
    release(g->core);
    delete g;
    return ZERO_OK;
}
