"""Run the oracle's own pieces (reduce-scatter + unscale, norm, decision,
AdamW + cast) over a large shard with host threads: the same arithmetic as
ora_shard_step, only spread over cores (the squared norm is an exact sum,
so its order does not matter).  The equality
with ora_shard_step is itself a CPU test (test_oracle_runner.py).
"""
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle

CHUNK = 1 << 22
_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def _chunks(n):
    return [(a, min(a + CHUNK, n)) for a in range(0, n, CHUNK)]


def reduce_rank(grads, ld, rank_off, n_contrib, S, first, full, avg, scale, bf16, g):
    """g[:] = reduced, unscaled gradient of one shard, computed chunk-parallel."""
    flat = grads.reshape(-1)

    def job(ab):
        a, b = ab
        oracle.reduce_unscale(flat, ld, rank_off + a, n_contrib, b - a, first + a, full, avg,
                              scale, grad_is_bf16=bf16, out=g[a:b])

    list(_pool().map(job, _chunks(S)))


def norm_exact(arrays, acc=None, overflow=0):
    """Exact accumulation of the squares of every array (chunk-parallel; the
    exact sum does not depend on the order)."""
    jobs = [(a, lo, hi) for a in arrays for lo, hi in _chunks(a.size)]

    def job(x):
        a, lo, hi = x
        return oracle.norm_accumulate(a[lo:hi])

    acc = oracle.ExactAcc() if acc is None else acc
    for part, of in _pool().map(job, jobs):
        oracle.acc_merge(acc, part)
        overflow |= of
    return acc, overflow


def adamw_slot(hp, t, coef, g, master, m, v, out, param_is_bf16=False):
    """oracle.adamw_cast over one shard, chunk-parallel (the update is
    elementwise, so the chunking changes no result); out: the shard's 16-bit
    slot (uint16, same length)."""
    def job(ab):
        a, b = ab
        oracle.adamw_cast(hp, t, coef, g[a:b], master[a:b], m[a:b], v[a:b],
                          param_is_bf16=param_is_bf16, out=out[a:b])

    list(_pool().map(job, _chunks(g.size)))


def _decide_and_apply(hp, st, S, ranks, gs, master, m, v, out, param_is_bf16, extra_norm_sq,
                      coef_override, scale):
    acc, of = norm_exact(gs)
    norm = math.sqrt(oracle.norm_sum(acc) + extra_norm_sq)
    coef, skip = oracle.scaler_decide(hp, st, of, norm)
    if not skip:
        c = coef if coef_override is None else float(coef_override)
        for j, r in enumerate(ranks):
            adamw_slot(hp, st.step_t, c, gs[j], master[j], m[j], v[j], out[r * S:(r + 1) * S],
                       param_is_bf16)
    return of, skip, norm, coef, scale


def shard_step(hp, st, world_size, full, S, ranks, grads, ld, mul, master, m, v, out,
               avg=True, grad_is_bf16=False, param_is_bf16=False, extra_norm_sq=0.0,
               coef_override=None):
    """Equivalent of oracle.shard_step; returns (overflow, skipped, norm, coef, scale_used).
    coef_override: update with this clip coefficient instead of the oracle's own
    (the decision is still the oracle's) -- separates the norm's summation error
    from the elementwise arithmetic."""
    scale = st.scale
    gs = []
    for r in ranks:
        g = np.empty(max(S, 1), np.float32)[:S]
        reduce_rank(grads, ld, r * mul, world_size, S, r * S, full, avg, scale, grad_is_bf16, g)
        gs.append(g)
    return _decide_and_apply(hp, st, S, ranks, gs, master, m, v, out, param_is_bf16,
                             extra_norm_sq, coef_override, scale)


def unscale_acc(acc, first, full, scale, g):
    """g[:] = oracle.unscale_acc of the accumulator acc (flat indices from
    `first`), chunk-parallel."""
    def job(ab):
        a, b = ab
        oracle.unscale_acc(acc[a:b], first + a, full, scale, out=g[a:b])

    list(_pool().map(job, _chunks(acc.size)))


def shard_step_acc(hp, st, world_size, full, S, ranks, acc, master, m, v, out,
                   param_is_bf16=False, extra_norm_sq=0.0):
    """Equivalent of oracle.shard_step_acc (the step from fp32 accumulators);
    returns (overflow, skipped, norm, coef, scale_used)."""
    scale = st.scale
    gs = []
    for j, r in enumerate(ranks):
        g = np.empty(max(S, 1), np.float32)[:S]
        unscale_acc(acc[j], r * S, full, scale, g)
        gs.append(g)
    return _decide_and_apply(hp, st, S, ranks, gs, master, m, v, out, param_is_bf16,
                             extra_norm_sq, None, scale)


def accumulate_rows(grads, ld, n_contrib, count, full, avg, bf16, acc, first):
    """The oracle's grad_accumulate over `count` columns of a [n_contrib, ld]
    contribution block (flat indices from 0, no padding inside), into the
    fp32 slice acc, chunk-parallel."""
    flat = grads.reshape(-1)

    def job(ab):
        a, b = ab
        oracle.grad_accumulate(n_contrib, full, b - a, [0], flat[a:], ld, 0, [acc[a:b]],
                               first, avg=avg, grad_is_bf16=bf16)

    list(_pool().map(job, _chunks(count)))
