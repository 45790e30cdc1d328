"""Full-size parity for the 7B (rank 0 of 8, 842,301,952 params) and 10B
(rank 7 of 8, 1.25e9 params) shards, and for a 2.2e9-element shard (past the
int32 index range), in the launch configuration the
benchmark times.  Every step: the oracle reduces the whole gradient (chunks
copied to the host, reduced by the oracle's own code on host threads, squared
norm summed exactly), takes the loss-scale / clip decision, and
computes the AdamW update one by one for ~1M sampled elements (both ends of
the shard and random positions); those are compared with the GPU's state and
flat-buffer slot.  The buffer outside the slot must keep its fill."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth import workloads as W  # noqa: E402
from synth.workloads import AVG, BF16  # noqa: E402

import tests.oracle_runner as runner  # noqa: E402
from tests.gpu_helpers import (assert_params_close, assert_result, assert_state,  # noqa: E402
                               host_grads, u16)

pytestmark = pytest.mark.gpu
SENTINEL = 0x5A5A
CHUNK = 1 << 26


def sample_indices(S, k, seed):
    rng = np.random.default_rng(seed)
    parts = [np.arange(64), np.arange(S - 64, S), rng.integers(0, S, k)]
    for edge in (1 << 31, 1 << 32):                  # int32 / uint32 index boundaries
        if S > edge + 64:
            parts.append(np.arange(edge - 64, edge + 64))
    return np.unique(np.concatenate(parts)).astype(np.int64)


# A shard of more than 2^31 elements (rank 1 of 2, slot starting 4.4 GB into the
# flat buffer; ~53 GB resident): 64-bit indexing in every kernel.
HUGE = W.Workload(name="shard_2p2e9", description="2.2e9-element shard, N=2, rank 1",
                  shapes=[(4_400_000_004,)], world_size=2, ranks=[1], grad_dtype=W.F16, op=AVG,
                  dynamic=True, steps=2, sigma_g=2e-4, sigma_n=2e-4, seed=9,
                  grads_layout="slice")


def oracle_reduce(ora, dw, w, scale, idx):
    """(sum of squares, overflow, reduced gradient at idx) by the oracle."""
    S, N, r = dw.S, w.world_size, w.ranks[0]
    bf16 = w.grad_dtype == BF16
    acc, of = ora.ExactAcc(), 0
    g_s = np.empty(idx.size, np.float32)
    for a in range(0, S, CHUNK):
        b = min(S, a + CHUNK)
        gh = host_grads(dw.grads[:, a:b].contiguous())
        g = np.empty(b - a, np.float32)
        runner.reduce_rank(gh, b - a, 0, N, b - a, r * S + a, dw.full, w.op == AVG, scale,
                           bf16, g)
        acc, of = runner.norm_exact([g], acc, of)
        lo, hi = np.searchsorted(idx, [a, b])
        g_s[lo:hi] = g[idx[lo:hi] - a]
    return ora.norm_sum(acc), of, g_s


@pytest.mark.parametrize("w", [W.LLAMA_7B, W.TEN_B, W.TEN_B_F32, HUGE], ids=lambda w: w.name)
def test_fullsize_sampled(ora, w):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    hp = ora.hparams(**w.hparams_kwargs())
    dw = DeviceWorkload(w, out_fill=SENTINEL)
    try:
        S, r = dw.S, w.ranks[0]
        bf16 = w.grad_dtype == BF16
        idx = sample_indices(S, 1_000_000, 99)
        idx_t = torch.from_numpy(idx).cuda()
        th = dw.master[0][idx_t].cpu().numpy().copy()
        m = dw.m[0][idx_t].cpu().numpy().copy()
        v = dw.v[0][idx_t].cpu().numpy().copy()
        st = ora.scaler_init(hp)
        for step in range(w.warm_steps + w.steps):
            sc = dw.scaler()
            assert sc.as_tuple() == st.as_tuple()
            dw.gen_grads(step, sc.scale)
            ss, of, g_s = oracle_reduce(ora, dw, w, st.scale, idx)
            scale_used = st.scale
            res = dw.step()
            norm = math.sqrt(ss)
            coef, skip = ora.scaler_decide(hp, st, of, norm)
            assert_result(res, (of, skip, norm, coef, scale_used))
            out_s = None
            if not skip:
                out_s = ora.adamw_cast(hp, st.step_t, coef, g_s, th, m, v, param_is_bf16=bf16)
            assert_state(dw.master[0][idx_t].cpu().numpy(), dw.m[0][idx_t].cpu().numpy(),
                         dw.v[0][idx_t].cpu().numpy(), th, m, v, tag=" (step %d)" % step)
            if out_s is not None:
                got = u16(dw.out[r * S + idx_t])
                assert_params_close(got, out_s, bf16, "slot (step %d)" % step)
        assert dw.scaler().as_tuple() == st.as_tuple()
        # nothing outside the slot was written
        outside = [torch.arange(0, 4096, device="cuda"),
                   torch.arange(dw.padded - 4096, dw.padded, device="cuda")]
        for o in outside:
            o = o[(o < r * S) | (o >= (r + 1) * S)]
            assert bool((dw.out.view(torch.int16)[o] == SENTINEL).all())
    finally:
        dw.close()


def _decode16(u, bf16):
    if bf16:
        return (u.astype(np.uint32) << 16).view(np.float32)
    return u.view(np.float16).astype(np.float32)


def test_fullsize_q8_sampled_blocks(ora):
    """10B rank-7 step with the int8 payload: the oracle updates every element
    of ~4K sampled 256-element blocks (both ends of the shard included) and
    quantizes them; codes and scales must match bit for bit."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = W.TEN_B
    hp = ora.hparams(**w.hparams_kwargs())
    dw = DeviceWorkload(w, out_fill=SENTINEL)
    try:
        S, r, B = dw.S, w.ranks[0], 256
        nb = -(-S // B)
        rng = np.random.default_rng(5)
        blocks = np.unique(np.concatenate([[0, 1, nb - 2, nb - 1], rng.integers(0, nb, 4096)]))
        idx = np.concatenate([np.arange(b * B, min((b + 1) * B, S)) for b in blocks])
        idx_t = torch.from_numpy(idx).cuda()
        th = dw.master[0][idx_t].cpu().numpy().copy()
        m = dw.m[0][idx_t].cpu().numpy().copy()
        v = dw.v[0][idx_t].cpu().numpy().copy()
        q8 = torch.empty(dw.padded, dtype=torch.int8, device="cuda")
        scales = torch.empty(w.world_size * nb, device="cuda")
        st = ora.scaler_init(hp)
        for step in range(2):
            dw.gen_grads(step, st.scale)
            ss, of, g_s = oracle_reduce(ora, dw, w, st.scale, idx)
            scale_used = st.scale
            res = dw.flat.step_q8(w.ranks, dw.grads, dw.master, dw.m, dw.v, dw.out, q8, scales,
                                  grad_rank_offset_mul=w.grad_rank_mul)
            norm = math.sqrt(ss)
            coef, skip = ora.scaler_decide(hp, st, of, norm)
            assert_result(res, (of, skip, norm, coef, scale_used))
            out_s = ora.adamw_cast(hp, st.step_t, coef, g_s, th, m, v)
            assert_params_close(u16(dw.out[r * S + idx_t]), out_s, False, "slot")
            p = _decode16(out_s, False)
            got_q = q8[r * S + idx_t].cpu().numpy()
            got_s = scales[r * nb + torch.from_numpy(blocks).cuda()].cpu().numpy()
            pos = 0
            for k, b in enumerate(blocks):
                n_b = min((b + 1) * B, S) - b * B
                qq, sc = ora.quantize_q8(np.ascontiguousarray(p[pos:pos + n_b]), B)
                assert np.array_equal(got_q[pos:pos + n_b], qq), "block %d" % b
                assert got_s[k] == sc[0], "scale of block %d" % b
                pos += n_b
    finally:
        dw.close()


def test_fullsize_accumulation_sampled(ora):
    """10B rank-7 shard, 2 optimizer steps of 2 micro-steps: the oracle
    accumulates the whole shard on the host (for the norm), the accumulator
    and the update are compared on ~1M sampled elements."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = W.TEN_B
    K = 2
    hp = ora.hparams(**w.hparams_kwargs())
    dw = DeviceWorkload(w, out_fill=SENTINEL)
    try:
        dw.alloc_acc()
        S, r, N = dw.S, w.ranks[0], w.world_size
        idx = sample_indices(S, 1_000_000, 17)
        idx_t = torch.from_numpy(idx).cuda()
        th = dw.master[0][idx_t].cpu().numpy().copy()
        m = dw.m[0][idx_t].cpu().numpy().copy()
        v = dw.v[0][idx_t].cpu().numpy().copy()
        acc = np.zeros(S, np.float32)                       # the oracle's full accumulator
        st = ora.scaler_init(hp)
        for step in range(2):
            for k in range(K):
                dw.gen_grads(step * K + k, st.scale)
                dw.accumulate(first=(k == 0))
                for a in range(0, S, CHUNK):                # oracle: whole shard, chunked
                    b = min(S, a + CHUNK)
                    gh = host_grads(dw.grads[:, a:b].contiguous())
                    runner.accumulate_rows(gh, b - a, N, b - a, dw.full, w.op == AVG, False,
                                           acc[a:b], first=(k == 0))
                got = dw.acc[0][idx_t].cpu().numpy()
                assert np.array_equal(got.view(np.uint32), acc[idx].view(np.uint32))
            g = (acc / np.float32(st.scale)).astype(np.float32)
            ssacc, of = runner.norm_exact([g])
            scale_used = st.scale
            res = dw.step_accumulated()
            norm = math.sqrt(ora.norm_sum(ssacc))
            coef, skip = ora.scaler_decide(hp, st, of, norm)
            assert_result(res, (of, skip, norm, coef, scale_used))
            out_s = ora.adamw_cast(hp, st.step_t, coef, np.ascontiguousarray(g[idx]), th, m, v)
            assert_state(dw.master[0][idx_t].cpu().numpy(), dw.m[0][idx_t].cpu().numpy(),
                         dw.v[0][idx_t].cpu().numpy(), th, m, v, tag=" (step %d)" % step)
            assert_params_close(u16(dw.out[r * S + idx_t]), out_s, False, "slot")
    finally:
        dw.close()
