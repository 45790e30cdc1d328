"""Element-complete parity at full size, in the launch configuration the
benchmark times: the 7B shard (rank 0 of 8, 842,301,952 params, every step:
one warm step and five more), the 10B shard (rank 7 of 8, 1.25e9 params) with
fp16 and with fp32 contributions, and a 2.2e9-element shard (past the int32
index range), two steps each.

The oracle keeps its own copy of the whole shard's master, m and v in host
memory and steps it with its own pieces on host threads (tests/oracle_runner,
pinned equal to ora_shard_step): the contributions are copied to the host in
chunks and reduced there, the squared norm is summed exactly, the loss-scale /
clip decision is the oracle's, and AdamW + the cast run over every element.
After every step every element of the GPU's master, m, v and 16-bit slot is
compared with the oracle's (bit-equal, or within the stated tolerances), and
the flat buffer outside the slot must keep its fill."""
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth import workloads as W  # noqa: E402
from synth.workloads import AVG, BF16  # noqa: E402

import tests.oracle_runner as runner  # noqa: E402
from tests.gpu_helpers import (MASTER_ATOL, MASTER_RTOL, MV_ATOL, MV_RTOL,  # noqa: E402
                               assert_params_close, assert_rel, assert_result, host_grads, u16)

pytestmark = pytest.mark.gpu
SENTINEL = 0x5A5A
CHUNK = 1 << 26

# A shard of more than 2^31 elements (rank 1 of 2, slot starting 4.4 GB into the
# flat buffer; ~53 GB resident): 64-bit indexing in every kernel.
HUGE = W.Workload(name="shard_2p2e9", description="2.2e9-element shard, N=2, rank 1",
                  shapes=[(4_400_000_004,)], world_size=2, ranks=[1], grad_dtype=W.F16, op=AVG,
                  dynamic=True, steps=2, sigma_g=2e-4, sigma_n=2e-4, seed=9,
                  grads_layout="slice")

# steps compared per workload: every step of the 7B run, two of the others
STEPS = {W.LLAMA_7B.name: W.LLAMA_7B.warm_steps + W.LLAMA_7B.steps, W.TEN_B.name: 2,
         W.TEN_B_F32.name: 2, HUGE.name: 2}

_POOL = ThreadPoolExecutor(max_workers=8)


def to_host(t):
    """A 1-D device tensor copied to a host numpy array in chunks (fp32, or
    uint16 encodings of a 16-bit tensor)."""
    n = t.numel()
    is16 = t.element_size() == 2
    out = np.empty(n, np.uint16 if is16 else np.float32)
    for a in range(0, n, CHUNK):
        b = min(n, a + CHUNK)
        out[a:b] = u16(t[a:b]) if is16 else t[a:b].cpu().numpy()
    return out


def oracle_reduce(dw, w, scale):
    """The oracle's reduced, unscaled gradient of the whole stepped shard."""
    S, N, r = dw.S, w.world_size, w.ranks[0]
    g = np.empty(S, np.float32)
    for a in range(0, S, CHUNK):
        b = min(S, a + CHUNK)
        gh = host_grads(dw.grads[:, a:b].contiguous())
        runner.reduce_rank(gh, b - a, 0, N, b - a, r * S + a, dw.full, w.op == AVG, scale,
                           w.grad_dtype == BF16, g[a:b])
    return g


def _cmp_f32(got, want, rtol, atol, what):
    neq = got.view(np.uint32) != want.view(np.uint32)
    k = int(neq.sum())
    if k:
        assert_rel(got[neq], want[neq], rtol, atol, what)
    return k


def compare_all(dw, r, state, out_slot, bf16, tag, in_flight=6):
    """Every element of master, m, v and the slot against the oracle's,
    chunk by chunk (copies on this thread, comparisons on the pool, at most
    `in_flight` chunks held on the host); returns the number of elements that
    were not bit-equal."""
    S = dw.S
    master, m, v = state

    def job(a, b, gm, gmm, gv, go):
        n = _cmp_f32(gm, master[a:b], MASTER_RTOL, MASTER_ATOL, "master" + tag)
        n += _cmp_f32(gmm, m[a:b], MV_RTOL, MV_ATOL, "m" + tag)
        n += _cmp_f32(gv, v[a:b], MV_RTOL, MV_ATOL, "v" + tag)
        if not np.array_equal(go, out_slot[a:b]):
            assert_params_close(go, out_slot[a:b], bf16, "slot" + tag)
            n += int((go != out_slot[a:b]).sum())
        return n

    pending, total = [], 0
    for a in range(0, S, CHUNK):
        b = min(S, a + CHUNK)
        pending.append(_POOL.submit(job, a, b, dw.master[0][a:b].cpu().numpy(),
                                    dw.m[0][a:b].cpu().numpy(), dw.v[0][a:b].cpu().numpy(),
                                    u16(dw.out[r * S + a:r * S + b])))
        if len(pending) >= in_flight:
            total += pending.pop(0).result()
    for f in pending:
        total += f.result()
    return total


def check_outside_slot(dw, r):
    S = dw.S
    outside = [torch.arange(0, 4096, device="cuda"),
               torch.arange(dw.padded - 4096, dw.padded, device="cuda")]
    for o in outside:
        o = o[(o < r * S) | (o >= (r + 1) * S)]
        assert bool((dw.out.view(torch.int16)[o] == SENTINEL).all())


@pytest.mark.parametrize("w", [W.LLAMA_7B, W.TEN_B, W.TEN_B_F32, HUGE], ids=lambda w: w.name)
def test_fullsize_every_element(ora, w):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    hp = ora.hparams(**w.hparams_kwargs())
    dw = DeviceWorkload(w, out_fill=SENTINEL)
    try:
        S, r = dw.S, w.ranks[0]
        bf16 = w.param_dtype == BF16
        state = [to_host(dw.master[0]), to_host(dw.m[0]), to_host(dw.v[0])]
        out_slot = to_host(dw.out[r * S:(r + 1) * S])
        st = ora.scaler_init(hp)
        for step in range(STEPS[w.name]):
            sc = dw.scaler()
            assert sc.as_tuple() == st.as_tuple()
            dw.gen_grads(step, sc.scale)
            g = oracle_reduce(dw, w, st.scale)
            scale_used = st.scale
            res = dw.step()
            acc, of = runner.norm_exact([g])
            norm = math.sqrt(ora.norm_sum(acc))
            coef, skip = ora.scaler_decide(hp, st, of, norm)
            assert_result(res, (of, skip, norm, coef, scale_used))
            if not skip:
                runner.adamw_slot(hp, st.step_t, coef, g, *state, out_slot, bf16)
            del g
            compare_all(dw, r, state, out_slot, bf16, " (step %d)" % step)
        assert dw.scaler().as_tuple() == st.as_tuple()
        check_outside_slot(dw, r)
    finally:
        dw.close()


def _decode16(u, bf16):
    if bf16:
        return (u.astype(np.uint32) << 16).view(np.float32)
    return u.view(np.float16).astype(np.float32)


def test_fullsize_q8_every_block(ora):
    """10B rank-7 step with the int8 payload, two steps: the oracle updates
    the whole shard and quantizes every 256-element block of its 16-bit
    values; every code and every block scale must match bit for bit."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = W.TEN_B
    B = 256
    hp = ora.hparams(**w.hparams_kwargs())
    dw = DeviceWorkload(w, out_fill=SENTINEL)
    try:
        S, r = dw.S, w.ranks[0]
        nb = -(-S // B)
        state = [to_host(dw.master[0]), to_host(dw.m[0]), to_host(dw.v[0])]
        out_slot = to_host(dw.out[r * S:(r + 1) * S])
        q8 = torch.empty(dw.padded, dtype=torch.int8, device="cuda")
        scales = torch.empty(w.world_size * nb, device="cuda")
        st = ora.scaler_init(hp)
        for step in range(2):
            dw.gen_grads(step, st.scale)
            g = oracle_reduce(dw, w, st.scale)
            scale_used = st.scale
            res = dw.flat.step_q8(w.ranks, dw.grads, dw.master, dw.m, dw.v, dw.out, q8, scales,
                                  grad_rank_offset_mul=w.grad_rank_mul)
            acc, of = runner.norm_exact([g])
            norm = math.sqrt(ora.norm_sum(acc))
            coef, skip = ora.scaler_decide(hp, st, of, norm)
            assert_result(res, (of, skip, norm, coef, scale_used))
            assert not skip
            runner.adamw_slot(hp, st.step_t, coef, g, *state, out_slot, False)
            del g
            compare_all(dw, r, state, out_slot, False, " (step %d)" % step)
            step_chunk = CHUNK // B * B                   # whole blocks per chunk

            def job(ab):
                a, b = ab
                p = _decode16(out_slot[a:b], False)
                qq, sc = ora.quantize_q8(np.ascontiguousarray(p), B)
                got_q = q8[r * S + a:r * S + b].cpu().numpy()
                got_s = scales[r * nb + a // B:r * nb + -(-b // B)].cpu().numpy()
                assert np.array_equal(got_q, qq), "codes in [%d, %d)" % (a, b)
                assert np.array_equal(got_s.view(np.uint32), sc.view(np.uint32)), \
                    "scales in [%d, %d)" % (a, b)

            list(_POOL.map(job, [(a, min(S, a + step_chunk)) for a in range(0, S, step_chunk)]))
    finally:
        dw.close()


def test_fullsize_accumulation_every_element(ora):
    """10B rank-7 shard, 2 optimizer steps of 2 micro-steps: the oracle
    accumulates the whole shard on the host (ora_grad_accumulate on host
    threads) and takes the step from its accumulator with its own pieces
    (runner.shard_step_acc, pinned equal to ora_shard_step_acc); every element
    of the accumulator, master, m, v and the slot is compared."""
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
        state = [to_host(dw.master[0]), to_host(dw.m[0]), to_host(dw.v[0])]
        out_slot = to_host(dw.out[r * S:(r + 1) * S])
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
                got = to_host(dw.acc[0])
                assert np.array_equal(got.view(np.uint32), acc.view(np.uint32)), \
                    "accumulator (step %d, micro-step %d)" % (step, k)
                del got
            scale_used = st.scale
            res = dw.step_accumulated()
            # the oracle's step from its accumulator; its flat buffer is the
            # rank's slot alone, so it is given as a one-rank layout
            want = runner.shard_step_acc(hp, st, N, dw.full, S, [r], [acc], [state[0]],
                                         [state[1]], [state[2]],
                                         _SlotView(out_slot, r * S), param_is_bf16=False)
            of, skip, norm, coef, _ = want
            assert_result(res, (of, skip, norm, coef, scale_used))
            compare_all(dw, r, state, out_slot, False, " (step %d)" % step)
    finally:
        dw.close()


class _SlotView:
    """The flat buffer as the runner indexes it (out[r*S:(r+1)*S]) when only
    rank r's slot is kept on the host."""

    def __init__(self, slot, base):
        self.slot, self.base = slot, base

    def __getitem__(self, sl):
        assert isinstance(sl, slice) and sl.start >= self.base
        return self.slot[sl.start - self.base:sl.stop - self.base]
