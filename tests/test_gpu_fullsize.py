"""Full-size parity for the 7B (rank 0 of 8, 842,301,952 params) and 10B
(rank 7 of 8, 1.25e9 params) shards, in the launch configuration the
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
                               u16)

pytestmark = pytest.mark.gpu
SENTINEL = 0x5A5A
CHUNK = 1 << 26


def sample_indices(S, k, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([np.arange(64), np.arange(S - 64, S),
                                     rng.integers(0, S, k)])).astype(np.int64)


def oracle_reduce(ora, dw, w, scale, idx):
    """(sum of squares, overflow, reduced gradient at idx) by the oracle."""
    S, N, r = dw.S, w.world_size, w.ranks[0]
    bf16 = w.grad_dtype == BF16
    acc, of = ora.ExactAcc(), 0
    g_s = np.empty(idx.size, np.float32)
    for a in range(0, S, CHUNK):
        b = min(S, a + CHUNK)
        gh = u16(dw.grads[:, a:b].contiguous())
        g = np.empty(b - a, np.float32)
        runner.reduce_rank(gh, b - a, 0, N, b - a, r * S + a, dw.full, w.op == AVG, scale,
                           bf16, g)
        acc, of = runner.norm_exact([g], acc, of)
        lo, hi = np.searchsorted(idx, [a, b])
        g_s[lo:hi] = g[idx[lo:hi] - a]
    return ora.norm_sum(acc), of, g_s


@pytest.mark.parametrize("w", [W.LLAMA_7B, W.TEN_B], ids=lambda w: w.name)
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
