"""GPU parity of zero_shard_step_q8 (the step plus the ZeRO++ int8 all-gather
payload): the update matches the oracle as for the plain step, the int8
codes and per-block scales match the oracle's quantizer bit for bit on every
stepped shard, the 16-bit output can be omitted, and a skipped step leaves
the payload untouched."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth.workloads import AVG, BF16, F16, F32, SUM, Workload  # noqa: E402

import tests.oracle_runner as runner  # noqa: E402
from tests.gpu_helpers import (assert_params_close, assert_result, assert_state, f32,  # noqa: E402
                               host_grads, u16)

pytestmark = pytest.mark.gpu
BLOCK = 256


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _wl(name, shapes, N, ranks, dtype=F16, op=AVG, dynamic=True, steps=3, layout="full",
        inf_at=None):
    return Workload(name=name, description=name, shapes=shapes, world_size=N, ranks=ranks,
                    grad_dtype=dtype, op=op, dynamic=dynamic, steps=steps, sigma_g=1e-3,
                    sigma_n=1e-3, inf_at=inf_at, grads_layout=layout)


def _decode(u, bf16):
    if bf16:
        return (u.astype(np.uint32) << 16).view(np.float32)
    return u.view(np.float16).astype(np.float32)


CASES = [
    _wl("tiny_all", [(512, 1024), (1024,), (1024, 512), (512,)], 4, [0, 1, 2, 3]),
    _wl("ragged_pad", [(7, 13), (5,), (3, 3)], 4, [0, 1, 2, 3], steps=4, inf_at=(2, 1, 4)),
    _wl("bf16_sum", [(40_000,), (33,)], 8, list(range(8)), dtype=BF16, op=SUM, dynamic=False),
    _wl("odd_slot_slice", [(3_000_001,)], 8, [3], layout="slice"),
    _wl("fp32_contrib", [(100_000,)], 2, [0, 1], dtype=F32),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("with_out", [True, False], ids=["with_params", "q8_only"])
def test_q8_step(ora, w, with_out):
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    hp = ora.hparams(**w.hparams_kwargs())
    dw = DeviceWorkload(w, out_fill=0x5A5A)
    try:
        S, N = dw.S, w.world_size
        nb = -(-S // BLOCK)
        q8 = torch.full((dw.padded,), 0x55, dtype=torch.int8, device="cuda")
        scales = torch.full((N * nb,), -1.0, device="cuda")
        master = [f32(t).copy() for t in dw.master]
        m = [f32(t).copy() for t in dw.m]
        v = [f32(t).copy() for t in dw.v]
        out = u16(dw.out).copy()
        st = ora.scaler_init(hp)
        pbf16 = w.param_dtype == BF16
        want_q = np.full(dw.padded, 0x55, np.int8)
        want_s = np.full(N * nb, -1.0, np.float32)
        for step in range(w.steps):
            sc = dw.scaler()
            dw.gen_grads(step, sc.scale)
            g = host_grads(dw.grads)
            res = dw.flat.step_q8(w.ranks, dw.grads, dw.master, dw.m, dw.v,
                                  dw.out if with_out else None, q8, scales,
                                  grad_rank_offset_mul=w.grad_rank_mul)
            want = runner.shard_step(hp, st, N, dw.full, S, w.ranks, g, w.grad_ld,
                                     w.grad_rank_mul, master, m, v, out, avg=w.op == AVG,
                                     grad_is_bf16=w.grad_dtype == BF16, param_is_bf16=pbf16)
            assert_result(res, want)
            if not want[1]:                                    # applied: new payload
                for r in w.ranks:
                    p = _decode(out[r * S:(r + 1) * S], pbf16)
                    qq, ss = ora.quantize_q8(np.ascontiguousarray(p), BLOCK)
                    want_q[r * S:(r + 1) * S] = qq
                    want_s[r * nb:(r + 1) * nb] = ss
            for j in range(len(w.ranks)):
                assert_state(f32(dw.master[j]), f32(dw.m[j]), f32(dw.v[j]), master[j], m[j],
                             v[j], tag=" (step %d)" % step)
            if with_out:
                assert_params_close(u16(dw.out), out, pbf16, "params (step %d)" % step)
            else:
                assert bool((dw.out.view(torch.int16) == 0x5A5A).all())
            got_q = q8.cpu().numpy()
            got_s = scales.cpu().numpy()
            assert np.array_equal(got_q, want_q), "codes (step %d)" % step
            assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32)), \
                "scales (step %d)" % step
        # the receiver's dequantized shard is within half a step of the params
        for r in w.ranks:
            p = _decode(out[r * S:(r + 1) * S], pbf16).astype(np.float64)
            deq = got_q[r * S:(r + 1) * S] * np.repeat(got_s[r * nb:(r + 1) * nb], BLOCK)[:S]
            step_sz = np.repeat(got_s[r * nb:(r + 1) * nb], BLOCK)[:S].astype(np.float64)
            assert np.all(np.abs(deq - p) <= step_sz * (0.5 + 1e-5))
    finally:
        dw.close()


@pytest.mark.parametrize("mant,exp2", [(3, -11), (5, -12), (7, -9), (15, -13), (9, -10), (1, -8)])
def test_q8_exact_ties_round_to_even(ora, mant, exp2):
    """Blocks whose quotients p/scale are exactly k + 1/2 (lr = 0 and no decay
    keep the master weights, so the parameters are the designed values): the
    codes must round half to even, as the oracle's IEEE division does."""
    _need_gpu()
    import fsdp_sharded_mixed_zero_gb300 as Z
    n = 8 * BLOCK
    s = mant * 2.0 ** exp2                                   # the block scale
    ks = np.arange(-64, 64)
    block = np.concatenate([[127 * s], (2 * ks + 1) * s / 2])[:BLOCK]
    block = np.concatenate([block, np.zeros(BLOCK - block.size)])
    theta = np.tile(block, n // BLOCK).astype(np.float32)
    assert np.array_equal(theta.astype(np.float16).astype(np.float32), theta)
    hp = Z.hparams(lr=0.0, weight_decay=0.0, dynamic=False)
    f = Z.ZeroFlat([(n,)], 1, hp=hp)
    master = [torch.from_numpy(theta.copy()).cuda()]
    m = [torch.zeros(n, device="cuda")]
    v = [torch.zeros(n, device="cuda")]
    g = torch.zeros((1, n), dtype=torch.float16, device="cuda")
    out = torch.zeros(n, dtype=torch.float16, device="cuda")
    q8 = torch.zeros(n, dtype=torch.int8, device="cuda")
    sc = torch.zeros(n // BLOCK, device="cuda")
    res = f.step_q8([0], g, master, m, v, out, q8, sc)
    assert res.skipped == 0
    assert torch.equal(master[0].cpu(), torch.from_numpy(theta))
    want_q, want_s = ora.quantize_q8(theta, BLOCK)
    got = q8.cpu().numpy()
    assert np.array_equal(sc.cpu().numpy(), want_s) and want_s[0] == np.float32(s)
    assert np.array_equal(got, want_q)
    ties = got[1:1 + ks.size].astype(int)
    assert np.all(ties % 2 == 0)                             # k + 1/2 -> the even neighbour
    f.close()
