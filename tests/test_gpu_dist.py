"""The multi-rank step with the library's kernels: two (or three) processes,
one rank each, joined by a gloo group on 127.0.0.1 and sharing this one GPU.  Each
process steps only its own shard (RankStep: the all-to-all of the
reduce-scatter, zero_shard_reduce, the all-gather of the two scalars,
zero_shard_apply_partials, the all-gather of the 16-bit slots); every
exchange goes through gloo on host-staged buffers, so no kernel of one
process waits on the other.  On every rank and every step, the result, the
loss-scale state, the rank's master / m / v and the whole gathered flat
buffer are compared with the oracle's step of all shards at once on the
stacked contributions, at the parity tolerances; one rank's inf must make
both ranks skip and halve the scale.  The ZeRO++ form exchanges only the int8
payload: every gathered code and block scale must equal the oracle's
quantization of every rank's parameters.  A last test runs one rank over NCCL
(a one-rank communicator on this GPU): the device-tensor branch of every
exchange, with no host staging, against the oracle."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as tdist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
F16, BF16, F32, SUM, AVG = 0, 1, 2, 0, 1

CASES = [
    # odd shard: rank 1's slice and the received rows are off 16-byte boundaries
    dict(name="fp16_avg_dynamic_ragged", full=1_000_003, dtype=F16, op=AVG, dynamic=True),
    # every row 64-byte aligned: the vectorised reduce
    dict(name="bf16_sum_static_aligned", full=2 * 262_144, dtype=BF16, op=SUM, dynamic=False),
    # fp32 contributions (a reduce_dtype=float32 reduce-scatter), fp16 parameters
    dict(name="fp32_contributions_avg", full=700_001, dtype=F16, gdtype=F32, op=AVG,
         dynamic=True),
    # three ranks, three processes
    dict(name="three_ranks_fp16_avg", full=900_005, dtype=F16, op=AVG, dynamic=True, world=3),
]
STEPS, INF_STEP = 4, 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, case):
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    torch.cuda.set_device(0)
    WORLD = case.get("world", 2)
    tdist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                             world_size=WORLD)
    import fsdp_sharded_mixed_zero_gb300 as Z
    import oracle
    import synth
    from fsdp_sharded_mixed_zero_gb300.dist import RankStep
    from tests.gpu_helpers import assert_params_close, assert_result, assert_state, f32, u16

    full, dt, bf16 = case["full"], case["dtype"], case["dtype"] == BF16
    gdt = case.get("gdtype", dt)
    kw = dict(dynamic=case["dynamic"], lr=1e-3, window=3, initial_scale_power=12)
    flat = Z.ZeroFlat([(full,)], WORLD, gdt, dt, case["op"], Z.hparams(**kw))
    ohp = oracle.hparams(**kw)
    S, padded = flat.shard_size, flat.padded_numel
    tdt = torch.bfloat16 if bf16 else torch.float16
    gtdt = torch.float32 if gdt == F32 else tdt
    sdt = synth.F32 if gdt == F32 else (synth.BF16 if bf16 else synth.F16)
    step_of = RankStep(flat, rank, grad_dtype=gdt)
    # this rank's shard, and the oracle's copy of every shard
    master_all = torch.empty(padded, device="cuda")
    synth.normal_device(master_all, 41, synth.MASTER, 0, 0.02)
    master_all[full:].zero_()
    master = master_all[rank * S:(rank + 1) * S].clone()
    m = torch.zeros(S, device="cuda")
    v = torch.zeros(S, device="cuda")
    out = torch.zeros(padded, dtype=tdt, device="cuda")
    o_state = [[f32(master_all[k * S:(k + 1) * S]).copy() for k in range(WORLD)],
               [np.zeros(S, np.float32) for _ in range(WORLD)],
               [np.zeros(S, np.float32) for _ in range(WORLD)]]
    o_out = np.zeros(padded, np.uint16)
    o_st = oracle.scaler_init(ohp)
    mine = torch.empty((1, padded), dtype=gtdt, device="cuda")
    everyone = torch.empty((WORLD, padded), dtype=gtdt, device="cuda")
    for step in range(STEPS):
        scale = flat.scaler_state().scale
        assert scale == o_st.scale
        # this rank's own gradient (contributor `rank`), and all of them for the oracle
        synth.grads_device(mine, 41, step, 0, padded, 1e-3, 1e-3, scale, sdt, zero_from=full,
                           c0=rank, n_contrib=1)
        synth.grads_device(everyone, 41, step, 0, padded, 1e-3, 1e-3, scale, sdt,
                           zero_from=full)
        if step == INF_STEP:                 # rank 1's gradient, inside rank 0's slice
            everyone[1, 777] = float("inf")
            if rank == 1:
                mine[0, 777] = float("inf")
        assert torch.equal(mine[0], everyone[rank]) if gdt == F32 else \
            torch.equal(mine[0].view(torch.int16), everyone[rank].view(torch.int16))
        g_host = everyone.cpu().numpy() if gdt == F32 else u16(everyone)
        scale_used = o_st.scale
        ro = oracle.shard_step(ohp, o_st, WORLD, full, S, list(range(WORLD)), g_host, padded, S,
                               *o_state, o_out, avg=case["op"] == AVG, grad_is_bf16=bf16,
                               param_is_bf16=bf16)
        res = step_of.step(mine.view(-1), master, m, v, out)
        torch.cuda.synchronize()
        tag = " (rank %d, step %d)" % (rank, step)
        assert_result(res, (ro.overflow, ro.skipped, ro.grad_norm, ro.clip_coef, scale_used))
        assert flat.scaler_state().as_tuple() == o_st.as_tuple(), tag
        assert_state(f32(master), f32(m), f32(v), o_state[0][rank], o_state[1][rank],
                     o_state[2][rank], tag=tag)
        assert_params_close(u16(out), o_out, bf16, "gathered flat buffer" + tag)
        assert res.skipped == (step == INF_STEP), tag
    assert o_st.overflow_count == 1
    flat.close()
    tdist.destroy_process_group()


@pytest.mark.parametrize("case", CASES, ids=lambda c: c["name"])
def test_two_ranks_on_gloo_match_the_all_shards_step(case):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    mp.start_processes(_worker, args=(_free_port(), case), nprocs=case.get("world", 2),
                       start_method="spawn")


def _nccl_worker(rank, port):
    """One rank over NCCL (a one-rank communicator on this GPU): the device-
    tensor branch of every exchange (no host staging, in-place slot all-gather)
    against the oracle's step."""
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    torch.cuda.set_device(0)
    tdist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % port, rank=0,
                             world_size=1, device_id=torch.device("cuda", 0))
    import fsdp_sharded_mixed_zero_gb300 as Z
    import oracle
    import synth
    from fsdp_sharded_mixed_zero_gb300.dist import RankStep
    from tests.gpu_helpers import assert_params_close, assert_result, assert_state, f32, u16

    assert tdist.get_backend() == "nccl"
    full = 300_007
    kw = dict(lr=1e-3, window=2, initial_scale_power=10)
    flat = Z.ZeroFlat([(full,)], 1, F16, F16, AVG, Z.hparams(**kw))
    ohp = oracle.hparams(**kw)
    S = flat.shard_size
    step_of = RankStep(flat, 0, grad_dtype=F16)
    master = torch.empty(S, device="cuda")
    synth.normal_device(master, 43, synth.MASTER, 0, 0.02)
    m = torch.zeros(S, device="cuda")
    v = torch.zeros(S, device="cuda")
    out = torch.zeros(S, dtype=torch.float16, device="cuda")
    o_state = [[f32(master).copy()], [np.zeros(S, np.float32)], [np.zeros(S, np.float32)]]
    o_out = np.zeros(S, np.uint16)
    o_st = oracle.scaler_init(ohp)
    g = torch.empty((1, S), dtype=torch.float16, device="cuda")
    side = torch.cuda.Stream()
    for step in range(3):
        scale = flat.scaler_state().scale
        synth.grads_device(g, 43, step, 0, S, 1e-3, 1e-3, scale, synth.F16)
        if step == 1:
            g[0, 5] = float("inf")
        scale_used = o_st.scale
        ro = oracle.shard_step(ohp, o_st, 1, full, S, [0], u16(g), S, 0, *o_state, o_out)
        side.wait_stream(torch.cuda.current_stream())
        res = step_of.step(g.view(-1), master, m, v, out, stream=side)   # not the current stream
        side.synchronize()
        assert_result(res, (ro.overflow, ro.skipped, ro.grad_norm, ro.clip_coef, scale_used))
        assert flat.scaler_state().as_tuple() == o_st.as_tuple()
        assert_state(f32(master), f32(m), f32(v), *(x[0] for x in o_state), tag=" %d" % step)
        assert_params_close(u16(out), o_out, False, "flat buffer (step %d)" % step)
    assert o_st.overflow_count == 1
    flat.close()
    tdist.destroy_process_group()


def test_one_rank_over_nccl_matches_the_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    if not tdist.is_nccl_available():
        pytest.skip("no NCCL in this torch build")
    mp.start_processes(_nccl_worker, args=(_free_port(),), nprocs=1, start_method="spawn")


def _q8_worker(rank, port):
    """The ZeRO++ form: each rank writes only the int8 payload of its slot and
    the ranks all-gather codes and block scales (no 16-bit buffer)."""
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    torch.cuda.set_device(0)
    world = 2
    tdist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                             world_size=world)
    import fsdp_sharded_mixed_zero_gb300 as Z
    import oracle
    import synth
    from fsdp_sharded_mixed_zero_gb300.dist import RankStep
    from tests.gpu_helpers import assert_result, assert_state, f32, u16

    full, B = 600_001, 256
    kw = dict(lr=1e-3, window=3, initial_scale_power=12)
    flat = Z.ZeroFlat([(full,)], world, F16, F16, AVG, Z.hparams(**kw))
    ohp = oracle.hparams(**kw)
    S, padded = flat.shard_size, flat.padded_numel
    nb = -(-S // B)
    step_of = RankStep(flat, rank, grad_dtype=F16)
    master_all = torch.empty(padded, device="cuda")
    synth.normal_device(master_all, 45, synth.MASTER, 0, 0.02)
    master_all[full:].zero_()
    master = master_all[rank * S:(rank + 1) * S].clone()
    m = torch.zeros(S, device="cuda")
    v = torch.zeros(S, device="cuda")
    q8 = torch.zeros(padded, dtype=torch.int8, device="cuda")
    scales = torch.zeros(world * nb, device="cuda")
    o_state = [[f32(master_all[k * S:(k + 1) * S]).copy() for k in range(world)],
               [np.zeros(S, np.float32) for _ in range(world)],
               [np.zeros(S, np.float32) for _ in range(world)]]
    o_out = np.zeros(padded, np.uint16)
    o_st = oracle.scaler_init(ohp)
    mine = torch.empty((1, padded), dtype=torch.float16, device="cuda")
    everyone = torch.empty((world, padded), dtype=torch.float16, device="cuda")
    for step in range(STEPS):
        scale = flat.scaler_state().scale
        synth.grads_device(mine, 45, step, 0, padded, 1e-3, 1e-3, scale, synth.F16,
                           zero_from=full, c0=rank, n_contrib=1)
        synth.grads_device(everyone, 45, step, 0, padded, 1e-3, 1e-3, scale, synth.F16,
                           zero_from=full)
        if step == INF_STEP:
            everyone[1, 777] = float("inf")
            if rank == 1:
                mine[0, 777] = float("inf")
        scale_used = o_st.scale
        ro = oracle.shard_step(ohp, o_st, world, full, S, list(range(world)), u16(everyone),
                               padded, S, *o_state, o_out)
        res = step_of.step(mine.view(-1), master, m, v, None, q8=q8, q8_scales=scales)
        torch.cuda.synchronize()
        tag = " (rank %d, step %d)" % (rank, step)
        assert_result(res, (ro.overflow, ro.skipped, ro.grad_norm, ro.clip_coef, scale_used))
        assert_state(f32(master), f32(m), f32(v), o_state[0][rank], o_state[1][rank],
                     o_state[2][rank], tag=tag)
        got_q, got_s = q8.cpu().numpy(), scales.cpu().numpy()
        for k in range(world):                            # every rank's payload, gathered
            p = oracle.decode_array(np.ascontiguousarray(o_out[k * S:(k + 1) * S]))
            want_q, want_s = oracle.quantize_q8(p, B)
            assert np.array_equal(got_q[k * S:(k + 1) * S], want_q), "codes of rank %d" % k + tag
            assert np.array_equal(got_s[k * nb:(k + 1) * nb].view(np.uint32),
                                  want_s.view(np.uint32)), "scales of rank %d" % k + tag
    assert o_st.overflow_count == 1
    flat.close()
    tdist.destroy_process_group()


def test_two_ranks_exchange_the_int8_payload():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    mp.start_processes(_q8_worker, args=(_free_port(),), nprocs=2, start_method="spawn")


def _acc_worker(rank, port):
    """Micro-step accumulation among real ranks: per micro-step the all-to-all
    and zero_grad_accumulate of the received rows, then the step from the
    accumulator with one decision over both ranks -- against the oracle's
    accumulation and accumulated step of all shards at once."""
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    torch.cuda.set_device(0)
    world, K = 2, 2
    tdist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                             world_size=world)
    import fsdp_sharded_mixed_zero_gb300 as Z
    import oracle
    import synth
    from fsdp_sharded_mixed_zero_gb300.dist import RankStep
    from tests.gpu_helpers import assert_params_close, assert_result, assert_state, f32, u16

    full = 500_003
    kw = dict(lr=1e-3, window=3, initial_scale_power=12)
    flat = Z.ZeroFlat([(full,)], world, F16, F16, AVG, Z.hparams(**kw))
    ohp = oracle.hparams(**kw)
    S, padded = flat.shard_size, flat.padded_numel
    step_of = RankStep(flat, rank, grad_dtype=F16)
    master_all = torch.empty(padded, device="cuda")
    synth.normal_device(master_all, 47, synth.MASTER, 0, 0.02)
    master_all[full:].zero_()
    master = master_all[rank * S:(rank + 1) * S].clone()
    m = torch.zeros(S, device="cuda")
    v = torch.zeros(S, device="cuda")
    acc = torch.empty(S, device="cuda")
    out = torch.zeros(padded, dtype=torch.float16, device="cuda")
    o_state = [[f32(master_all[k * S:(k + 1) * S]).copy() for k in range(world)],
               [np.zeros(S, np.float32) for _ in range(world)],
               [np.zeros(S, np.float32) for _ in range(world)]]
    o_acc = [np.zeros(S, np.float32) for _ in range(world)]
    o_out = np.zeros(padded, np.uint16)
    o_st = oracle.scaler_init(ohp)
    mine = torch.empty((1, padded), dtype=torch.float16, device="cuda")
    everyone = torch.empty((world, padded), dtype=torch.float16, device="cuda")
    for step in range(3):
        scale = flat.scaler_state().scale
        for k in range(K):
            micro = K * step + k
            synth.grads_device(mine, 47, micro, 0, padded, 1e-3, 1e-3, scale, synth.F16,
                               zero_from=full, c0=rank, n_contrib=1)
            synth.grads_device(everyone, 47, micro, 0, padded, 1e-3, 1e-3, scale, synth.F16,
                               zero_from=full)
            if micro == 3:                    # rank 1's gradient, inside rank 0's slice
                everyone[1, 99] = float("inf")
                if rank == 1:
                    mine[0, 99] = float("inf")
            oracle.grad_accumulate(world, full, S, list(range(world)), u16(everyone), padded, S,
                                   o_acc, k == 0)
            step_of.accumulate(mine.view(-1), acc, k == 0)
        torch.cuda.synchronize()
        tag = " (rank %d, step %d)" % (rank, step)
        assert np.array_equal(f32(acc).view(np.uint32), o_acc[rank].view(np.uint32)), tag
        scale_used = o_st.scale
        ro = oracle.shard_step_acc(ohp, o_st, world, full, S, list(range(world)), o_acc,
                                   *o_state, o_out)
        res = step_of.step_accumulated(acc, master, m, v, out)
        torch.cuda.synchronize()
        assert_result(res, (ro.overflow, ro.skipped, ro.grad_norm, ro.clip_coef, scale_used))
        assert flat.scaler_state().as_tuple() == o_st.as_tuple(), tag
        assert_state(f32(master), f32(m), f32(v), o_state[0][rank], o_state[1][rank],
                     o_state[2][rank], tag=tag)
        assert_params_close(u16(out), o_out, False, "gathered flat buffer" + tag)
        assert res.skipped == (step == 1), tag
    flat.close()
    tdist.destroy_process_group()


def test_two_ranks_accumulate_micro_steps():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    mp.start_processes(_acc_worker, args=(_free_port(),), nprocs=2, start_method="spawn")
