"""The multi-rank step's exchanges on CPU ranks (gloo, 2 and 3 processes):

- the all-to-all of the reduce-scatter delivers, on rank r, slice r of every
  rank's gradient in contributor order, bit for bit for fp16, bf16 (every
  2-byte pattern) and fp32 contributions;
- the partials' all-gather delivers every rank's values in rank order;
- the slot all-gather leaves every rank with every owner's slot;
- the composition: every rank reduces the rows it received, the ranks
  exchange their exact squared-norm accumulators and take one decision, each
  updates its own shard and the slots are gathered -- with the oracle's own
  pieces as each rank's local arithmetic -- equals, bit for bit on every
  rank, the oracle's step of all shards at once on the stacked contributions
  (ZeRO computes what the unsharded step computes: ZeRO reading §5.2),
  including a step that one rank's inf makes every rank skip.
Each test runs as real processes (spawned) joined by a gloo group on
127.0.0.1."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as tdist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    tdist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                             world_size=world)


def _grad_of(c, padded, step=0):
    """Rank c's whole flat fp16 gradient at `step` (uint16 encodings)."""
    rng = np.random.default_rng(1000 * step + c)
    return (rng.standard_normal(padded) * 40.0).astype(np.float16).view(np.uint16)


def _exchange_worker(rank, world, port, S):
    _init(rank, world, port)
    from fsdp_sharded_mixed_zero_gb300 import dist as D
    padded = world * S
    mine = torch.from_numpy(_grad_of(rank, padded).view(np.int16).copy()).view(torch.float16)
    recv = torch.empty((world, S), dtype=torch.float16)
    D.exchange_contributions(mine, recv)
    got = recv.view(torch.int16).numpy().view(np.uint16)
    for c in range(world):
        assert np.array_equal(got[c], _grad_of(c, padded)[rank * S:(rank + 1) * S]), (rank, c)
    # bf16 contributions travel as the same 2-byte words (every bit pattern,
    # NaN payloads included), fp32 ones as they are
    bits = np.random.default_rng(77 + rank).integers(0, 1 << 16, padded, dtype=np.uint16)
    mine_b = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    recv_b = torch.empty((world, S), dtype=torch.bfloat16)
    D.exchange_contributions(mine_b, recv_b)
    got_b = recv_b.view(torch.int16).numpy().view(np.uint16)
    for c in range(world):
        want = np.random.default_rng(77 + c).integers(0, 1 << 16, padded, dtype=np.uint16)
        assert np.array_equal(got_b[c], want[rank * S:(rank + 1) * S]), ("bf16", rank, c)
    f32 = np.random.default_rng(99 + rank).standard_normal(padded).astype(np.float32)
    recv_f = torch.empty((world, S), dtype=torch.float32)
    D.exchange_contributions(torch.from_numpy(f32), recv_f)
    for c in range(world):
        want = np.random.default_rng(99 + c).standard_normal(padded).astype(np.float32)
        assert np.array_equal(recv_f[c].numpy().view(np.uint32),
                              want[rank * S:(rank + 1) * S].view(np.uint32)), ("f32", rank, c)
    ss = torch.tensor([rank + 0.25], dtype=torch.float64)
    of = torch.tensor([rank % 2], dtype=torch.int32)
    all_ss = torch.empty(world, dtype=torch.float64)
    all_of = torch.empty(world, dtype=torch.int32)
    D.gather_partials(ss, all_ss)
    D.gather_partials(of, all_of, name="of")
    assert all_ss.tolist() == [k + 0.25 for k in range(world)]
    assert all_of.tolist() == [k % 2 for k in range(world)]
    flat = torch.full((padded,), -1, dtype=torch.int16)
    flat[rank * S:(rank + 1) * S] = rank + 1
    D.gather_slots(flat, rank, S)
    assert flat.tolist() == sum([[k + 1] * S for k in range(world)], [])
    # the int8 payload: codes (1 byte) and block scales (fp32) per rank
    codes = torch.full((padded,), -1, dtype=torch.int8)
    codes[rank * S:(rank + 1) * S] = rank + 3
    D.gather_slots(codes, rank, S)
    assert codes.tolist() == sum([[k + 3] * S for k in range(world)], [])
    nb = -(-S // 256)
    scales = torch.full((world * nb,), -1.0)
    scales[rank * nb:(rank + 1) * nb] = rank + 0.5
    D.gather_slots(scales, rank, nb)
    assert scales.tolist() == sum([[k + 0.5] * nb for k in range(world)], [])
    # RankStep refuses a handle that does not fit the group (checked before
    # anything is allocated)
    from types import SimpleNamespace
    fake = SimpleNamespace(world_size=world, grad_dtype=0, shard_size=S)
    with pytest.raises(ValueError, match="grad dtype"):
        D.RankStep(fake, rank, grad_dtype=1)
    with pytest.raises(ValueError, match="sharded"):
        D.RankStep(SimpleNamespace(world_size=world + 1, grad_dtype=0, shard_size=S), rank)
    with pytest.raises(ValueError, match="out of range"):
        D.RankStep(fake, world)
    tdist.destroy_process_group()


@pytest.mark.parametrize("world,S", [(2, 1_001), (3, 4_096)])
def test_exchanges_on_gloo_ranks(world, S):
    mp.start_processes(_exchange_worker, args=(world, _free_port(), S), nprocs=world,
                       start_method="spawn")


def _oracle_rank_worker(rank, world, port, full):
    """Rank `rank`'s step with the oracle's pieces as local arithmetic, checked
    against the oracle's all-shards step."""
    _init(rank, world, port)
    import oracle
    from fsdp_sharded_mixed_zero_gb300 import dist as D
    full_, S, padded = oracle.layout([full], world)
    hp = oracle.hparams(lr=1e-3, window=2, initial_scale_power=4)
    rng = np.random.default_rng(5)
    theta = (rng.standard_normal(padded) * 0.02).astype(np.float32)
    theta[full:] = 0.0
    # this rank's state, and the reference: every shard stepped at once
    mine = [theta[rank * S:(rank + 1) * S].copy(), np.zeros(S, np.float32),
            np.zeros(S, np.float32)]
    flat = np.zeros(padded, np.uint16)
    st = oracle.scaler_init(hp)
    ref = [[theta[k * S:(k + 1) * S].copy() for k in range(world)],
           [np.zeros(S, np.float32) for _ in range(world)],
           [np.zeros(S, np.float32) for _ in range(world)]]
    ref_flat = np.zeros(padded, np.uint16)
    ref_st = oracle.scaler_init(hp)
    for step in range(4):
        grads = [_grad_of(c, padded, step) for c in range(world)]
        for c in range(world):
            grads[c][full:] = 0
        if step == 1:
            grads[world - 1][5] = 0x7C00                 # rank world-1's gradient, slice 0
        stacked = np.ascontiguousarray(np.stack(grads))
        r_ref = oracle.shard_step(hp, ref_st, world, full, S, list(range(world)), stacked,
                                  padded, S, *ref, ref_flat)
        # ---- the rank's own step
        send = torch.from_numpy(grads[rank].view(np.int16).copy()).view(torch.float16)
        recv = torch.empty((world, S), dtype=torch.float16)
        D.exchange_contributions(send, recv)
        rows = recv.view(torch.int16).numpy().view(np.uint16)
        scale_used = st.scale
        g = oracle.reduce_unscale(rows.reshape(-1), S, 0, world, S, rank * S, full, True,
                                  st.scale)
        acc, of = oracle.norm_accumulate(g)
        limbs = torch.from_numpy(np.frombuffer(bytes(acc), dtype=np.int64).copy())
        all_limbs = torch.empty(world * limbs.numel(), dtype=torch.int64)
        D.gather_partials(limbs, all_limbs, name="acc")
        all_of = torch.empty(world, dtype=torch.int32)
        D.gather_partials(torch.tensor([of], dtype=torch.int32), all_of, name="of")
        total = oracle.ExactAcc()
        for k in range(world):
            part = oracle.ExactAcc.from_buffer_copy(
                all_limbs[k * limbs.numel():(k + 1) * limbs.numel()].numpy().tobytes())
            oracle.acc_merge(total, part)
        any_of = int(all_of.max())
        norm = float(np.sqrt(oracle.norm_sum(total)))
        coef, skip = oracle.scaler_decide(hp, st, any_of, norm)
        if not skip:
            oracle.adamw_cast(hp, st.step_t, coef, g, *mine,
                              out=flat[rank * S:(rank + 1) * S])
        ft = torch.from_numpy(flat.view(np.int16))
        D.gather_slots(ft, rank, S)
        flat = ft.numpy().view(np.uint16)
        # ---- every rank equals the all-shards step
        assert (any_of, skip, coef, scale_used) == \
               (r_ref.overflow, r_ref.skipped, r_ref.clip_coef, r_ref.scale_used), step
        if not any_of:
            assert norm == r_ref.grad_norm
        assert st.as_tuple() == ref_st.as_tuple()
        for x, y in zip(mine, (ref[0][rank], ref[1][rank], ref[2][rank])):
            assert np.array_equal(x, y), (rank, step)
        assert np.array_equal(flat, ref_flat), (rank, step)
    assert st.overflow_count == 1 and st.step_t == 3
    tdist.destroy_process_group()


@pytest.mark.parametrize("world,full", [(2, 20_001), (3, 30_000)])
def test_rank_composition_equals_all_shards_step(world, full):
    mp.start_processes(_oracle_rank_worker, args=(world, _free_port(), full), nprocs=world,
                       start_method="spawn")
