"""One rank's ZeRO shard step in a process group: each process owns one rank's
shard, and the method's three cross-rank exchanges run as collectives of the
group (torch.distributed).

Per step, on rank r of N (shard size S, flat buffer of N*S elements):
  1. the exchange of the reduce-scatter ("PyTorch FSDP ... 深度解析" §3.3:
     every rank ends with the sum of every rank's gradient over its own
     slice; "DeepSpeed 与 FSDP" §ZeRO-2): an all-to-all sends slice k of this
     rank's full gradient to rank k and brings slice r of every rank's
     gradient here, rows in contributor order.  The sum itself is the
     library's reduce over those N rows (fp32, contributor order), so every
     rank gets exactly the sums of the single-GPU step; a collective's own
     reduction would add in fp16/bf16 or in an order of its own choosing.
  2. zero_shard_reduce: the reduced, unscaled gradient of the shard, and this
     rank's squared norm and overflow flag, in device memory.
  3. the two-scalar exchange (ZeRO reading §5.3: overflow detection and
     clipping are one decision over every rank's gradient): an all-gather of
     every rank's (norm^2, flag);
  4. zero_shard_apply_partials: the decision from all N partials, totalled on
     the device in one fixed order, so every rank takes the same skip / clip /
     loss-scale decision; AdamW and the cast into slot r of the flat buffer;
  5. the all-gather of the 16-bit slots ("DeepSpeed 与 FSDP" §ZeRO-1 step 3;
     "PyTorch FSDP ... 深度解析" §3.2): every rank's flat buffer holds every
     rank's new parameters -- or, in the ZeRO++ form ("DeepSpeed 与 FSDP"
     §ZeRO++; ZeRO reading §4.2), the all-gather of every rank's int8 codes
     and block scales, half the bytes of the 16-bit slots.

The collectives are the process group's (NCCL moves device tensors; a gloo
group moves host tensors, so the step stages its buffers through pinned host
memory).  Every step of the optimizer runs in the library's kernels; this
module moves bytes and passes pointers.
"""
import torch
import torch.distributed as dist

from . import ZERO_BF16, ZERO_F16, ZERO_F32

_TORCH_DTYPE = {ZERO_F16: torch.float16, ZERO_BF16: torch.bfloat16, ZERO_F32: torch.float32}


def _stages_on_host(t, group):
    return t.is_cuda and dist.get_backend(group) == "gloo"


def _wire(t):
    """The tensor as the collectives move it: no collective here does any
    arithmetic, so every 2-byte encoding travels as float16 bits (a type
    every backend moves)."""
    return t.view(torch.float16) if t.element_size() == 2 else t


class _Staging:
    """Pinned host twins of device buffers, for groups whose collectives take
    host tensors."""

    def __init__(self):
        self.bufs = {}

    def host(self, name, like):
        b = self.bufs.get(name)
        if b is None or b.shape != like.shape or b.dtype != like.dtype:
            b = torch.empty(like.shape, dtype=like.dtype, pin_memory=True)
            self.bufs[name] = b
        return b


def exchange_contributions(grads, recv, group=None, staging=None):
    """The all-to-all of the reduce-scatter: grads holds this rank's whole
    flat gradient (N*S elements, slice k at [k*S, (k+1)*S)); recv ([N, S],
    contiguous) receives slice `rank` of rank c's gradient in row c."""
    send, out = _wire(grads.reshape(-1)), _wire(recv.reshape(-1))
    assert send.numel() == out.numel()
    if _stages_on_host(out, group):
        staging = staging or _Staging()
        hs, hr = staging.host("send", send), staging.host("recv", out)
        hs.copy_(send)
        dist.all_to_all_single(hr, hs, group=group)
        out.copy_(hr)
    else:
        dist.all_to_all_single(out, send, group=group)


def gather_partials(mine, everyone, group=None, staging=None, name="part"):
    """All-gather of one small tensor per rank, in rank order."""
    if _stages_on_host(mine, group):
        staging = staging or _Staging()
        hm, he = staging.host(name + "_mine", mine), staging.host(name + "_all", everyone)
        hm.copy_(mine)
        dist.all_gather_into_tensor(he, hm, group=group)
        everyone.copy_(he)
    else:
        dist.all_gather_into_tensor(everyone, mine, group=group)


def gather_slots(flat, rank, shard_size, group=None, staging=None):
    """The all-gather of the parameter slots: slot k of every rank's flat
    buffer ends up equal to rank k's."""
    flat = _wire(flat)
    slot = flat[rank * shard_size:(rank + 1) * shard_size]
    if _stages_on_host(flat, group):
        staging = staging or _Staging()
        tag = "%s_%d" % (flat.dtype, flat.numel())
        hs, hf = staging.host("slot_" + tag, slot), staging.host("flat_" + tag, flat)
        hs.copy_(slot)
        dist.all_gather_into_tensor(hf, hs, group=group)
        flat.copy_(hf)
    elif flat.is_cuda:
        dist.all_gather_into_tensor(flat, slot, group=group)     # in place
    else:
        dist.all_gather_into_tensor(flat, slot.clone(), group=group)


class RankStep:
    """The ZeRO step of rank `rank` of a process group whose size is the
    handle's world size.  flat: a ZeroFlat of the FlatParameter (world size N,
    grad dtype, op and hyper-parameters as every other rank's); grad_dtype,
    if given, must be the handle's."""

    def __init__(self, flat, rank, grad_dtype=None, group=None, device=None):
        n = dist.get_world_size(group)
        if n != flat.world_size:
            raise ValueError("process group of %d ranks for a FlatParameter sharded %d ways"
                             % (n, flat.world_size))
        if not 0 <= rank < n:
            raise ValueError("rank %d out of range" % rank)
        if grad_dtype is None:
            grad_dtype = flat.grad_dtype
        elif grad_dtype != flat.grad_dtype:
            raise ValueError("grad dtype %d differs from the handle's (%d)"
                             % (grad_dtype, flat.grad_dtype))
        self.flat, self.rank, self.group = flat, rank, group
        self.N, self.S = n, flat.shard_size
        dev = torch.device(device) if device is not None else torch.device("cuda")
        self.recv = torch.empty((n, self.S), dtype=_TORCH_DTYPE[grad_dtype], device=dev)
        self.norm_sq = torch.zeros(1, dtype=torch.float64, device=dev)
        self.overflow = torch.zeros(1, dtype=torch.int32, device=dev)
        self.all_norm_sq = torch.zeros(n, dtype=torch.float64, device=dev)
        self.all_overflow = torch.zeros(n, dtype=torch.int32, device=dev)
        self.staging = _Staging()

    def accumulate(self, grads, acc, first_micro_step, stream=None):
        """One micro-step ("DeepSpeed 与 FSDP" §实践要点, gradient
        accumulation): the all-to-all of this micro-step's gradient slices,
        then zero_grad_accumulate of the N received rows into this rank's
        fp32 accumulator (acc = r on the first micro-step, acc += r after)."""
        stream = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(stream):
            exchange_contributions(grads, self.recv, self.group, self.staging)
            self.flat.accumulate([self.rank], self.recv, [acc], first_micro_step,
                                 grad_rank_offset_mul=0, stream=stream)

    def step_accumulated(self, acc, master, m, v, out, stream=None, want_result=True,
                         gather=True):
        """The optimizer step from the accumulator: this rank's norm^2 and flag
        (zero_shard_reduce_accumulated), their all-gather, the one decision
        (zero_shard_apply_partials), AdamW and the slot all-gather."""
        stream = stream if stream is not None else torch.cuda.current_stream()
        r = [self.rank]
        with torch.cuda.stream(stream):
            self.flat.reduce_accumulated(r, [acc], self.norm_sq, self.overflow, stream=stream)
            gather_partials(self.norm_sq, self.all_norm_sq, self.group, self.staging, "ss")
            gather_partials(self.overflow, self.all_overflow, self.group, self.staging, "of")
            res = self.flat.apply_partials(r, [master], [m], [v], out, self.all_norm_sq,
                                           self.all_overflow, stream=stream,
                                           want_result=want_result)
            if gather:
                gather_slots(out, self.rank, self.S, self.group, self.staging)
        return res

    def step(self, grads, master, m, v, out, stream=None, want_result=True, gather=True,
             q8=None, q8_scales=None):
        """grads: this rank's whole flat gradient (padded_numel elements of the
        grad dtype); master, m, v: this rank's fp32 shard (S elements each);
        out: the flat 16-bit parameter buffer (padded_numel elements), slot
        `rank` written by the update and, with gather, every slot refreshed
        from its owner.  q8, q8_scales: the int8 weight payload (int8
        codes, padded_numel; fp32 block scales, world_size * ceil(S/256)),
        written for this rank as zero_shard_step_q8 writes it and, with
        gather, all-gathered; out may then be None (only the payload is
        written and exchanged).  stream: the CUDA stream every part of the
        step runs on -- the library's kernels, the collectives and the
        staging copies (None: the current stream).  Returns the step result
        (want_result) or None."""
        stream = stream if stream is not None else torch.cuda.current_stream()
        r = [self.rank]
        with torch.cuda.stream(stream):
            exchange_contributions(grads, self.recv, self.group, self.staging)
            self.flat.reduce(r, self.recv, self.norm_sq, self.overflow, grad_rank_offset_mul=0,
                             stream=stream)
            gather_partials(self.norm_sq, self.all_norm_sq, self.group, self.staging, "ss")
            gather_partials(self.overflow, self.all_overflow, self.group, self.staging, "of")
            res = self.flat.apply_partials(r, [master], [m], [v], out, self.all_norm_sq,
                                           self.all_overflow, stream=stream,
                                           want_result=want_result, q8=q8, q8_scales=q8_scales)
            if gather:
                if out is not None:
                    gather_slots(out, self.rank, self.S, self.group, self.staging)
                if q8 is not None:
                    nb = -(-self.S // 256)
                    gather_slots(q8, self.rank, self.S, self.group, self.staging)
                    gather_slots(q8_scales, self.rank, nb, self.group, self.staging)
        return res
