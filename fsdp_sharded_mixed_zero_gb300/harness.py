"""Device-resident setup of a synthetic workload for the ZeRO shard step.

Allocates the gradient contributions, the per-rank fp32 master/m/v shards and
the flat 16-bit parameter buffer with PyTorch, fills them with the seeded
generator (synth), and steps them through the C ABI.  Plumbing only: every
step of the optimizer runs in libzero_gb300's kernels.
"""
import torch

import synth
from synth.workloads import Workload

from . import ZeroFlat, hparams

_TORCH_DTYPE = {0: torch.float16, 1: torch.bfloat16, 2: torch.float32}


class DeviceWorkload:
    def __init__(self, w: Workload, device="cuda", out_fill=None):
        self.w = w
        self.device = torch.device(device)
        hp = hparams(**w.hparams_kwargs())
        self.flat = ZeroFlat(w.shapes, w.world_size, w.grad_dtype, w.param_dtype, w.op, hp)
        self.S = self.flat.shard_size
        self.full = self.flat.full_numel
        self.padded = self.flat.padded_numel
        self.grads = torch.empty((w.world_size, w.grad_ld), dtype=_TORCH_DTYPE[w.grad_dtype],
                                 device=self.device)
        dt = _TORCH_DTYPE[w.param_dtype]
        self.master = [torch.empty(self.S, dtype=torch.float32, device=self.device)
                       for _ in w.ranks]
        self.m = [torch.zeros(self.S, dtype=torch.float32, device=self.device) for _ in w.ranks]
        self.v = [torch.zeros(self.S, dtype=torch.float32, device=self.device) for _ in w.ranks]
        self.out = torch.empty(self.padded, dtype=dt, device=self.device)
        if out_fill is None:
            self.out.zero_()
        else:
            self.out.view(torch.int16).fill_(out_fill)
        self.init_state()

    # ------------------------------------------------------------ inputs
    def valid_len(self, r):
        """Elements of rank r's shard that are real parameters (rest: padding)."""
        return max(0, min(self.S, self.full - r * self.S))

    def init_state(self):
        w = self.w
        for j, r in enumerate(w.ranks):
            first = r * self.S
            synth.normal_device(self.master[j], w.seed, synth.MASTER, first, w.sigma_master)
            if w.sigma_m > 0:
                synth.normal_device(self.m[j], w.seed, synth.MOMENT_M, first, w.sigma_m)
            if w.sigma_v > 0:
                synth.normal_device(self.v[j], w.seed, synth.MOMENT_V, first, w.sigma_v,
                                    absval=True)
            n = self.valid_len(r)
            for t in (self.master[j], self.m[j], self.v[j]):
                t[n:].zero_()                        # padding carries zeros

    def gen_grads(self, step, scale):
        """Contributions of `step`: fp16((g + n_c) * scale) or bf16(g + n_c)."""
        w = self.w
        dtype = {0: synth.F16, 1: synth.BF16, 2: synth.F32}[w.grad_dtype]
        if w.grads_layout == "full":
            synth.grads_device(self.grads, w.seed, step, 0, self.padded, w.sigma_g, w.sigma_n,
                               scale, dtype, zero_from=self.full)
        else:
            assert len(w.ranks) == 1
            r = w.ranks[0]
            synth.grads_device(self.grads, w.seed, step, r * self.S, self.S, w.sigma_g,
                               w.sigma_n, scale, dtype, zero_from=self.full)
        if w.inf_at is not None and w.inf_at[0] == step:
            _, c, i = w.inf_at
            col = i if w.grads_layout == "slice" else w.ranks[0] * self.S + i
            self.grads[c, col] = float("inf")

    # ------------------------------------------------------------ step
    def step(self, want_result=True, stream=None, extra_norm_sq=0.0):
        return self.flat.step(self.w.ranks, self.grads, self.master, self.m, self.v, self.out,
                              grad_rank_offset_mul=self.w.grad_rank_mul,
                              extra_norm_sq=extra_norm_sq, stream=stream,
                              want_result=want_result)

    # ------------------------------------------------------------ micro-steps
    def alloc_acc(self):
        """Per-rank fp32 accumulators, views of one contiguous buffer."""
        buf = torch.empty(len(self.w.ranks) * self.S, dtype=torch.float32, device=self.device)
        self.acc = [buf[j * self.S:(j + 1) * self.S] for j in range(len(self.w.ranks))]
        return self.acc

    def accumulate(self, first, stream=None):
        self.flat.accumulate(self.w.ranks, self.grads, self.acc, first,
                             grad_rank_offset_mul=self.w.grad_rank_mul, stream=stream)

    def step_accumulated(self, want_result=True, stream=None, extra_norm_sq=0.0):
        return self.flat.step_accumulated(self.w.ranks, self.acc, self.master, self.m, self.v,
                                          self.out, extra_norm_sq=extra_norm_sq, stream=stream,
                                          want_result=want_result)

    def scaler(self):
        return self.flat.scaler_state()

    def close(self):
        self.flat.close()
