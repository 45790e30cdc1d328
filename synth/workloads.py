"""The five synthetic workloads of the ZeRO shard step: parameter tables,
sharding, dtypes and input distributions.  No optimizer arithmetic here.

Shapes follow the pages' examples: a tiny 2-layer MLP; a GPT-2-small flat
buffer wrapped one FSDP unit per transformer block ("PyTorch FSDP ...
深度解析" §7.1, transformer auto-wrap); the 1.5B GPT-like model of the ZeRO
reading §1 at its 64-way example (§3.1); a 7B Llama-shaped model ("DeepSpeed
与 FSDP", FSDP usage example loads Llama-2-7b); the 10B model on 8 GPUs of
"DeepSpeed 与 FSDP" §逐步推导 / §ZeRO-1.  All values are synthetic (no data,
no weights): see each field for the distribution.
"""
from dataclasses import dataclass, field
from typing import List, Optional, Tuple

F16, BF16, F32 = 0, 1, 2
SUM, AVG = 0, 1


def gpt2_shapes(d, n_layer, vocab, ctx, ff=None):
    """GPT-2 parameter list in module order (wte, wpe, blocks, ln_f)."""
    ff = ff or 4 * d
    shapes = [(vocab, d), (ctx, d)]
    for _ in range(n_layer):
        shapes += [(d,), (d,),                 # ln_1 weight, bias
                   (d, 3 * d), (3 * d,),       # attn c_attn
                   (d, d), (d,),               # attn c_proj
                   (d,), (d,),                 # ln_2
                   (d, ff), (ff,),             # mlp c_fc
                   (ff, d), (d,)]              # mlp c_proj
    shapes += [(d,), (d,)]                     # ln_f
    return shapes


def llama_shapes(d, n_layer, ff, vocab):
    """Llama parameter list (untied output head)."""
    shapes = [(vocab, d)]
    for _ in range(n_layer):
        shapes += [(d, d), (d, d), (d, d), (d, d),     # q, k, v, o
                   (ff, d), (ff, d), (d, ff),           # gate, up, down
                   (d,), (d,)]                          # input / post-attn norms
    shapes += [(d,), (vocab, d)]
    return shapes


def numel_of(shapes):
    total = 0
    for s in shapes:
        n = 1
        for d in s:
            n *= d
        total += n
    return total


@dataclass
class Workload:
    name: str
    description: str
    shapes: List[Tuple[int, ...]]
    world_size: int
    ranks: List[int]                 # stepped ranks
    grad_dtype: int
    op: int
    dynamic: bool
    steps: int
    sigma_g: float                   # shared gradient g ~ N(0, sigma_g)
    sigma_n: float                   # per-rank noise n_c ~ N(0, sigma_n)
    sigma_master: float = 0.02       # fp32 master ~ N(0, 0.02)
    sigma_m: float = 0.0             # warm m ~ N(0, sigma_m) (0: cold, m = 0)
    sigma_v: float = 0.0             # warm v = |N(0, sigma_v)| (0: cold, v = 0)
    warm_steps: int = 0              # untimed steps before the measured ones
    seed: int = 0
    inf_at: Optional[Tuple[int, int, int]] = None   # (step, contributor, shard index): +inf
    hp: dict = field(default_factory=dict)
    grads_layout: str = "full"       # "full": [N, padded], mul = S; "slice": [N, ld], mul = 0
    micro_steps: int = 1             # >1: contributions accumulated over micro-steps per step
    pdtype: Optional[int] = None     # parameter dtype if it differs from the default below

    @property
    def param_dtype(self):
        """16-bit parameter dtype (the grad dtype, or fp16 under fp32 contributions)."""
        if self.pdtype is not None:
            return self.pdtype
        return self.grad_dtype if self.grad_dtype in (F16, BF16) else F16

    @property
    def full_numel(self):
        return numel_of(self.shapes)

    @property
    def shard_size(self):
        n = self.full_numel
        return -(-n // self.world_size)

    @property
    def padded_numel(self):
        return self.shard_size * self.world_size

    @property
    def grad_ld(self):
        if self.grads_layout == "full":
            return self.padded_numel
        return -(-self.shard_size // 8) * 8          # rows padded to 16 (fp32: 32) bytes

    @property
    def grad_rank_mul(self):
        return self.shard_size if self.grads_layout == "full" else 0

    @property
    def initial_scale(self):
        return float(2 ** self.hp.get("initial_scale_power", 16)) if self.dynamic else \
            float(self.hp.get("static_scale", 1.0))

    def hparams_kwargs(self):
        kw = dict(lr=3e-5, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
                  max_grad_norm=1.0, dynamic=self.dynamic, initial_scale_power=16,
                  window=1000, static_scale=1.0, min_scale=1.0)
        kw.update(self.hp)
        return kw


TINY = Workload(
    name="tiny_mlp", description="2-layer MLP FlatParameter [512x1024, 1024, 1024x512, 512], "
    "N=4 emulated ranks, all 4 shards stepped, fp16 AVG, dynamic loss scale 2^16",
    shapes=[(512, 1024), (1024,), (1024, 512), (512,)], world_size=4, ranks=[0, 1, 2, 3],
    grad_dtype=F16, op=AVG, dynamic=True, steps=5, sigma_g=1e-3, sigma_n=1e-3, seed=0)

GPT2 = Workload(
    name="gpt2_small", description="GPT-2-small flat buffer (124,439,808 params, 148 tensors, "
    "12 FSDP units), N=8 emulated ranks, all shards stepped, bf16 SUM, no loss scaling, "
    "clipping active, warm m/v",
    shapes=gpt2_shapes(768, 12, 50257, 1024), world_size=8, ranks=list(range(8)),
    grad_dtype=BF16, op=SUM, dynamic=False, steps=20, sigma_g=1e-4, sigma_n=1e-4,
    sigma_m=1e-5, sigma_v=1e-8, seed=1)

GPT_1P5B = Workload(
    name="gpt_1p5b_rank17", description="1.5B GPT-like (d=1600, 48 layers, 580 tensors) "
    "flattened, N=64, rank 17's shard only (24,337,675 params), fp16 AVG, dynamic loss "
    "scale 2^16 window 1000, +inf injected at step 3",
    shapes=gpt2_shapes(1600, 48, 50257, 1024), world_size=64, ranks=[17], grad_dtype=F16,
    op=AVG, dynamic=True, steps=10, sigma_g=1e-3, sigma_n=1e-3, seed=2,
    inf_at=(3, 5, 12345), grads_layout="slice")

LLAMA_7B = Workload(
    name="llama_7b_rank0", description="7B Llama-shaped (d=4096, 32 layers, ff=11008, "
    "vocab 32000, 291 tensors) flattened, N=8, rank 0's shard (842,301,952 params), "
    "fp16 AVG at loss scale 2^16, warm m/v from one prior step",
    shapes=llama_shapes(4096, 32, 11008, 32000), world_size=8, ranks=[0], grad_dtype=F16,
    op=AVG, dynamic=True, steps=5, warm_steps=1, sigma_g=5e-4, sigma_n=5e-4, seed=3,
    grads_layout="slice")

TEN_B = Workload(
    name="10b_rank7", description="10B params in one flat buffer, N=8, rank 7's shard "
    "(1.25e9 params, 15 GB fp32 master/m/v), fp16 AVG at loss scale 2^16, param shard "
    "written into a 20 GB flat buffer at the rank's offset",
    shapes=[(10_000_000_000,)], world_size=8, ranks=[7], grad_dtype=F16, op=AVG,
    dynamic=True, steps=5, sigma_g=2e-4, sigma_n=2e-4, seed=4, grads_layout="slice")

# A smaller case of the 10B rank-7 step (same kernels and launch shape, ~5 GB
# resident: still far larger than L2) for hardware-counter captures.
FLAT_800M = Workload(
    name="flat800m_rank7", description="800M params in one flat buffer, N=8, rank 7's shard "
    "(1e8 params), fp16 AVG at loss scale 2^16 (profiling size of the 10B step)",
    shapes=[(800_000_000,)], world_size=8, ranks=[7], grad_dtype=F16, op=AVG, dynamic=True,
    steps=5, sigma_g=2e-4, sigma_n=2e-4, seed=5, grads_layout="slice")

# The profiling case with an odd shard size in the full [N, padded] layout:
# rank 7's slice of every contributor row starts 2-byte aligned, so the
# reduce takes the staged (bulk-copy) kernel; ~3 GB resident.
FLAT_800M_ODD = Workload(
    name="flat800m_odd_rank7", description="800M + 8 params in one flat buffer, N=8, rank 7's "
    "shard (100,000,001 params) in the full contributor layout (2-byte aligned slices), fp16 AVG "
    "at loss scale 2^16 (profiling size of the staged reduce)",
    shapes=[(800_000_008,)], world_size=8, ranks=[7], grad_dtype=F16, op=AVG, dynamic=True,
    steps=5, sigma_g=2e-4, sigma_n=2e-4, seed=5, grads_layout="full")

# The 10B rank-7 step with fp32 contributions (reduce_dtype=float32): 40 GB of
# contributions, fp16 parameters.
TEN_B_F32 = Workload(
    name="10b_rank7_fp32", description="10B params, N=8, rank 7's shard, fp32 contributions "
    "(reduce_dtype=float32), fp16 params, dynamic loss scale 2^16",
    shapes=[(10_000_000_000,)], world_size=8, ranks=[7], grad_dtype=F32, op=AVG,
    dynamic=True, steps=5, sigma_g=2e-4, sigma_n=2e-4, seed=6, grads_layout="slice")

ALL = [TINY, GPT2, GPT_1P5B, LLAMA_7B, TEN_B]
EXTRA = [FLAT_800M, FLAT_800M_ODD, TEN_B_F32]
BY_NAME = {w.name: w for w in ALL + EXTRA}
