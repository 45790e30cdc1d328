#!/usr/bin/env python
"""Benchmark of the ZeRO shard optimizer step on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

One step = one zero_shard_step call on the workload's stepped shard(s): the
N-way gradient reduce + unscale + overflow check + global norm, the
loss-scale / clip decision, and AdamW + cast into the flat buffer.  The
default workload is the 10B FlatParameter's rank-7 shard (1.25e9 params,
8 fp16 contributions, 60 GB resident).  Prints one JSON line on rank 0.

value: Gparams/s stepped, device-timed (CUDA events on the step's stream)
over K steps with inputs resident in HBM; the working set (tens of GB) is
far larger than L2, so no flush is needed between steps.
e2e: the same metric through the public API with the contributions in pinned
host memory (read over the host link every step) and the step result read
back every step; the explicit copy-then-step time is reported beside it.
roofline: the dominant kernel's algorithmic bytes per launch over its mean
event-timed duration, against the measured HBM copy peak.
cpu_baseline: the oracle (plain single-threaded C) on a bounded sample of the
same workload, timed on this host.
workloads (default workload, N = 1): the tiny MLP, GPT-2-small, 1.5B and 7B
configs' steps measured in the same run, each with its kernels' achieved GB/s
and its dominant kernel's fraction of the measured copy peak.
--impl reference: the oracle on the host cores as the reference arm.
--offload: the ZeRO-Offload step instead (zero_shard_step_offload: reduce and
decision on the GPU, AdamW over host-resident fp32 state on the host cores),
its own JSON line with the per-phase times and the host update against the
host copy bandwidth measured in the same run.
--collective: the rank step among real processes (RankStep over NCCL: the
all-to-all of the gradient slices, the reduce, the all-gather of every rank's
norm^2 and overflow flag, AdamW, the all-gather of the 16-bit slots), one
rank per GPU under torchrun, weak scaling.
Otherwise, under torchrun each rank runs an independent replica (weak scaling).
"""
import argparse
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ZeRO shard AdamW step Gparams/s; achieved HBM GB/s as % of GB300 peak"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
RESULT_D2H_BYTES = 64            # the device state block read back with the result


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default="10b_rank7")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--e2e-steps", type=int, default=5)
    p.add_argument("--graph", action="store_true",
                   help="capture one step in a CUDA graph and replay it (no per-kernel split)")
    p.add_argument("--q8", action="store_true",
                   help="also write the int8 all-gather payload (zero_shard_step_q8)")
    p.add_argument("--micro-steps", type=int, default=1,
                   help="K > 1: each step accumulates K micro-steps' contributions into an "
                        "fp32 shard (zero_grad_accumulate) and steps from it "
                        "(zero_shard_step_accumulated)")
    p.add_argument("--offload", action="store_true",
                   help="time the ZeRO-Offload step (optimizer on the host cores)")
    p.add_argument("--offload-threads", type=int, default=0,
                   help="host threads of the offload update (0: every available CPU)")
    p.add_argument("--offload-gpu-share", type=float, default=0.0,
                   help="fraction of each shard the GPU updates over the host link")
    p.add_argument("--group", type=int, default=0,
                   help="time a group of this many FlatParameters (one rank's shard each) "
                        "stepped with one global decision, against per-FlatParameter steps")
    p.add_argument("--group-params", type=int, default=1_000_000,
                   help="params in each group member's shard")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the other configs' steps (tiny_mlp, gpt2_small, gpt_1p5b_rank17, "
                        "llama_7b_rank0) reported beside the headline workload")
    p.add_argument("--workload-steps", type=int, default=20,
                   help="timed steps of each of those configs")
    p.add_argument("--collective", action="store_true",
                   help="time the rank step among real processes (RankStep over NCCL, one "
                        "rank per GPU under torchrun) instead of the single-GPU emulation")
    p.add_argument("--collective-shard", type=int, default=1_250_000_000,
                   help="params in each rank's shard for --collective (weak scaling)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target length of the oracle's timed sample")
    p.add_argument("--ref-seconds", type=float, default=120.0,
                   help="target length of the whole --impl reference run")
    args = p.parse_args(argv)
    if bool(args.q8) + (args.micro_steps > 1) + bool(args.offload) + bool(args.collective) > 1:
        p.error("--q8, --micro-steps K > 1, --offload and --collective exclude one another")
    return args


# ---------------------------------------------------------------- plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class RankGroup:
    """The ranks of a torchrun launch (one process per GPU): rendezvous from
    RANK / WORLD_SIZE / MASTER_ADDR / MASTER_PORT, a barrier, and the maximum
    of a host value over ranks.  Each rank runs an independent replica of the
    step; nothing on the data path is exchanged.  backend: "nccl" for GPU
    ranks, "gloo" for CPU ranks."""

    def __init__(self, backend=None, device=None):
        self.world, self.rank, self.local = dist_env()
        self.device = device
        self.dist = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            if backend is None:
                backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend=backend)
            self.dist = dist

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, x):
        if self.dist is None:
            return float(x)
        import torch
        t = torch.tensor([float(x)], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()
            self.dist = None


def whole_job_value(params_per_rank, steps, world, max_elapsed_ms):
    """Gparams/s of the whole job: every rank's stepped parameters over the
    slowest rank's time."""
    return params_per_rank * steps * world / (max_elapsed_ms / 1e3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha():
    """Hash of the kernels' code (comments and blank lines left out, so that a
    comment edit does not void the profiles taken on the same code)."""
    h = hashlib.sha256()
    for name in ("zero_kernels.cu", "zero_kernels.cuh"):
        with open(os.path.join(ROOT, "fsdp_sharded_mixed_zero_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())
        h.update(code.encode())
    return h.hexdigest()[:16]


def reduce_name(flat):
    """The name of the reduce kernel the handle's last contribution reduce
    launched (the planner stages misaligned rows and large launches)."""
    return "reduce_staged_kernel" if flat.reduce_form() == "staged" else "reduce_kernel"


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (kernel, workload))
    if not os.path.exists(path):
        return None
    text = open(path).read()
    sha = re.search(r"kernel_source_sha:\s*(\w+)", text)
    tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not sha or not tr or sha.group(1) != kernel_source_sha():
        return None
    return float(tr.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for name, val in zip(self.NAMES, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- CPU baseline
def oracle_sample_step(w, k):
    """Host inputs for one oracle step on k params of the workload's first
    stepped shard (same flat indices, distributions and contributor count)."""
    import numpy as np

    import oracle
    import synth
    r = w.ranks[0]
    S = w.shard_size
    first = r * S
    k = min(k, S)
    scale = w.initial_scale if w.dynamic else 1.0
    dtype = synth.BF16 if w.grad_dtype == 1 else synth.F16
    g = synth.grads_host(w.seed, 0, w.world_size, first, k, w.sigma_g, w.sigma_n, scale, dtype,
                         zero_from=w.full_numel)
    g = np.ascontiguousarray(g)
    master = synth.normal_host(w.seed, synth.MASTER, first, k, w.sigma_master)
    m = (synth.normal_host(w.seed, synth.MOMENT_M, first, k, w.sigma_m) if w.sigma_m
         else np.zeros(k, np.float32))
    v = (synth.normal_host(w.seed, synth.MOMENT_V, first, k, w.sigma_v, absval=True)
         if w.sigma_v else np.zeros(k, np.float32))
    out = np.zeros(k, np.uint16)
    hp = oracle.hparams(**w.hparams_kwargs())
    st = oracle.scaler_init(hp)

    def run():
        # one shard of k params, N contributions of k elements each
        return oracle.shard_step(hp, st, w.world_size, k * w.world_size, k, [0], g, k, 0,
                                 [master], [m], [v], out, avg=w.op == 1,
                                 grad_is_bf16=w.grad_dtype == 1,
                                 param_is_bf16=w.grad_dtype == 1)
    return run, k


_ARM_PARTS = {0xd40: "Neoverse-V1", 0xd49: "Neoverse-N2", 0xd4f: "Neoverse-V2",
              0xd84: "Neoverse-V3", 0xd0c: "Neoverse-N1"}


def host_cpu(cpuinfo=None):
    """The host's CPU model (from /proc/cpuinfo, or the text `cpuinfo`: "model
    name" where the kernel gives one, else the Arm implementer/part pair), its
    online CPU count and the CPUs this process may run on."""
    model, impl, part = None, None, None
    try:
        if cpuinfo is None:
            with open("/proc/cpuinfo") as f:
                cpuinfo = f.read()
        for line in cpuinfo.splitlines():
            k, _, v = line.partition(":")
            k, v = k.strip(), v.strip()
            if k == "model name" and model is None:
                model = v
            elif k == "CPU implementer" and impl is None:
                impl = v
            elif k == "CPU part" and part is None:
                part = v
    except OSError:
        pass
    if model is None and part is not None:
        try:
            name = _ARM_PARTS.get(int(part, 16))
        except ValueError:
            name = None
        model = ("Arm " + name) if impl == "0x41" and name else \
            "implementer %s part %s" % (impl, part)
    try:
        usable = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        usable = os.cpu_count()
    return {"cpu_model": model or platform.processor() or platform.machine(),
            "nproc": os.cpu_count(), "usable_cpus": usable}


def cpu_baseline(w, target_s):
    run, k0 = oracle_sample_step(w, 1 << 20)
    t = time.perf_counter()
    run()
    t0 = time.perf_counter() - t
    k = int(min(w.shard_size, 192 << 20, max(k0, k0 * target_s / max(t0, 1e-6))))
    run, k = oracle_sample_step(w, k)
    t = time.perf_counter()
    run()
    dt = time.perf_counter() - t
    return {"value": k / dt / 1e9, "unit": "Gparams/s", "cores": 1, "kind": "oracle",
            "sample": "%d params of the %s shard (%d fp16/bf16 contributions each), one full "
                      "oracle step (reduce, norm, decision, AdamW, cast), single thread, "
                      "%.1f s" % (k, w.name, w.world_size, dt), "host": host_cpu()}


# ---------------------------------------------------------------- arms
def run_collective(args):
    """The rank step among real processes: each rank (one process per GPU,
    NCCL) steps its own shard of an N-rank FlatParameter with RankStep -- the
    all-to-all of the gradient slices, the fp32 reduce over the N received
    rows, the all-gather of every rank's norm^2 and overflow flag, the
    decision, AdamW, and the all-gather of the 16-bit slots.  Weak scaling:
    every rank's shard holds --collective-shard params (the 10B config's 1.25e9
    by default), so the model is N times that; each rank generates its own
    contribution (the whole flat fp16 gradient of N shards)."""
    import torch
    import torch.distributed as dist

    import fsdp_sharded_mixed_zero_gb300 as Z
    import synth
    from fsdp_sharded_mixed_zero_gb300.dist import RankStep

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init = rendezvous_method(os.environ, world)
    if init == "env://":
        dist.init_process_group("nccl", device_id=dev)
    else:
        dist.init_process_group("nccl", init_method=init, rank=0, world_size=1, device_id=dev)
    S = args.collective_shard
    full = S * world
    flat = Z.ZeroFlat([(full,)], world, Z.ZERO_F16, Z.ZERO_F16, Z.ZERO_AVG, Z.hparams())
    stream = torch.cuda.current_stream(dev)
    scale = flat.scaler_state().scale
    grads = torch.empty((1, full), dtype=torch.float16, device=dev)
    synth.grads_device(grads, 11, 0, 0, full, 2e-4, 2e-4, scale, synth.F16, c0=rank, n_contrib=1)
    master = torch.empty(S, device=dev)
    synth.normal_device(master, 11, synth.MASTER, rank * S, 0.02)
    m = torch.zeros(S, device=dev)
    v = torch.zeros(S, device=dev)
    out = torch.zeros(full, dtype=torch.float16, device=dev)
    step = RankStep(flat, rank, grad_dtype=Z.ZERO_F16, device=dev)
    for _ in range(args.warmup):
        step.step(grads.view(-1), master, m, v, out, stream=stream, want_result=False)
    dist.barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step.step(grads.view(-1), master, m, v, out, stream=stream, want_result=False)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    t = torch.tensor([e0.elapsed_time(e1)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    elapsed_ms = float(t.item())
    res = step.step(grads.view(-1), master, m, v, out, stream=stream, want_result=True)
    assert res.skipped == 0 and res.overflow == 0, "benchmark inputs overflowed"
    line = None
    if rank == 0:
        line = json.dumps({
            "metric": METRIC, "value": whole_job_value(S, args.steps, world, elapsed_ms),
            "unit": "Gparams/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "rank_step_%d_params_per_rank" % S,
                       "params_stepped_per_gpu": S, "world_size": world,
                       "storage": "f16 grads, f16 params, f32 master/m/v",
                       "exchanges": "NCCL all-to-all of 16-bit slices, all-gather of "
                                    "(norm^2, flag), all-gather of 16-bit slots",
                       "parallelism": "zero%d" % world},
            # per step: the reduce, the decision, AdamW (the NCCL kernels are not ours)
            "gpu_launches": 3 * args.steps})
    flat.close()
    dist.destroy_process_group()
    if line is not None:                 # after the library's own messages: the last line
        print(line, flush=True)


def rendezvous_method(env, world):
    """How a rank finds the others: the launcher's store ("env://") whenever
    torchrun started the process -- even for one rank, since under its agent
    a tcp:// address makes every rank a client of a store that nobody serves
    -- else, for a single process started directly, a private store on a free
    local port."""
    if world > 1 or ("MASTER_ADDR" in env and "MASTER_PORT" in env):
        return "env://"
    return "tcp://127.0.0.1:%d" % _free_port()


def _free_port():
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    k = None
    times = []
    for i in range(args.warmup + args.steps):
        if k is None:
            run, k0 = oracle_sample_step(w, 1 << 20)
            t = time.perf_counter()
            run()
            t0 = time.perf_counter() - t
            per_step = max(0.05, min(5.0, args.ref_seconds / max(1, args.warmup + args.steps)))
            k = int(min(w.shard_size, max(k0, k0 * per_step / max(t0, 1e-6))))
            run, k = oracle_sample_step(w, k)
        t = time.perf_counter()
        run()
        if i >= args.warmup:
            times.append(time.perf_counter() - t)
    total = sum(times)
    value = k * len(times) / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "Gparams/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "sample_params_per_step": k},
        "cpu_baseline": {"value": value, "unit": "Gparams/s", "cores": 1, "kind": "oracle",
                         "sample": "%d params of the %s shard per step, single thread" %
                                   (k, w.name), "host": host_cpu()},
        "e2e": {"value": value, "unit": "Gparams/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, w):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    group = RankGroup(backend="nccl", device=dev)
    barrier, max_over_ranks = group.barrier, group.max

    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload

    dw = DeviceWorkload(w, device=dev)
    dw.gen_grads(0, dw.scaler().scale)
    stream = torch.cuda.current_stream(dev)
    params = dw.S * len(w.ranks)
    n_batches = -(-len(w.ranks) // 64)
    K = max(1, args.micro_steps)
    # the reduce launches (the last block makes the decision), the AdamW launches,
    # and with micro-steps the accumulate launches
    launches_per_step = 2 * n_batches + (K * n_batches if K > 1 else 0)
    acc_events = []
    if K > 1:
        dw.alloc_acc()
    q8 = q8_scales = None
    if args.q8:
        q8 = torch.empty(dw.padded, dtype=torch.int8, device=dev)
        q8_scales = torch.empty(w.world_size * -(-dw.S // 256), device=dev)

    def one_step(timed=False):
        if q8 is not None:
            dw.flat.step_q8(w.ranks, dw.grads, dw.master, dw.m, dw.v, dw.out, q8, q8_scales,
                            grad_rank_offset_mul=w.grad_rank_mul, stream=stream,
                            want_result=False)
            return
        if K == 1:
            dw.step(want_result=False, stream=stream)
            return
        if timed:
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
        for k in range(K):
            dw.accumulate(first=(k == 0), stream=stream)
        if timed:
            a1.record(stream)
            acc_events.append((a0, a1))
        dw.step_accumulated(want_result=False, stream=stream)

    torch.cuda.synchronize(dev)
    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize(dev)
    graph = None
    if args.graph:
        # the warm-up steps above allocated the handle's scratch; capture one step
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            saved = stream
            stream = cap
            one_step()
            stream = saved
        stream.wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize(dev)

    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = str(local)
    sampler = ClockSampler(uuid)
    sampler.start()
    barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            one_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop()
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1))
    # the per-kernel split: a separate pass with CUDA events around every
    # launch (kept out of the timed steps above, whose time they would add to)
    Z.zero_flat_profile_enable(dw.flat.handle, True)
    Z.zero_flat_profile_read(dw.flat.handle)              # clear
    for _ in range(min(args.steps, 20)):
        one_step(timed=True)
    torch.cuda.synchronize(dev)
    Z.zero_flat_profile_enable(dw.flat.handle, False)
    ms_red, ms_fin, ms_adam, nrec = Z.zero_flat_profile_read(dw.flat.handle)
    res = (dw.step(want_result=True, stream=stream) if K == 1 else
           dw.step_accumulated(want_result=True, stream=stream))   # sanity: a clean step
    assert res.skipped == 0 and res.overflow == 0, "benchmark inputs overflowed"
    ms_acc = sum(a0.elapsed_time(a1) for a0, a1 in acc_events)

    N = w.world_size
    esize = 4 if w.grad_dtype == 2 else 2
    ms_step = elapsed_ms / args.steps
    value = whole_job_value(params, args.steps, world, elapsed_ms)
    peak, peak_kind = measured_peaks()
    # algorithmic bytes per parameter: the reduce reads the N contributions
    # (N*esize) and writes the fp32 reduced gradient (4); AdamW reads it (4)
    # and master/m/v (12), writes master/m/v (12) and the 16-bit param (2).
    # With micro-steps the reduce kernel is the norm pass over the fp32
    # accumulator (4) and the accumulate launches read N*esize, read (after
    # the first) and write the accumulator.
    kernels = {
        (reduce_name(dw.flat) if K == 1 else "reduce_kernel"): {
            "ms_mean": ms_red / max(nrec, 1),
            "bytes_per_param": N * esize + 4 if K == 1 else 4},
        ("adamw_q8_kernel" if args.q8 else "adamw_kernel"): {
            "ms_mean": ms_adam / max(nrec, 1),
            "bytes_per_param": 30 + (1 + 4 / 256 if args.q8 else 0)},
        "finalize_kernel": {"ms_mean": ms_fin / max(nrec, 1), "bytes_per_param": 0},
    }
    if K > 1:
        kernels["accumulate_launch"] = {
            "ms_mean": ms_acc / max(len(acc_events), 1) / K,
            "bytes_per_param": N * esize + (4 + 8 * (K - 1)) / K,
            "kernel": reduce_name(dw.flat)}
    for k in kernels.values():
        k["achieved_gbs"] = (k["bytes_per_param"] * params / (k["ms_mean"] / 1e3) / 1e9
                             if k["ms_mean"] > 0 else None)
    dom = max(kernels, key=lambda n: kernels[n]["ms_mean"] * (K if n == "accumulate_launch" else 1))
    dk = kernels[dom]
    traffic = profiled_traffic(dom, w.name)
    min_bytes = (K * N * esize + 26) * params               # the method's minimum per step
    step_gbs = min_bytes / (ms_step / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": dk["achieved_gbs"], "peak": peak,
                "unit": "GB/s", "frac": dk["achieved_gbs"] / peak if dk["achieved_gbs"] else None,
                "peak_kind": peak_kind, "traffic": traffic,
                "bytes_per_launch": dk["bytes_per_param"] * params}

    e2e = None
    if not args.no_e2e and K == 1 and not args.q8:
        e2e = measure_e2e(args, dw, stream, dev, params, barrier, max_over_ranks, world)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)
    side = None
    if (world == 1 and not args.no_workloads and w.name == "10b_rank7" and K == 1
            and not args.q8 and not args.graph):
        from synth.workloads import BY_NAME
        l2_note = (dw.flat.device_bytes() / 1e9 + (dw.grads.numel() * esize +
                   (3 + (K > 1)) * params * 4 + dw.out.numel() * 2) / 1e9)
        dw.close()
        del dw
        torch.cuda.empty_cache()
        dw = None
        side = {name: measure_workload(BY_NAME[name], args.workload_steps, 3, dev)
                for name in SIDE_WORKLOADS}
    else:
        l2_note = (dw.flat.device_bytes() / 1e9 + (dw.grads.numel() * esize +
                   (3 + (K > 1)) * params * 4 + dw.out.numel() * 2) / 1e9)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "Gparams/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "params_stepped_per_gpu": params,
                       "emulated_world_size": N, "stepped_ranks": w.ranks,
                       "storage": "%s grads, %s params, f32 master/m/v" %
                                  (("f16", "bf16", "f32")[w.grad_dtype],
                                   ("f16", "bf16")[w.param_dtype]),
                       "micro_steps": K,
                       "q8_payload": bool(args.q8),
                       "cuda_graph": bool(args.graph),
                       "l2": "inputs larger than L2 (%.0f GB resident vs 129 MB)" % l2_note,
                       "parallelism": "replicas%d" % world},
            "step_hbm": {"min_bytes_per_param": K * N * esize + 26, "achieved_gbs": step_gbs,
                         "frac_of_measured": step_gbs / peak,
                         "frac_of_nominal_8tbs": step_gbs / NOMINAL_HBM_GBS},
            "kernels": kernels,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clocks,
            "gpu_launches": launches_per_step * args.steps,
        }
        if side is not None:
            line["workloads"] = side
        print(json.dumps(line), flush=True)
    if dw is not None:
        dw.close()
    group.close()


# The configs reported beside the headline step (each its own FlatParameter,
# stepped alone on the device after the headline workload has been freed).
SIDE_WORKLOADS = ("tiny_mlp", "gpt2_small", "gpt_1p5b_rank17", "llama_7b_rank0")


def measure_workload(w, steps, warmup, dev):
    """Device-timed steps of one more config: ms per step, Gparams/s, each
    kernel's event-timed duration and achieved GB/s (algorithmic bytes), the
    step's HBM rate at the method's minimum bytes, and the dominant kernel's
    fraction of the measured copy peak."""
    import torch

    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    peak, peak_kind = measured_peaks()
    dw = DeviceWorkload(w, device=dev)
    try:
        stream = torch.cuda.current_stream(dev)
        dw.gen_grads(0, dw.scaler().scale)
        for _ in range(warmup):
            dw.step(want_result=False, stream=stream)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            dw.step(want_result=False, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
        Z.zero_flat_profile_enable(dw.flat.handle, True)    # per-kernel split, its own pass
        Z.zero_flat_profile_read(dw.flat.handle)
        for _ in range(steps):
            dw.step(want_result=False, stream=stream)
        torch.cuda.synchronize(dev)
        Z.zero_flat_profile_enable(dw.flat.handle, False)
        ms_red, _, ms_adam, nrec = Z.zero_flat_profile_read(dw.flat.handle)
        res = dw.step(want_result=True, stream=stream)
        assert res.skipped == 0 and res.overflow == 0, "%s inputs overflowed" % w.name
        params = dw.S * len(w.ranks)
        N = w.world_size
        esize = 4 if w.grad_dtype == 2 else 2
        kernels = {reduce_name(dw.flat): {"ms_mean": ms_red / max(nrec, 1),
                                          "bytes_per_param": N * esize + 4},
                   "adamw_kernel": {"ms_mean": ms_adam / max(nrec, 1), "bytes_per_param": 30}}
        for k in kernels.values():
            k["achieved_gbs"] = k["bytes_per_param"] * params / (k["ms_mean"] / 1e3) / 1e9
            k["frac_of_measured"] = k["achieved_gbs"] / peak
        dom = max(kernels, key=lambda n: kernels[n]["ms_mean"])
        min_b = (N * esize + 26) * params
        moved_b = (N * esize + 34) * params
        return {"ms_per_step": ms, "value": params / (ms / 1e3) / 1e9, "unit": "Gparams/s",
                "params_stepped": params, "emulated_world_size": N, "stepped_ranks": w.ranks,
                "steps": steps, "warmup": warmup,
                "step_hbm": {"min_bytes_per_param": N * esize + 26,
                             "achieved_gbs_at_min_bytes": min_b / (ms / 1e3) / 1e9,
                             "frac_of_nominal_8tbs_at_min_bytes":
                                 min_b / (ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                             "moved_bytes_per_param": N * esize + 34,
                             "achieved_gbs_moved": moved_b / (ms / 1e3) / 1e9,
                             "frac_of_nominal_8tbs_moved":
                                 moved_b / (ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                             "frac_of_measured_moved": moved_b / (ms / 1e3) / 1e9 / peak},
                "kernels": kernels,
                "roofline": {"bound": "hbm", "kernel": dom,
                             "achieved": kernels[dom]["achieved_gbs"], "peak": peak,
                             "unit": "GB/s", "frac": kernels[dom]["achieved_gbs"] / peak,
                             "peak_kind": peak_kind},
                "launches_per_step": 2}
    finally:
        dw.close()
        del dw
        torch.cuda.empty_cache()


def measure_e2e(args, dw, stream, dev, params, barrier, max_over_ranks, world):
    """The step through the C ABI with the contributions in pinned host memory:
    the kernels read them over the host link (every step moves all of them
    host -> device) and the step result is read back every step.  The time of
    the two-call form (an explicit host -> device copy, then the step on the
    device copy) is reported beside it."""
    import torch
    try:
        host = torch.empty(dw.grads.shape, dtype=dw.grads.dtype, pin_memory=True)
    except RuntimeError as e:
        return {"value": None, "unit": "Gparams/s", "error": "pinned host buffer: %s" % e}
    host.copy_(dw.grads)
    nbytes = host.numel() * host.element_size()
    w = dw.w

    def host_step():
        return dw.flat.step(w.ranks, host, dw.master, dw.m, dw.v, dw.out,
                            grad_rank_offset_mul=w.grad_rank_mul, stream=stream,
                            want_result=True)

    def copy_step():
        dw.grads.copy_(host, non_blocking=True)
        return dw.step(want_result=True, stream=stream)

    timings = {}
    for name, fn in (("zero_copy", host_step), ("copy_then_step", copy_step)):
        for _ in range(2):
            fn()
        barrier()
        torch.cuda.synchronize(dev)
        t = time.perf_counter()
        for _ in range(args.e2e_steps):
            res = fn()
            assert res.skipped == 0
        torch.cuda.synchronize(dev)
        timings[name] = max_over_ranks(time.perf_counter() - t)
        barrier()
    del host
    dt = timings["zero_copy"]
    return {"value": params * args.e2e_steps * world / dt / 1e9, "unit": "Gparams/s",
            "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": RESULT_D2H_BYTES,
            "ms_per_step": 1e3 * dt / args.e2e_steps, "steps": args.e2e_steps,
            "method": "kernels read the pinned host contributions over the host link",
            "copy_then_step_ms": 1e3 * timings["copy_then_step"] / args.e2e_steps}


def host_copy_gbs(nbytes=2 << 30, reps=3):
    """Host memory bandwidth of a multi-threaded torch CPU copy (bytes read +
    written per second, best of `reps`), the peak the host update is held to."""
    import torch
    n = nbytes // 4
    src = torch.ones(n, dtype=torch.float32)
    dst = torch.empty_like(src)
    best = 0.0
    for _ in range(reps + 1):
        t = time.perf_counter()
        dst.copy_(src)
        dt = time.perf_counter() - t
        best = max(best, 2 * n * 4 / dt / 1e9)
    return best, torch.get_num_threads()


def run_offload(args, w):
    """The ZeRO-Offload step on the workload: K1 reduces on the GPU and writes
    the fp32 gradient rows into pinned host memory, K2 decides, the host
    threads update master/m/v (host memory) and the 16-bit parameters are
    copied back into the device flat buffer."""
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    group = RankGroup(backend="nccl", device=dev)
    barrier, max_over_ranks = group.barrier, group.max

    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload

    dw = DeviceWorkload(w, device=dev)
    dw.gen_grads(0, dw.scaler().scale)
    stream = torch.cuda.current_stream(dev)
    hm, hmm, hv = ([t.cpu().pin_memory() for t in ts] for ts in (dw.master, dw.m, dw.v))
    dw.master = dw.m = dw.v = None                       # the state lives on the host
    torch.cuda.empty_cache()
    params = dw.S * len(w.ranks)
    n_batches = -(-len(w.ranks) // 64)

    def one_step():
        return dw.flat.step_offload(w.ranks, dw.grads, hm, hmm, hv, dw.out,
                                    grad_rank_offset_mul=w.grad_rank_mul,
                                    n_threads=args.offload_threads,
                                    gpu_share=args.offload_gpu_share, stream=stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize(dev)
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = str(local)
    sampler = ClockSampler(uuid)
    Z.zero_flat_profile_enable(dw.flat.handle, True)
    Z.zero_flat_profile_read(dw.flat.handle)
    sampler.start()
    barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        res = one_step()
        assert res.skipped == 0 and res.overflow == 0, "benchmark inputs overflowed"
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop()
    Z.zero_flat_profile_enable(dw.flat.handle, False)
    ms_red, ms_fin, ms_host, nrec = Z.zero_flat_profile_read(dw.flat.handle)
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1))
    peak, threads = host_copy_gbs()

    N = w.world_size
    esize = 4 if w.grad_dtype == 2 else 2
    # K1 reads the N contributions and writes the fp32 gradient rows in HBM.
    # On the host threads' share the update moves, in host memory: the DMA
    # write of the gradient (4 B/param), the CPU's reads of it (4) and of
    # master/m/v (12), its writes of master/m/v (12) and of the 16-bit staging
    # (2), and the DMA read of the staging (2) -- 36 B/param, 6 of them over
    # the link.  On the GPU's share the AdamW kernel reads and writes
    # master/m/v over the link: 24 B/param of host memory and of link traffic.
    f = max(0.0, min(1.0, args.offload_gpu_share))
    host_bpp = f * 24 + (1 - f) * 36
    kernels = {
        reduce_name(dw.flat): {"ms_mean": ms_red / max(nrec, 1),
                               "bytes_per_param": N * esize + 4},
        "finalize_kernel": {"ms_mean": ms_fin / max(nrec, 1), "bytes_per_param": 0},
        "host_update": {"ms_mean": ms_host / max(nrec, 1), "bytes_per_param": host_bpp,
                        "link_bytes_per_param": f * 24 + (1 - f) * 6},
    }
    for k in kernels.values():
        k["achieved_gbs"] = (k["bytes_per_param"] * params / (k["ms_mean"] / 1e3) / 1e9
                             if k["ms_mean"] > 0 else None)
    hu = kernels["host_update"]
    if rank == 0:
        line = {
            "metric": METRIC, "value": whole_job_value(params, args.steps, world, elapsed_ms),
            "unit": "Gparams/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "params_stepped_per_gpu": params,
                       "emulated_world_size": N, "stepped_ranks": w.ranks,
                       "offload": "AdamW on host cores, fp32 master/m/v in host memory",
                       "host_threads": args.offload_threads or len(os.sched_getaffinity(0)),
                       "gpu_share": f,
                       "parallelism": "replicas%d" % world},
            "kernels": kernels,
            "roofline": {"bound": "host-memory", "kernel": "host_update",
                         "achieved": hu["achieved_gbs"], "peak": peak, "unit": "GB/s",
                         "frac": hu["achieved_gbs"] / peak if hu["achieved_gbs"] else None,
                         "peak_kind": "measured here: torch CPU copy on %d threads" % threads,
                         "traffic": None, "bytes_per_launch": host_bpp * params},
            "cpu_baseline": None, "e2e": None, "clocks": clocks,
            "gpu_launches": n_batches * (2 if f > 0 else 1) * args.steps,
        }
        print(json.dumps(line), flush=True)
    dw.close()
    group.close()


def run_group(args):
    """M FlatParameters (N=8, rank 7's shard of group_params each, fp16 AVG,
    dynamic loss scale) stepped three ways: one zero_group_step (one global
    decision, two launches per 64 members); the split step per member with
    the totals summed on the device (the same global decision, two launches
    per member plus the decision); and one zero_shard_step per member (a
    decision per member -- a timing baseline only).  With --micro-steps K a
    step is K accumulations and the step from the accumulators, grouped
    (K + 1 launches per 64 members) or per member; with --q8 the steps also
    write the int8 all-gather payload (zero_group_step_q8 / zero_shard_step_q8);
    with --offload the fp32 state lives in pinned host memory and the update
    runs on the host threads (zero_group_step_offload / zero_shard_step_offload)."""
    import torch
    import fsdp_sharded_mixed_zero_gb300 as Z
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    from synth.workloads import AVG, F16, Workload

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    group = RankGroup(backend="nccl", device=dev)
    M, P = args.group, args.group_params
    ws = [Workload(name="member%d" % k, description="", shapes=[(8 * P,)], world_size=8,
                   ranks=[7], grad_dtype=F16, op=AVG, dynamic=True, steps=1, sigma_g=1e-3,
                   sigma_n=1e-3, grads_layout="slice", seed=k) for k in range(M)]
    ds = [DeviceWorkload(w, device=dev) for w in ws]
    for d in ds:
        d.gen_grads(0, d.scaler().scale)
    grp = Z.ZeroGroup([d.flat for d in ds])
    margs = [dict(ranks=w.ranks, grads=d.grads, master=d.master, m=d.m, v=d.v, out=d.out,
                  grad_rank_offset_mul=0) for w, d in zip(ws, ds)]
    ss = [torch.zeros((), dtype=torch.float64, device=dev) for _ in ds]
    of = [torch.zeros((), dtype=torch.int32, device=dev) for _ in ds]
    stream = torch.cuda.current_stream(dev)

    micro = max(1, args.micro_steps)
    q8 = bool(args.q8)
    off = bool(args.offload)
    if off:                                 # fp32 state in pinned host memory
        hargs = []
        for a in margs:
            h = dict(a)
            for name in ("master", "m", "v"):
                h[name] = [t.detach().cpu().pin_memory() for t in a[name]]
            hargs.append(h)
    if q8:                                  # the int8 all-gather payload as well
        for a, d in zip(margs, ds):
            a["q8"] = torch.empty(d.padded, dtype=torch.int8, device=dev)
            a["q8_scales"] = torch.empty(8 * -(-d.S // 256), dtype=torch.float32, device=dev)
    if micro > 1:                           # accumulation: micro-steps, then the step
        for d in ds:
            d.alloc_acc()
        aargs = [dict(ranks=w.ranks, grads=d.grads, acc=d.acc, grad_rank_offset_mul=0)
                 for w, d in zip(ws, ds)]
        sargs = [dict(ranks=w.ranks, acc=d.acc, master=d.master, m=d.m, v=d.v, out=d.out)
                 for w, d in zip(ws, ds)]

    def grouped():
        if off:
            grp.step_offload(hargs, n_threads=args.offload_threads,
                             gpu_share=args.offload_gpu_share, stream=stream)
            return
        if q8:
            grp.step_q8(margs, stream=stream, want_result=False)
            return
        if micro == 1:
            grp.step(margs, stream=stream, want_result=False)
            return
        for k in range(micro):
            grp.accumulate(aargs, first_micro_step=(k == 0), stream=stream)
        grp.step_accumulated(sargs, stream=stream, want_result=False)

    def split():
        for w, d, a, b in zip(ws, ds, ss, of):
            d.flat.reduce(w.ranks, d.grads, a, b, grad_rank_offset_mul=0, stream=stream)
        tot, mx = torch.stack(ss).sum(), torch.stack(of).max()
        for w, d in zip(ws, ds):
            d.flat.apply(w.ranks, d.master, d.m, d.v, d.out, tot, mx, stream=stream,
                         want_result=False)

    def per_member():
        for w, d, a, h in zip(ws, ds, margs, hargs if off else margs):
            if off:
                d.flat.step_offload(w.ranks, d.grads, h["master"], h["m"], h["v"], d.out,
                                    grad_rank_offset_mul=0, n_threads=args.offload_threads,
                                    gpu_share=args.offload_gpu_share, stream=stream)
                continue
            if q8:
                d.flat.step_q8(w.ranks, d.grads, d.master, d.m, d.v, d.out, a["q8"],
                               a["q8_scales"], grad_rank_offset_mul=0, stream=stream,
                               want_result=False)
                continue
            if micro == 1:
                d.step(want_result=False, stream=stream)
                continue
            for k in range(micro):
                d.accumulate(first=(k == 0), stream=stream)
            d.step_accumulated(want_result=False, stream=stream)

    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = str(local)
    times = {}
    clocks = None
    arms = [("group", grouped), ("split", split), ("per_flat_parameter", per_member)]
    if micro > 1 or q8 or off:
        arms = [arms[0], arms[2]]           # the split step has no accumulation, int8 or offload form
    for name, fn in arms:
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        sampler = ClockSampler(uuid) if name == "group" else None
        if sampler:
            sampler.start()
        group.barrier()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        group.barrier()
        if sampler:
            clocks = sampler.stop()
        times[name] = group.max(e0.elapsed_time(e1))
    if off:
        res = grp.step_offload(hargs, n_threads=args.offload_threads,
                               gpu_share=args.offload_gpu_share, stream=stream)
    elif q8:
        res = grp.step_q8(margs, stream=stream)
    elif micro == 1:
        res = grp.step(margs, stream=stream)
    else:
        for k in range(micro):
            grp.accumulate(aargs, first_micro_step=(k == 0), stream=stream)
        res = grp.step_accumulated(sargs, stream=stream)
    assert res.skipped == 0 and res.overflow == 0, "benchmark inputs overflowed"
    params = M * ds[0].S
    n_batches = -(-M // 64)
    if rank == 0:
        line = {
            "metric": METRIC, "value": whole_job_value(params, args.steps, world, times["group"]),
            "unit": "Gparams/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": times["group"] / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "group%dx%d" % (M, ds[0].S)
                       + ("_micro%d" % micro if micro > 1 else "") + ("_q8" if q8 else "")
                       + ("_offload" if off else ""),
                       "flat_parameters": M, "micro_steps": micro, "q8_payload": q8,
                       "offload": off,
                       "params_per_flat_parameter_shard": ds[0].S, "emulated_world_size": 8,
                       "stepped_ranks": [7], "parallelism": "replicas%d" % world},
            "compare_ms_per_step": {k: v / args.steps for k, v in times.items()},
            "clocks": clocks,
            "gpu_launches": ((micro + 1) * n_batches if not off
                             else n_batches * (1 + (args.offload_gpu_share > 0))) * args.steps,
        }
        print(json.dumps(line), flush=True)
    grp.close()
    for d in ds:
        d.close()
    group.close()


def main():
    args = parse_args()
    from synth.workloads import BY_NAME
    w = BY_NAME[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    elif args.group:
        run_group(args)
    elif args.offload:
        run_offload(args, w)
    elif args.collective:
        run_collective(args)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
