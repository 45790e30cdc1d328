"""The N>1 host path of the benchmark on CPU ranks (gloo): rendezvous on
127.0.0.1, barrier, the maximum of the timed region over ranks, the
whole-job value of independent replicas, and a real two-process torchrun of
the reference arm (rank 0 alone runs it and prints one JSON line; the other
rank exits 0 without output)."""
import json
import os
import socket
import subprocess
import sys
import tempfile

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    g = bench.RankGroup(backend="gloo", device="cpu")
    assert (g.world, g.rank) == (world, rank)
    g.barrier()
    elapsed = 100.0 + 25.0 * rank                   # the slowest rank decides
    mx = g.max(elapsed)
    value = bench.whole_job_value(1_250_000_000, 10, g.world, mx)
    g.barrier()
    g.close()
    with open(os.path.join(out_dir, "r%d.json" % rank), "w") as f:
        json.dump({"max": mx, "value": value}, f)


def test_rank_group_gloo_two_ranks():
    world = 2
    port = _free_port()
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_worker, args=(world, port, d), nprocs=world, join=True,
                           start_method="spawn")
        res = [json.load(open(os.path.join(d, "r%d.json" % r))) for r in range(world)]
    for r in res:
        assert r["max"] == 125.0
        # 2 ranks x 10 steps x 1.25e9 params in 125 ms
        assert abs(r["value"] - 2 * 10 * 1.25e9 / 0.125 / 1e9) < 1e-9


def test_single_rank_group_is_local():
    import bench
    g = bench.RankGroup()
    assert g.world == int(os.environ.get("WORLD_SIZE", "1"))
    if g.world == 1:
        assert g.max(3.5) == 3.5
        g.barrier()
    g.close()


def test_torchrun_reference_arm_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2",
           "--impl", "reference", "--steps", "1", "--warmup", "1", "--workload", "tiny_mlp",
           "--ref-seconds", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.parametrize("argv", [["--q8", "--micro-steps", "2"], ["--offload", "--q8"],
                                  ["--group", "4", "--offload", "--micro-steps", "3"],
                                  ["--collective", "--q8"], ["--collective", "--offload"]])
def test_bench_rejects_step_forms_that_exclude_one_another(argv):
    """The step forms are refused at argument parsing, before any device work."""
    import bench
    with pytest.raises(SystemExit) as e:
        bench.parse_args(argv)
    assert e.value.code == 2


def test_bench_accepts_each_step_form_alone():
    import bench
    for argv in ([], ["--q8"], ["--micro-steps", "4"], ["--offload"], ["--group", "8", "--q8"],
                 ["--collective", "--collective-shard", "1000"]):
        bench.parse_args(argv)


def test_host_cpu_names_the_model():
    import bench
    arm = ("processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\n"
           "CPU architecture: 8\nCPU variant\t: 0x0\nCPU part\t: 0xd4f\n\n"
           "processor\t: 1\nCPU implementer\t: 0x41\nCPU part\t: 0xd4f\n")
    h = bench.host_cpu(arm)
    assert h["cpu_model"] == "Arm Neoverse-V2"
    assert h["nproc"] >= 1 and 1 <= h["usable_cpus"] <= h["nproc"]
    assert bench.host_cpu("processor\t: 0\nCPU implementer\t: 0x51\nCPU part\t: 0x001\n")[
        "cpu_model"] == "implementer 0x51 part 0x001"
    assert bench.host_cpu("model name\t: Some CPU @ 3GHz\n")["cpu_model"] == "Some CPU @ 3GHz"


def test_collective_rendezvous_under_torchrun_uses_the_launchers_store():
    # one rank under torchrun: the agent's store (a tcp:// address would make
    # the rank a client of a store nobody serves and wait for its timeout)
    import bench
    env = {"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": "29500", "WORLD_SIZE": "1",
           "TORCHELASTIC_USE_AGENT_STORE": "True"}
    assert bench.rendezvous_method(env, 1) == "env://"
    assert bench.rendezvous_method({}, 2) == "env://"
    m = bench.rendezvous_method({}, 1)                   # started directly: a private store
    assert m.startswith("tcp://127.0.0.1:") and int(m.rsplit(":", 1)[1]) > 0
