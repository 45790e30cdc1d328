"""The C-ABI library: loads, exports every function include/*.h declares,
validates arguments on the host before touching the GPU, and its host-only
memory accounting equals the oracle's (pinned to the pages' figures).
No kernel runs here."""
import ctypes as C
import os
import re

import pytest

import fsdp_sharded_mixed_zero_gb300 as Z

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))


def declared_functions():
    names = set()
    for path in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
        names.update(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(zero_\w+)\s*\(", text, re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("zero_flat_init", "zero_flat_layout", "zero_shard_step",
                 "zero_loss_scaler_state", "zero_set_loss_scaler_state", "zero_memory_bytes",
                 "zero_flat_free", "zero_status_string", "zero_last_error",
                 "zero_shard_step_offload", "zero_debug_set_stage_tx_pad"):
        assert want in names


def test_library_exports_every_declared_symbol():
    lib = C.CDLL(Z.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_library_is_in_tree():
    assert os.path.dirname(Z.LIB_PATH) == os.path.join(ROOT, "fsdp_sharded_mixed_zero_gb300")


def test_status_strings():
    for s in range(8):
        assert Z.zero_status_string(s) not in ("", "unknown status")
    assert Z.zero_status_string(99) == "unknown status"


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
@pytest.mark.parametrize("psi,N", [(10 ** 10, 8), (1_500_000_000, 64), (175 * 10 ** 9, 1024),
                                   (1, 3), (7, 7), (12345, 17), (2 ** 60, 5)])
def test_memory_bytes_matches_oracle(ora, stage, psi, N):
    try:
        p, g, o, t = ora.memory_breakdown(stage, psi, N)
    except ValueError:                                # both sides refuse to overflow
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_memory_bytes(stage, psi, N)
        assert e.value.status == 5
        return
    assert Z.zero_memory_bytes(stage, psi, N) == (t, p, g, o)


def test_memory_bytes_pages_figures():
    GB = 10 ** 9
    assert Z.zero_memory_bytes(0, 10 * GB, 8)[0] == 160 * GB
    assert Z.zero_memory_bytes(1, 10 * GB, 8)[0] == 55 * GB
    assert Z.zero_memory_bytes(2, 10 * GB, 8)[0] == 37_500_000_000
    assert Z.zero_memory_bytes(3, 10 * GB, 8)[0] == 20 * GB
    assert Z.zero_memory_bytes(1, 10 * GB, 8)[3] == 15 * GB


def test_memory_bytes_errors():
    out = [C.c_uint64() for _ in range(4)]
    lib = Z._lib
    assert lib.zero_memory_bytes(4, 1, 1, *[C.byref(o) for o in out]) == 1
    assert lib.zero_memory_bytes(1, 1, 0, *[C.byref(o) for o in out]) == 1
    assert lib.zero_memory_bytes(0, 2 ** 63, 1, *[C.byref(o) for o in out]) == 5
    assert lib.zero_memory_bytes(1, 5, 2, None, None, None, None) == 0


def _init_status(infos, world=4, gdt=0, pdt=0, op=1, hp=None):
    h = C.c_void_p()
    hp = hp if hp is not None else Z.hparams()
    n = len(infos)
    return Z._lib.zero_flat_init(infos, n, world, gdt, pdt, op, C.byref(hp), C.byref(h))


def test_init_validates_on_the_host():
    good = Z.param_infos([(4, 4), (3,)])
    assert _init_status(good, world=0) == 1
    assert _init_status(good, gdt=7) == 2
    assert _init_status(good, op=3) == 1
    bad = Z.param_infos([(4, 4), (3,)])
    bad[1].offset = 17                              # gap after the first param
    assert _init_status(bad) == 1
    bad = Z.param_infos([(4, 4)])
    bad[0].numel = 15                               # numel != prod(shape)
    assert _init_status(bad) == 1
    bad = Z.param_infos([(4, 4)])
    bad[0].ndim = 9
    assert _init_status(bad) == 1
    bad = Z.param_infos([(2 ** 40, 2 ** 40)])
    assert _init_status(bad) == 5                   # shape product overflows
    for kw in (dict(beta1=1.0), dict(beta2=-0.1), dict(eps=0.0), dict(window=0),
               dict(lr=float("nan")), dict(initial_scale_power=200),
               dict(dynamic=False, static_scale=0.0), dict(min_scale=0.0)):
        assert _init_status(good, hp=Z.hparams(**kw)) == 1, kw
    hp = Z.hparams()
    hp.reserved = 1
    assert _init_status(good, hp=hp) == 1
    assert Z._lib.zero_flat_init(good, 2, 4, 0, 0, 1, C.byref(Z.hparams()), None) == 1
    assert Z._lib.zero_flat_init(None, 0, 4, 0, 0, 1, C.byref(Z.hparams()),
                                 C.byref(C.c_void_p())) == 1


def test_null_handle_is_rejected():
    lib = Z._lib
    one = (C.c_int32 * 1)(0)
    ptrs = (C.c_void_p * 1)(None)
    assert lib.zero_shard_step(None, one, 1, None, 0, 0, ptrs, ptrs, ptrs, None, 0.0, None,
                               None) == 1
    assert lib.zero_flat_layout(None, None, None, None) == 1
    assert lib.zero_loss_scaler_state(None, None, None) == 1
    assert lib.zero_flat_free(None) == 0


def test_no_cpu_fallback_without_a_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = _init_status(Z.param_infos([(64,)]))
    assert st == 4, Z.zero_last_error()              # ZERO_ERR_CUDA: fails loudly
