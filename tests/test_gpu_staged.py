"""GPU parity of the staged reduce (reduce_staged_kernel): contributor rows
go through TMA bulk copies of 64-byte-aligned spans into shared memory and
are re-aligned there.  The planner takes it for rows whose starts are not
64-byte aligned, and for aligned rows once a reduce reads at least 1 GiB of
contributions.  Every case is compared with the oracle element by element on
every step, and the CUDA profiler confirms which kernel ran.

Layouts: the full [N, padded] layout with an odd shard size (rank slices
2-byte aligned, or 4-byte for fp32 contributions), a slice layout whose
row stride is 32 bytes off a 64-byte multiple, fewer contributors than one
stage holds, more contributors than several stages hold, padding, the
micro-step accumulation modes, and aligned rows below and above 1 GiB."""
import warnings

import pytest

torch = pytest.importorskip("torch")

from synth.workloads import AVG, BF16, F16, F32, SUM, Workload  # noqa: E402

from tests.test_gpu_accumulate import run_accum_parity  # noqa: E402
from tests.test_gpu_parity import run_parity  # noqa: E402

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _wl(name, numel, N, ranks, dtype=F16, op=AVG, dynamic=True, steps=3, layout="full",
        micro=1, inf_at=None):
    return Workload(name=name, description=name, shapes=[(numel,)], world_size=N, ranks=ranks,
                    grad_dtype=dtype, op=op, dynamic=dynamic, steps=steps, sigma_g=1e-3,
                    sigma_n=1e-3, inf_at=inf_at, grads_layout=layout, micro_steps=micro)


def _kernels_launched(fn):
    """Names of the CUDA kernels fn launched (empty if the profiler has no
    CUDA activity here)."""
    from torch.profiler import ProfilerActivity, profile
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    return {e.name for e in prof.events()}


def _step_kernels(w):
    """Kernel names of one step of w (the profiler's first session in a
    process may come back empty while it initialises: one retry)."""
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    dw = DeviceWorkload(w)
    try:
        dw.gen_grads(0, dw.scaler().scale)
        names = set()
        for _ in range(2):
            names = _kernels_launched(lambda: dw.step(want_result=False))
            if names:
                break
        return names
    finally:
        dw.close()


def _assert_staged(w):
    names = _step_kernels(w)
    if not names:
        warnings.warn("the CUDA profiler recorded no kernels: kernel choice not checked")
        return
    assert any("reduce_staged_kernel" in n for n in names), sorted(names)


STEP_CASES = [
    # rank slices at r * 20001 elements: odd ranks 2-byte aligned; padding on rank 7
    _wl("f16_full_odd_shard", 8 * 20_001 - 3, 8, list(range(8)), steps=4, inf_at=(2, 3, 7)),
    # five contributors (one partial stage), bf16 SUM, static scale
    _wl("bf16_full_n5", 5 * 9_999 + 2, 5, list(range(5)), dtype=BF16, op=SUM, dynamic=False),
    # fp32 contributions with 4-byte aligned slices, padding on the last rank
    _wl("f32_full_odd_shard", 4 * 30_001 - 2, 4, [0, 1, 2, 3], dtype=F32),
    # 70 contributors (nine row groups) and two launches of ranks
    _wl("n70_full", 70 * 2_501 + 13, 70, list(range(70)), steps=2),
    # slice layout: rows 250000 elements apart = 32 bytes off a 64-byte multiple
    _wl("f16_slice_stride32", 16 * 250_000, 16, [5], layout="slice"),
]


@pytest.mark.parametrize("w", STEP_CASES, ids=lambda w: w.name)
def test_staged_step_matches_oracle(ora, w):
    _need_gpu()
    _assert_staged(w)
    res = run_parity(ora, w)
    if w.inf_at is not None:
        assert res[w.inf_at[0]][1] == 1


# Shard sizes that are multiples of 4 keep the accumulator rows (views of one
# buffer at j * S floats) 16-byte aligned, as staging needs, while the
# contributor slices at r * S stay off 64-byte boundaries.
ACC_CASES = [
    _wl("accum_full_s50004", 4 * 50_004 - 3, 4, [0, 1, 2, 3], micro=3, steps=2,
        inf_at=(4, 1, 3)),
    _wl("accum_f32_full_s40004", 2 * 40_004 - 1, 2, [0, 1], dtype=F32, micro=2, steps=2),
]


def _assert_accumulate_staged(w):
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    dw = DeviceWorkload(w)
    try:
        dw.alloc_acc()
        dw.gen_grads(0, dw.scaler().scale)
        names = set()
        for _ in range(2):
            names = _kernels_launched(lambda: dw.accumulate(first=True))
            if names:
                break
    finally:
        dw.close()
    if not names:
        warnings.warn("the CUDA profiler recorded no kernels: kernel choice not checked")
        return
    assert any("reduce_staged_kernel" in n for n in names), sorted(names)


@pytest.mark.parametrize("w", ACC_CASES, ids=lambda w: w.name)
def test_staged_accumulation_matches_oracle(ora, w):
    _need_gpu()
    _assert_accumulate_staged(w)
    skipped = run_accum_parity(ora, w)
    if w.inf_at is not None:
        assert skipped[w.inf_at[0] // w.micro_steps] == 1


def test_small_aligned_launch_keeps_the_plain_kernel():
    """Rows 128-byte aligned and 1 MB of contributions: the plain reduce
    (its fixed cost is lower; staging pays off from 1 GiB per reduce)."""
    _need_gpu()
    names = _step_kernels(_wl("aligned_slice", 8 * 64 * 1000, 8, [3], layout="slice"))
    if not names:
        pytest.skip("the CUDA profiler recorded no kernels")
    assert not any("reduce_staged_kernel" in n for n in names)
    assert any("reduce_kernel" in n for n in names)


def test_large_aligned_launch_is_staged_and_matches_oracle(ora):
    """Rows 64-byte aligned (slice layout, 8 contributions of 70M elements,
    1.12 GB): at least 1 GiB of contributions takes the staged reduce; the
    step must match the oracle, and the handle must report the form."""
    _need_gpu()
    from fsdp_sharded_mixed_zero_gb300.harness import DeviceWorkload
    w = _wl("aligned_slice_1gib", 8 * 70_000_000, 8, [3], layout="slice", steps=2)
    _assert_staged(w)
    run_parity(ora, w)
    dw = DeviceWorkload(w)
    try:
        assert dw.flat.reduce_form() is None
        dw.gen_grads(0, dw.scaler().scale)
        dw.step()
        assert dw.flat.reduce_form() == "staged"
    finally:
        dw.close()
    small = DeviceWorkload(_wl("aligned_small", 8 * 64 * 1000, 8, [3], layout="slice"))
    try:
        small.gen_grads(0, small.scaler().scale)
        small.step()
        assert small.flat.reduce_form() == "plain"
    finally:
        small.close()
