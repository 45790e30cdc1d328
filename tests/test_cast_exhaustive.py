"""Every one of the 2^32 fp32 bit patterns through the round-to-nearest-even
16-bit casts: the oracle's fp16 cast against numpy's float16 conversion and
its bf16 cast against torch's bfloat16 conversion (both libraries round to
nearest even, with subnormals, overflow to inf and NaN), and the same for the
host casts of the offload step (zero_offload_adamw_host with lr = 0 and no
decay leaves theta unchanged, so its output is the cast alone).  NaN inputs
must give a NaN encoding; every other pattern must match exactly.

The 2^32 patterns are split into 2^24-pattern ranges checked by a spawn
process pool (one process per CPU)."""
import multiprocessing as mp
import os

import numpy as np
import pytest

RANGE = 1 << 24


def _check_range(k):
    """Mismatch counts over the patterns [k * RANGE, (k + 1) * RANGE)."""
    import torch

    import fsdp_sharded_mixed_zero_gb300 as Z
    import oracle as ora

    torch.set_num_threads(1)
    u = np.arange(RANGE, dtype=np.uint32) + np.uint32(k * RANGE)
    x = u.view(np.float32)
    nan = np.isnan(x)
    with np.errstate(over="ignore"):
        want16 = x.astype(np.float16).view(np.uint16)
    wantb = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    def bad(got, want, exp_mask, man_mask):
        n = int(np.count_nonzero(got[~nan] != want[~nan]))
        g = got[nan]
        n += int(np.count_nonzero(((g & exp_mask) != exp_mask) | ((g & man_mask) == 0)))
        return n

    out = {"oracle_f16": bad(ora.cast_array(x), want16, 0x7C00, 0x03FF),
           "oracle_bf16": bad(ora.cast_array(x, to_bf16=True), wantb, 0x7F80, 0x007F)}
    hp = Z.hparams(lr=0.0, weight_decay=0.0)
    z = np.zeros(RANGE, np.float32)
    for name, dt, want, em, mm in (("host_f16", Z.ZERO_F16, want16, 0x7C00, 0x03FF),
                                   ("host_bf16", Z.ZERO_BF16, wantb, 0x7F80, 0x007F)):
        th = x.copy()
        m, v = z.copy(), z.copy()
        got = np.empty(RANGE, np.uint16)
        Z.zero_offload_adamw_host(hp, 1, 1.0, z.ctypes.data, th.ctypes.data, m.ctypes.data,
                                  v.ctypes.data, got.ctypes.data, RANGE, dt, 1)
        out[name] = bad(got, want, em, mm)
    return k, out


def test_all_fp32_patterns():
    pytest.importorskip("torch")
    n_ranges = (1 << 32) // RANGE
    totals = {}
    ctx = mp.get_context("spawn")
    with ctx.Pool(processes=max(1, min(len(os.sched_getaffinity(0)), 16))) as pool:
        for k, counts in pool.imap_unordered(_check_range, range(n_ranges)):
            for name, c in counts.items():
                totals[name] = totals.get(name, 0) + c
                assert c == 0, "%s: %d mismatches in patterns [%#x, %#x)" % (
                    name, c, k * RANGE, (k + 1) * RANGE)
    assert set(totals) == {"oracle_f16", "oracle_bf16", "host_f16", "host_bf16"}
