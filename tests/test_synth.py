"""The seeded input generator: Philox4x32-10 against the published
known-answer vectors, the Box-Muller normal's moments and tails,
counter-based regeneration of single elements, thread-count independence."""
import numpy as np
import pytest

import synth

# Known-answer tests distributed with Random123 (Salmon et al., SC'11) for
# philox4x32 with 10 rounds: (counter, key) -> output.
KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,want", KAT)
def test_philox_known_answers(ctr, key, want):
    assert tuple(synth.philox(ctr, key)) == want


def test_normal_moments_and_tails():
    n = 4_000_000
    x = synth.normal_host(0, synth.MASTER, 0, n, 1.0).astype(np.float64)
    assert abs(x.mean()) < 3e-3
    assert abs(x.var() - 1.0) < 5e-3
    kurt = ((x - x.mean()) ** 4).mean() / x.var() ** 2 - 3.0
    assert abs(kurt) < 0.03                           # a normal has excess kurtosis 0
    assert np.abs(x).max() <= np.sqrt(2 * 24 * np.log(2)) + 1e-5   # u1 >= 2^-24
    # tail mass beyond 3 and 4 sigma: 2.70e-3 and 6.33e-5 for a normal
    # (binomial standard errors ~2.6e-5 and ~4e-6 at this n)
    assert abs(np.mean(np.abs(x) > 3.0) - 2.6998e-3) < 2e-4
    assert abs(np.mean(np.abs(x) > 4.0) - 6.334e-5) < 2.5e-5
    y = synth.normal_host(0, synth.MASTER, 0, 1000, 0.02)
    assert np.array_equal(y, (x[:1000] * 0.02).astype(np.float32))


def test_counter_based_regeneration_and_threads():
    big = synth.normal_host(7, synth.GRAD_SHARED, 10 ** 9, 300_000, 1e-3)
    for k in (0, 1, 12345, 299_999):
        one = synth.normal_host(7, synth.GRAD_SHARED, 10 ** 9 + k, 1, 1e-3)
        assert one[0] == big[k]
    g = synth.grads_host(3, 2, 4, 5_000_000, 200_000, 1e-3, 1e-3, scale=65536.0)
    g2 = np.concatenate([synth.grads_host(3, 2, 4, 5_000_000 + a, 50_000, 1e-3, 1e-3,
                                          scale=65536.0) for a in range(0, 200_000, 50_000)],
                        axis=1)
    assert np.array_equal(g, g2)


def test_grads_recipe():
    # grad[c][i] = fp16((g_i + n_{c,i}) * scale): shared part identical across c
    n, N = 100_000, 4
    g = synth.grads_host(5, 1, N, 0, n, 1e-3, 0.0, scale=1024.0)
    assert all(np.array_equal(g[0], g[c]) for c in range(N))
    shared = synth.normal_host(5, synth.GRAD_SHARED, 0, n, 1e-3, step=1)
    assert np.array_equal(g[0], (shared * np.float32(1024.0)).astype(np.float16).view(np.uint16))
    b = synth.grads_host(5, 1, 2, 0, n, 1e-3, 1e-3, dtype=synth.BF16)
    assert b.shape == (2, n) and b.dtype == np.uint16
    z = synth.grads_host(5, 1, 2, 0, 10, 1.0, 1.0, zero_from=6)
    assert not z[:, 6:].any() and z[:, :6].all()


def test_workload_shapes_are_the_architectures():
    # the FlatParameters of the synthetic workloads hold exactly the parameters of
    # the architectures they stand for (element counts and tensor counts):
    # GPT-2 small with a tied head 124,439,808 in 148 tensors; the 48-layer,
    # d=1600 GPT-2 (the 1.5B model) 1,557,611,200 in 580; the Llama-shaped 7B
    # with an untied head 6,738,415,616 in 291
    from synth import workloads as W
    for w, numel, tensors in ((W.GPT2, 124_439_808, 148), (W.GPT_1P5B, 1_557_611_200, 580),
                              (W.LLAMA_7B, 6_738_415_616, 291)):
        assert sum(int(np.prod(s)) for s in w.shapes) == numel, w.name
        assert len(w.shapes) == tensors, w.name
    # the tiny MLP: [512x1024, 1024, 1024x512, 512]
    assert sum(int(np.prod(s)) for s in W.TINY.shapes) == 1_050_112
