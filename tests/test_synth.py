"""The seeded input generator: its converters against library routines, its
stream against the published SplitMix64 definition, and the shapes of its
distributions."""
import numpy as np
import torch

import synth


def splitmix64_ref(seed, n):
    """SplitMix64 written out in Python integers (the published definition)."""
    out = []
    mask = (1 << 64) - 1
    state = seed
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & mask
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & mask
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & mask
        out.append(z ^ (z >> 31))
    return out


def test_stream_matches_definition():
    for seed in (0, 1, 301, 2 ** 63 + 5):
        assert synth.raw(50, seed).tolist() == splitmix64_ref(seed, 50)


def test_fp16_cast_matches_numpy():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(300000) * np.exp2(rng.integers(-30, 15, 300000))
    assert np.array_equal(synth.f64_to_fp16(x), x.astype(np.float16).view(np.uint16))


def test_e4m3_cast_matches_torch():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(300000) * np.exp2(rng.integers(-12, 9, 300000))).astype(np.float32)
    x = np.clip(x, -448, 448).astype(np.float64)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(synth.f64_to_e4m3(x), ref)
    # saturation: beyond +-448 clamps to the largest finite code
    assert synth.f64_to_e4m3(np.array([1e6, -1e6, 460.0])).tolist() == [0x7E, 0xFE, 0x7E]


def test_bf16_cast_matches_torch():
    """On doubles that are binary32 values, torch's binary32 -> bfloat16
    conversion (one RNE rounding) is the reference."""
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(300000) * np.exp2(rng.integers(-60, 60, 300000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.f64_to_bf16(x.astype(np.float64)), ref)
    h = synth.gauss_bf16(1000, 7)
    assert np.array_equal(h, synth.f64_to_bf16(synth.gauss_f64(1000, 7)))


def test_sign_and_gauss_statistics():
    s = synth.sign_fp16(200000, 101)
    assert set(np.unique(s).tolist()) == {0x3C00, 0xBC00}
    assert abs(np.mean(s == 0x3C00) - 0.5) < 0.01
    g = synth.gauss_f64(400000, 201)
    assert abs(g.mean()) < 0.01 and abs(g.std() - 1.0) < 0.01
    h = synth.gauss_fp16(1000, 201)
    assert np.array_equal(h, synth.f64_to_fp16(synth.gauss_f64(1000, 201)))


def test_e4m3_quantisation_maps_max_to_448():
    q, scale = synth.gauss_e4m3(100000, 501)
    vals = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
    assert np.max(np.abs(vals)) == 448.0
    amax = np.max(np.abs(synth.gauss_f64(100000, 501)))
    assert abs(scale * 448.0 - amax) <= 1e-6 * amax


def test_workload_table():
    w = synth.WORKLOADS["sq_8192"]
    assert (w.M, w.N, w.K, w.rotating) == (8192, 8192, 8192, 4)
    assert w.seeds(1) == (303, 304)
    f = synth.WORKLOADS["ffn_8192"]
    assert (f.M, f.N, f.K, f.dtype) == (8192, 28672, 8192, "f16")
    A, B, sa, sb = synth.make_inputs(synth.WORKLOADS["pm1_512"])
    assert A.size == 512 * 512 and sa == 1.0
