"""Pins of the oracle's E4M3 encoder and per-tensor quantiser (CPU only).

The encoder is pinned by the E4M3 definition (OCP OFP8): every finite code
round-trips, every midpoint between neighbouring codes goes to the code with
the even fraction (the code's lowest bit), hand-derived ties and saturation
cases, and torch's own float8_e4m3fn conversion below 448.  The quantiser
(amax over the tensor, s_q = 448 / amax in binary32, one rounding of x * s_q)
is pinned by closed forms (power-of-two amax), sign symmetry, the zero tensor,
the dequantisation error bound, layout invariance, and equality across the
three input types for values all of them hold.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_encode_roundtrip_exhaustive():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue                       # NaN codes
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def test_e4m3_encode_nan():
    assert oracle.e4m3_encode(float("nan")) & 0x7F == 0x7F


def test_e4m3_midpoints_go_to_even_fraction():
    """Between neighbouring positive codes c and c+1 (both finite), the exact
    midpoint rounds to the one whose lowest bit -- the fraction's last bit --
    is 0; a hair either side rounds to the nearer code."""
    for c in range(0x00, 0x7E):
        lo, hi = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = (lo + hi) / 2.0
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == even, hex(c)
        assert oracle.e4m3_encode(-mid) == 0x80 | even, hex(c)
        d = (hi - lo) / 1024.0
        assert oracle.e4m3_encode(mid - d) == c
        assert oracle.e4m3_encode(mid + d) == c + 1


def test_e4m3_encode_hand_cases():
    with open(os.path.join(GOLDEN, "e4m3_encode_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        assert oracle.e4m3_encode(float(c["x"])) == int(c["code"], 16), c


def test_e4m3_encode_vs_torch_below_448():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(20000) * 60, rng.standard_normal(5000) * 1e-3,
                        rng.uniform(-447.9, 447.9, 5000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, ref)


def _f32(x):
    return np.asarray(x, np.float32)


@pytest.mark.parametrize("k", [-3, 0, 5])
def test_quantize_power_of_two_amax_closed_form(k):
    """With amax = 448 * 2^k, s_q = 2^-k exactly and scale = 2^k exactly, so
    every code is the encoding of x * 2^-k and the largest element maps to 448."""
    rng = np.random.default_rng(11 + k)
    x = _f32(rng.uniform(-1, 1, (37, 53)) * 448 * 2.0 ** k)
    amax = np.float32(448 * 2.0 ** k)
    x[5, 7] = -amax
    q, scale = oracle.quantize_e4m3(x, "f32", 37, 53)
    assert scale == 2.0 ** k
    want = np.array([oracle.e4m3_encode(float(v) * 2.0 ** -k) for v in x.reshape(-1)], np.uint8)
    assert np.array_equal(q, want)
    assert q[5 * 53 + 7] == 0xFE


def test_quantize_zero_tensor():
    x = _f32(np.zeros((4, 9)))
    x[1, 2] = -0.0
    q, scale = oracle.quantize_e4m3(x, "f32", 4, 9)
    assert scale == 0.0
    assert np.all((q & 0x7F) == 0)
    assert q[1 * 9 + 2] == 0x80 and q[0] == 0x00


def test_quantize_sign_symmetry():
    rng = np.random.default_rng(3)
    x = _f32(rng.standard_normal((20, 33)))
    q1, s1 = oracle.quantize_e4m3(x, "f32", 20, 33)
    q2, s2 = oracle.quantize_e4m3(-x, "f32", 20, 33)
    assert s1 == s2
    assert np.array_equal(q1 ^ 0x80, q2)


def test_quantize_dequantisation_error_bound():
    """decode(q) * scale is within 2^-4 (E4M3 rounding) plus a few binary32
    roundings of x, or within half a subnormal quantum (2^-10 * scale)."""
    rng = np.random.default_rng(9)
    x = _f32(rng.standard_normal((64, 257)) * np.exp(rng.uniform(-6, 6, (64, 257))))
    q, scale = oracle.quantize_e4m3(x, "f32", 64, 257)
    back = np.array([oracle.e4m3_decode(int(c)) for c in q], np.float64) * scale
    err = np.abs(back - x.reshape(-1).astype(np.float64))
    bound = (2.0 ** -4 + 2.0 ** -20) * np.abs(x.reshape(-1)) + 2.0 ** -10 * scale * (1 + 2.0 ** -20)
    assert np.all(err <= bound)
    amax = np.max(np.abs(x))
    assert scale == np.float32(amax) / np.float32(448)


def test_quantize_strided_equals_contiguous():
    rng = np.random.default_rng(4)
    rows, cols, ldx, ldq = 13, 29, 40, 35
    x = _f32(rng.standard_normal((rows, ldx)) * 3)
    x[:, cols:] = 1e6                       # padding beyond cols must be ignored
    q, s = oracle.quantize_e4m3(x, "f32", rows, cols, ldx, ldq)
    qc, sc = oracle.quantize_e4m3(np.ascontiguousarray(x[:, :cols]), "f32", rows, cols)
    assert s == sc
    assert np.array_equal(q.reshape(rows, ldq)[:, :cols], qc.reshape(rows, cols))


def test_quantize_input_types_agree():
    """binary16 and bfloat16 codes quantise like the binary32 values they
    encode (decoded here by numpy / bit shifting, not by the oracle)."""
    rng = np.random.default_rng(8)
    h = rng.standard_normal(500).astype(np.float16)
    q16, s16 = oracle.quantize_e4m3(h.view(np.uint16), "f16", 20, 25)
    q32, s32 = oracle.quantize_e4m3(h.astype(np.float32), "f32", 20, 25)
    assert s16 == s32 and np.array_equal(q16, q32)
    bits = (rng.integers(0, 1 << 16, 500, dtype=np.uint32) & 0xBFFF).astype(np.uint16)   # no Inf / NaN
    qb, sb = oracle.quantize_e4m3(bits, "bf16", 20, 25)
    as32 = (bits.astype(np.uint32) << 16).view(np.float32)
    qf, sf = oracle.quantize_e4m3(as32, "f32", 20, 25)
    assert sb == sf and np.array_equal(qb, qf)


def test_quantize_vs_torch_conversion():
    """The codes equal torch's float8_e4m3fn conversion of the binary32
    products x * (448 / amax), saturated at 448 (torch maps larger values to
    NaN, the quantiser to the largest finite value)."""
    rng = np.random.default_rng(21)
    x = _f32(rng.standard_normal(4096) * 7.3)
    q, scale = oracle.quantize_e4m3(x, "f32", 1, 4096)
    amax = np.float32(np.max(np.abs(x)))
    prod = x * (np.float32(448) / amax)
    prod = np.clip(prod, np.float32(-448), np.float32(448))
    ref = torch.from_numpy(prod).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    assert scale == amax / np.float32(448)


def test_quantize_overflowing_reciprocal_uses_flt_max():
    """bfloat16 subnormals: 448 / amax overflows binary32, so s_q = FLT_MAX."""
    bits = np.array([0x0001, 0x8003, 0x0002, 0x0000], np.uint16)     # 2^-133 * (1, -3, 2, 0)
    q, scale = oracle.quantize_e4m3(bits, "bf16", 1, 4)
    fmax = np.float32(np.finfo(np.float32).max)
    vals = [float(np.float32(v) * fmax) for v in (2.0 ** -133, -3 * 2.0 ** -133, 2 * 2.0 ** -133, 0.0)]
    assert list(q) == [oracle.e4m3_encode(v) for v in vals]
    assert scale == np.float32(3 * 2.0 ** -133) / np.float32(448)
