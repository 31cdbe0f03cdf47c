"""Pins for the CPU oracle, each against something other than the oracle itself.

* values the pages print (the worked example, its partial sums and the
  outer-product intermediates: hello-gpu ch.11 "GEMM-Like", sections 11.1,
  11.2 and exercise 1 of 11.7) -- tests/golden/worked_example.json;
* closed forms (all-ones gives K, identity gives B, permutations permute B);
* exact rational brute force (Python ``fractions``) on the edge shapes listed
  in section 11.4 of the same chapter;
* the codecs against numpy / torch CPU conversions, exhaustively, plus
  hand-derived round-to-nearest-even ties.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

EDGE_SHAPES = [(1, 1, 1), (3, 5, 7), (15, 17, 19), (17, 19, 23), (31, 33, 29)]


def f16(vals):
    return np.asarray(vals, np.float64).astype(np.float16).view(np.uint16)


def dec16(codes):
    return np.asarray(codes, np.uint16).view(np.float16).astype(np.float64)


def tn_from_math(Am, Bm):
    """Math-view A (M x K) and B (K x N) to TN storage (A row-major, B col-major)."""
    Am, Bm = np.asarray(Am, np.float64), np.asarray(Bm, np.float64)
    return f16(Am.reshape(-1)), f16(Bm.T.reshape(-1))


@pytest.fixture(scope="module")
def worked(golden_dir):
    with open(os.path.join(golden_dir, "worked_example.json")) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# values printed on the pages
def test_worked_example(worked):
    A, B = f16(worked["A_tn"]), f16(worked["B_tn"])
    C, S, X = oracle.gemm_f16_tn(2, 2, 3, A, 3, B, 3)
    assert dec16(C).tolist() == worked["C_colmajor"]
    # storage of the math-view matrices in TN layout is what the fixture holds
    A2, B2 = tn_from_math(worked["A_math"], worked["B_math"])
    assert A2.tolist() == A.tolist() and B2.tolist() == B.tolist()
    # C column-major vs the math view
    assert oracle.c_as_nm(dec16(C), 2, 2, 2).T.tolist() == worked["C_math"]


def test_partial_sums_follow_k_order(worked):
    """C[0,0] runs 1, 5, 5 and C[1,1] runs 0, 5, 17 as k advances (Fig. 11.1 and
    exercise 1).  Truncating K with lda = ldb = 3 also pins the ld indexing."""
    A, B = f16(worked["A_tn"]), f16(worked["B_tn"])
    c00, c11 = [], []
    for k in (1, 2, 3):
        C, _, X = oracle.gemm_f16_tn(2, 2, k, A, 3, B, 3)
        c00.append(X[0, 0])
        c11.append(X[1, 1])
    assert c00 == worked["partial_sums"]["C00"]
    assert c11 == worked["partial_sums"]["C11"]


def test_outer_product_intermediates(worked):
    """C^(k) = C^(k-1) + A[:,k] B[k,:] (section 11.2, Fig. 11.2)."""
    A, B = f16(worked["A_tn"]), f16(worked["B_tn"])
    for k in (1, 2, 3):
        C, _, X = oracle.gemm_f16_tn(2, 2, k, A, 3, B, 3)
        assert X.T.tolist() == worked["outer_product_steps"][k]


def test_outer_product_identity_integers():
    """Sum of rank-1 updates (independent int64 numpy) equals the oracle on
    integer inputs, where every sum is exact."""
    rng = np.random.default_rng(7)
    M, N, K = 13, 11, 37
    Am = rng.integers(-8, 9, size=(M, K))
    Bm = rng.integers(-8, 9, size=(K, N))
    ref = np.zeros((M, N), np.int64)
    for k in range(K):
        ref += np.outer(Am[:, k], Bm[k, :])
    A, B = tn_from_math(Am, Bm)
    C, _, X = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    assert np.array_equal(X.T, ref.astype(np.float64))
    assert np.array_equal(dec16(oracle.c_as_nm(C, M, N, M)).T, ref.astype(np.float64))


def test_k_split_additivity():
    rng = np.random.default_rng(8)
    M, N, K, K1 = 9, 10, 40, 17
    Am = rng.integers(-5, 6, size=(M, K))
    Bm = rng.integers(-5, 6, size=(K, N))
    A, B = tn_from_math(Am, Bm)
    _, _, X = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    _, _, X1 = oracle.gemm_f16_tn(M, N, K1, A, K, B, K)
    A2 = f16(Am[:, K1:].reshape(-1))
    B2 = f16(Bm[K1:, :].T.reshape(-1))
    _, _, X2 = oracle.gemm_f16_tn(M, N, K - K1, A2, K - K1, B2, K - K1)
    assert np.array_equal(X, X1 + X2)


# --------------------------------------------------------------------------
# closed forms
@pytest.mark.parametrize("K,expect", [(1, 1.0), (7, 7.0), (2048, 2048.0), (2049, 2048.0),
                                      (4097, 4096.0), (4098, 4096.0), (4102, 4104.0)])
def test_all_ones_is_rne_of_k(K, expect):
    """C == fp16_rne(K) with all-ones operands; the expected values are the
    hand-rounded K (ties to even at 2049, 4098 and 4102)."""
    M, N = 3, 2
    A = f16(np.ones(M * K))
    B = f16(np.ones(N * K))
    C, S, X = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    assert np.all(X == K) and np.all(S == K)
    assert np.all(dec16(C) == expect)
    # a sign flip in A flips every output
    C2, _, _ = oracle.gemm_f16_tn(M, N, K, f16(-np.ones(M * K)), K, B, K)
    assert np.all(dec16(C2) == -expect)


def test_identity_returns_b():
    """A = I (M = K): each output is one product, so C == B bit for bit."""
    K = 48
    N = 20
    Bc = synth.gauss_fp16(N * K, 99)
    Bc[::7] = f16([65504.0])[0]      # extremes survive unchanged
    Bc[3] = 0x0001                   # smallest subnormal
    Bc[5] = 0x83ff                   # negative subnormal
    A = f16(np.eye(K).reshape(-1))
    C, _, _ = oracle.gemm_f16_tn(K, N, K, A, K, Bc, K)
    assert np.array_equal(C, Bc)     # column n of C is column n of B


def test_permutation_permutes_b():
    K, N = 31, 9
    rng = np.random.default_rng(3)
    perm = rng.permutation(K)
    P = np.zeros((K, K))
    P[np.arange(K), perm] = 1.0      # row m of A selects B row perm[m]
    Bc = synth.gauss_fp16(N * K, 5)
    C, _, _ = oracle.gemm_f16_tn(K, N, K, f16(P.reshape(-1)), K, Bc, K)
    Cnm = oracle.c_as_nm(C, K, N, K)
    Bnk = Bc.reshape(N, K)
    assert np.array_equal(Cnm, Bnk[:, perm])


# --------------------------------------------------------------------------
# brute force
def _exact_products(Am, Bm):
    """Exact rational C (M x N) and magnitude sums from math-view float arrays."""
    M, K = Am.shape
    N = Bm.shape[1]
    Fa = [[Fraction(float(v)) for v in row] for row in Am]
    Fb = [[Fraction(float(Bm[k, n])) for k in range(K)] for n in range(N)]
    C = [[sum((Fa[m][k] * Fb[n][k] for k in range(K)), Fraction(0)) for n in range(N)]
         for m in range(M)]
    S = [[sum((abs(Fa[m][k] * Fb[n][k]) for k in range(K)), Fraction(0)) for n in range(N)]
         for m in range(M)]
    return C, S


@pytest.mark.parametrize("M,N,K", EDGE_SHAPES)
def test_bruteforce_dyadic_edge_shapes(M, N, K):
    """Dyadic inputs j/16 (|j| <= 64): every partial sum is exact in double, so
    the oracle must equal the exact rational sum rounded once (numpy's
    double -> binary16 conversion) bit for bit."""
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    Am = rng.integers(-64, 65, size=(M, K)) / 16.0
    Bm = rng.integers(-64, 65, size=(K, N)) / 16.0
    A, B = tn_from_math(Am, Bm)
    C, S, X = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    Cx, Sx = _exact_products(Am, Bm)
    for m in range(M):
        for n in range(N):
            assert X[n, m] == float(Cx[m][n])
            assert S[n, m] == float(Sx[m][n])
            want = int(np.array([float(Cx[m][n])]).astype(np.float16).view(np.uint16)[0])
            assert int(C[m + n * M]) == want


@pytest.mark.parametrize("M,N,K", EDGE_SHAPES)
def test_bruteforce_gaussian_edge_shapes(M, N, K):
    """Gaussian fp16 inputs: the double sum is within K * 2^-53 * S of the exact
    rational sum, and C is that sum rounded once."""
    A = synth.gauss_fp16(M * K, 11 + K)
    B = synth.gauss_fp16(N * K, 12 + K)
    Am = dec16(A).reshape(M, K)
    Bm = dec16(B).reshape(N, K).T
    C, S, X = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    Cx, Sx = _exact_products(Am, Bm)
    for m in range(M):
        for n in range(N):
            ex = Cx[m][n]
            assert abs(Fraction(X[n, m]) - ex) <= Fraction(K) * Fraction(2) ** -53 * Sx[m][n]
            got = float(dec16([C[m + n * M]])[0])
            want = float(np.array([X[n, m]]).astype(np.float16)[0])
            assert got == want


def test_leading_dimensions_and_padding():
    """Padded lda/ldb/ldc: garbage in the padding changes nothing, and C's
    padding rows are left untouched."""
    M, N, K = 7, 5, 9
    lda, ldb, ldc = 13, 11, 10
    rng = np.random.default_rng(1)
    Am = rng.integers(-4, 5, size=(M, K)).astype(np.float64)
    Bm = rng.integers(-4, 5, size=(K, N)).astype(np.float64)
    A = np.full(M * lda, f16([1000.0])[0], np.uint16)
    B = np.full(N * ldb, f16([-777.0])[0], np.uint16)
    for m in range(M):
        A[m * lda: m * lda + K] = f16(Am[m])
    for n in range(N):
        B[n * ldb: n * ldb + K] = f16(Bm[:, n])
    C, _, X = oracle.gemm_f16_tn(M, N, K, A, lda, B, ldb, ldc=ldc)
    assert np.array_equal(X.T, Am @ Bm)
    Cm = C.reshape(N, ldc)
    assert np.all(Cm[:, M:] == 0)
    assert np.array_equal(dec16(Cm[:, :M]).T, Am @ Bm)


def test_sampled_equals_full():
    M, N, K = 37, 29, 53
    A = synth.gauss_fp16(M * K, 1)
    B = synth.gauss_fp16(N * K, 2)
    C, S, X = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    rng = np.random.default_rng(0)
    mi = rng.integers(0, M, 200)
    ni = rng.integers(0, N, 200)
    c, s, x = oracle.gemm_f16_tn_at(M, N, K, A, K, B, K, mi, ni)
    assert np.array_equal(c, C[mi + ni * M])
    assert np.array_equal(s, S[ni, mi]) and np.array_equal(x, X[ni, mi])


def test_against_torch_fp64_midsize():
    """Secondary sanity check (not a pin of the definition): torch fp64 matmul
    of the decoded operands agrees with X to fp64 rounding."""
    M, N, K = 64, 80, 96
    A = synth.gauss_fp16(M * K, 21)
    B = synth.gauss_fp16(N * K, 22)
    _, S, X = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    Am = torch.from_numpy(dec16(A).reshape(M, K))
    Bt = torch.from_numpy(dec16(B).reshape(N, K))
    ref = (Bt @ Am.T).numpy()        # (N, M) like X
    assert np.all(np.abs(ref - X) <= 1e-13 * S)


def test_degenerate_sizes():
    C, S, X = oracle.gemm_f16_tn(3, 2, 0, np.zeros(1, np.uint16), 1, np.zeros(1, np.uint16), 1)
    assert np.all(C[:6] == 0) and np.all(X == 0)
    C, S, X = oracle.gemm_f16_tn(0, 4, 5, np.zeros(1, np.uint16), 5, f16(np.ones(20)), 5, ldc=1)
    assert X.shape == (4, 0)
    with pytest.raises(ValueError):
        oracle.gemm_f16_tn(2, 2, 3, f16(np.ones(6)), 2, f16(np.ones(6)), 3)   # lda < K


# --------------------------------------------------------------------------
# F8 variant
E4M3 = {1.0: 0x38, 2.0: 0x40, 3.0: 0x44, 4.0: 0x48, 5.0: 0x4A, 6.0: 0x4C, 0.0: 0x00}


def bf16_of_f32(x):
    """Independent bf16 rounding: torch's float32 -> bfloat16 (RNE)."""
    t = torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().astype(np.uint16)


def test_f8_worked_example(worked):
    A = np.array([E4M3[v] for v in worked["A_tn"]], np.uint8)
    B = np.array([E4M3[v] for v in worked["B_tn"]], np.uint8)
    C, S, X = oracle.gemm_f8e4m3_tn(2, 2, 3, A, 3, B, 3, 1.0, 1.0)
    vals = torch.from_numpy(C.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert vals.tolist() == worked["C_colmajor"]


@pytest.mark.parametrize("K", [1, 64, 4097])
def test_f8_all_ones_with_scales(K):
    """All-ones codes with dequantisation factors 0.5 and 4: C = bf16(2K)."""
    A = np.full(3 * K, 0x38, np.uint8)
    B = np.full(2 * K, 0x38, np.uint8)
    C, S, X = oracle.gemm_f8e4m3_tn(3, 2, K, A, K, B, K, 0.5, 4.0)
    assert np.all(X == K) and np.all(S == 2.0 * K)
    assert np.all(C[:6] == bf16_of_f32(np.full(6, 2.0 * K)))


@pytest.mark.parametrize("M,N,K", EDGE_SHAPES)
def test_f8_bruteforce_edge_shapes(M, N, K):
    """E4M3 codes restricted to |v| in [1/8, 16] so the exact sum fits binary32;
    scales are powers of two, so C = bf16(exact * sa * sb) with one rounding."""
    rng = np.random.default_rng(K)
    codes = [q for q in range(256) if 0.125 <= abs(oracle.e4m3_decode(q)) <= 16.0]
    A = rng.choice(codes, size=M * K).astype(np.uint8)
    B = rng.choice(codes, size=N * K).astype(np.uint8)
    sa, sb = 0.25, 8.0
    C, S, X = oracle.gemm_f8e4m3_tn(M, N, K, A, K, B, K, sa, sb)
    tv = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    Am, Bn = tv[A].reshape(M, K), tv[B].reshape(N, K)
    Cx, Sx = _exact_products(Am, Bn.T)
    for m in range(M):
        for n in range(N):
            ex = Cx[m][n] * Fraction(sa) * Fraction(sb)
            assert float(ex) == np.float32(float(ex))           # fits binary32
            assert C[m + n * M] == bf16_of_f32([float(ex)])[0]
            assert S[n, m] == float(Sx[m][n] * Fraction(sa) * Fraction(sb))


def test_f8_sampled_equals_full():
    M, N, K = 21, 17, 45
    A, sa = synth.gauss_e4m3(M * K, 3)
    B, sb = synth.gauss_e4m3(N * K, 4)
    C, S, X = oracle.gemm_f8e4m3_tn(M, N, K, A, K, B, K, sa, sb)
    mi = np.arange(M * N) % M
    ni = np.arange(M * N) // M
    c, s, x = oracle.gemm_f8e4m3_tn_at(M, N, K, A, K, B, K, sa, sb, mi, ni)
    assert np.array_equal(c, C[: M * N]) and np.array_equal(x, X[ni, mi])


# --------------------------------------------------------------------------
# codecs
def test_fp16_decode_exhaustive():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_decode(int(h)) for h in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_fp16_encode_roundtrip_exhaustive():
    for h in range(65536):
        v = oracle.fp16_decode(h)
        if v != v:
            continue
        assert oracle.fp16_encode(v) == h


def test_fp16_encode_hand_ties(golden_dir):
    with open(os.path.join(golden_dir, "fp16_rne_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        assert oracle.fp16_encode(float(c["x"])) == int(c["bits"], 16), c
        assert oracle.fp16_encode(-float(c["x"])) == int(c["bits"], 16) ^ 0x8000, c


def test_fp16_encode_random_vs_numpy():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(200000) * np.exp2(rng.integers(-30, 18, 200000))
    ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle.fp16_encode(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_codec_vs_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_decode(int(h)) for h in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], ref[~nan])
    rng = np.random.default_rng(6)
    x = (rng.standard_normal(100000) * np.exp2(rng.integers(-140, 128, 100000))).astype(np.float32)
    want = bf16_of_f32(x)
    enc = np.array([oracle.bf16_encode(float(v)) for v in x], np.uint16)
    assert np.array_equal(enc, want)
    # ties: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1.0)
    assert oracle.bf16_encode(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle.bf16_encode(1.0 + 3 * 2.0 ** -8) == 0x3F82


def test_e4m3_decode_exhaustive_and_hand_cases(golden_dir):
    ref = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_decode(q) for q in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], ref[~nan])
    with open(os.path.join(golden_dir, "e4m3_cases.json")) as f:
        for c in json.load(f)["cases"]:
            v = oracle.e4m3_decode(int(c["code"], 16))
            w = float(c["value"])
            assert (v != v and w != w) or (v == w and np.signbit(v) == np.signbit(w)), c
