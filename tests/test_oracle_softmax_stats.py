"""Pins of the oracle's scaled-score GEMM with softmax row statistics (CPU).

Y = scale * A B; C = binary16(Y); per row m: row_max = max_n Y[m,n] and
row_sum = sum_n exp(Y[m,n] - row_max).  The pins: closed forms (all-ones
operands, scale 0, a hand-worked 1 x 3 row), agreement with the plain GEMM
oracle (whose sums are pinned in test_oracle.py) followed by numpy's
reductions, invariance of row_sum under a shift of a row's scores, and the
degenerate sizes.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def f16(vals):
    return np.asarray(vals, np.float64).astype(np.float16).view(np.uint16)


@pytest.mark.parametrize("K,scale", [(1, 1.0), (64, 0.125), (4097, 1.0 / 64)])
def test_all_ones_closed_form(K, scale):
    M, N = 9, 13
    A = f16(np.ones(M * K)); B = f16(np.ones(N * K))
    C, mx, sm, S = oracle.gemm_f16_tn_softmax_stats(M, N, K, A, K, B, K, scale)
    assert np.all(mx == scale * K)
    assert np.all(sm == N)                        # every term is exp(0) = 1
    assert np.all(C[: M * N].view(np.float16) == np.float16(scale * K))
    assert np.all(S == scale * K)


def test_scale_zero():
    M, N, K = 4, 6, 5
    A = synth.gauss_fp16(M * K, 3); B = synth.gauss_fp16(N * K, 4)
    C, mx, sm, _ = oracle.gemm_f16_tn_softmax_stats(M, N, K, A, K, B, K, 0.0)
    assert np.all(mx == 0.0) and np.all(sm == N)
    assert np.all((C[: M * N] & 0x7FFF) == 0)


def test_hand_worked_row():
    """One query row against three keys with scores 1, 2, 3 (scale 1):
    max 3, sum e^-2 + e^-1 + e^0."""
    A = f16([1.0, 0.0])                 # M = 1, K = 2
    B = f16([1.0, 0.0, 2.0, 0.0, 3.0, 0.0])   # N = 3 columns of B, each K = 2 long
    C, mx, sm, _ = oracle.gemm_f16_tn_softmax_stats(1, 3, 2, A, 2, B, 2, 1.0)
    assert mx[0] == 3.0
    assert sm[0] == pytest.approx(math.exp(-2) + math.exp(-1) + 1.0, rel=1e-15)
    assert C[:3].view(np.float16).tolist() == [1.0, 2.0, 3.0]


@pytest.mark.parametrize("M,N,K", [(17, 33, 29), (64, 200, 128)])
def test_matches_plain_gemm_then_numpy_reductions(M, N, K):
    A = synth.gauss_fp16(M * K, 11); B = synth.gauss_fp16(N * K, 12)
    scale = 1.0 / math.sqrt(K)
    C, mx, sm, S = oracle.gemm_f16_tn_softmax_stats(M, N, K, A, K, B, K, scale)
    _, S0, X = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    Y = scale * X                                   # (N, M)
    assert np.array_equal(mx, Y.max(axis=0))
    ref_sum = np.exp(Y - Y.max(axis=0)).sum(axis=0)
    assert np.allclose(sm, ref_sum, rtol=1e-13, atol=0)
    assert np.array_equal(C[: M * N], synth.f64_to_fp16(Y.reshape(-1)))
    assert np.allclose(S, scale * S0, rtol=1e-15)


def test_row_sum_invariant_under_shift():
    """An extra k column with A[m,K] = 1 and B[K,n] = c adds scale*c to every
    score of every row: row_max moves by scale*c, row_sum does not change."""
    M, N, K = 8, 50, 16
    A = synth.gauss_fp16(M * K, 21).reshape(M, K); B = synth.gauss_fp16(N * K, 22).reshape(N, K)
    scale = 0.25
    _, mx0, sm0, _ = oracle.gemm_f16_tn_softmax_stats(M, N, K, A.reshape(-1), K, B.reshape(-1), K, scale)
    A1 = np.concatenate([A, f16(np.ones((M, 1)))], axis=1)
    B1 = np.concatenate([B, f16(np.full((N, 1), 8.0))], axis=1)
    _, mx1, sm1, _ = oracle.gemm_f16_tn_softmax_stats(M, N, K + 1, A1.reshape(-1), K + 1, B1.reshape(-1), K + 1,
                                                      scale)
    assert np.allclose(mx1, mx0 + scale * 8.0, rtol=0, atol=1e-12)
    assert np.allclose(sm1, sm0, rtol=1e-12)


def test_degenerate_sizes():
    A = f16(np.ones(12)); B = f16(np.ones(12))
    # K = 0: every score is 0
    C, mx, sm, _ = oracle.gemm_f16_tn_softmax_stats(3, 4, 0, A, 1, B, 1, 2.0)
    assert np.all(mx == 0.0) and np.all(sm == 4.0) and np.all(C[:12] == 0)
    # N = 0: no scores, the statistics stay unwritten (NaN here)
    C, mx, sm, _ = oracle.gemm_f16_tn_softmax_stats(3, 0, 4, A, 4, B, 4, 1.0)
    assert np.all(np.isnan(mx)) and np.all(np.isnan(sm))
