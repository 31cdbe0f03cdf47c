"""GPU parity of the fused attention-score epilogue (gemm_f16_tn_softmax_stats)
against the CPU oracle.

C = fp16(fp32(acc * scale)) is held to the FP16 GEMM tolerance with S scaled
by |scale|.  The statistics are formed from the FP32 scores: with an error of
at most E = 2^-16 S + 2^-23 |y| on each score (FP32 accumulation of exact
FP16 products, well inside the GEMM tolerance's 2^-12 S), row_max is within
max_n E, and row_sum within a relative 2 max_n E (the scores and the maximum
move together), plus 2^-19 for the exponentials (formed as 2^(x log2 e) with
the hardware ex2: about 2^-22 each, and the rounding of x log2 e) and 2^-22
per merge of partial sums.
Cases whose FP32 arithmetic is exact (equal scores, integer scores) are
compared bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import F16_TOL, GuardedC, assert_tol, f16_values, to_dev_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    return g


def run_stats(M, N, K, A, B, scale, stream=None):
    import dense_gemm_tn_gb300 as g
    dA, dB = to_dev_u16(A), to_dev_u16(B)
    C = GuardedC(M, N, M)
    row_max = torch.full((max(M, 1),), float("nan"), dtype=torch.float32, device="cuda")
    row_sum = torch.full((max(M, 1),), float("nan"), dtype=torch.float32, device="cuda")
    g.gemm_f16_tn_softmax_stats(M, N, K, dA, max(K, 1), dB, max(K, 1), C.ptr, max(M, 1), scale, row_max, row_sum,
                                stream)
    g.gemm_poll_device_status(stream)
    return C.nm(), row_max.cpu().numpy()[:M].astype(np.float64), row_sum.cpu().numpy()[:M].astype(np.float64)


def check(M, N, K, A, B, scale, what):
    got_c, got_max, got_sum = run_stats(M, N, K, A, B, scale)
    c_ref, mx_ref, sm_ref, S = oracle.gemm_f16_tn_softmax_stats(M, N, K, A, K, B, K, scale)
    assert_tol(f16_values(got_c), f16_values(oracle.c_as_nm(c_ref, M, N, M)), S, F16_TOL, what + " C")
    Y = np.abs(f16_values(oracle.c_as_nm(c_ref, M, N, M)))          # |scores|, close enough for a bound
    E = (2.0 ** -16 * S + 2.0 ** -23 * Y).max(axis=0)               # per row m
    assert np.all(np.abs(got_max - mx_ref) <= E + 1e-30), f"{what}: row_max off by {np.max(np.abs(got_max - mx_ref) - E)}"
    nparts = 4 * ((N + 127) // 128)
    rel = 2.0 * E + 2.0 ** -19 + (nparts + 8) * 2.0 ** -22
    err = np.abs(got_sum - sm_ref) / sm_ref
    assert np.all(err <= rel), f"{what}: row_sum rel error {err.max()} > {rel[np.argmax(err)]}"
    return got_c, got_max, got_sum


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (17, 33, 29), (300, 200, 136), (513, 640, 520), (1000, 1300, 64),
                                   (2048, 2304, 256)])
def test_matches_oracle(M, N, K):
    A = synth.gauss_fp16(M * K, 900 + M); B = synth.gauss_fp16(N * K, 901 + N)
    check(M, N, K, A, B, 1.0 / math.sqrt(K), f"{M}x{N}x{K}")


def test_qk_1024_workload():
    w = synth.WORKLOADS["qk_1024"]
    A, B, _, _ = synth.make_inputs(w)
    check(w.M, w.N, w.K, A, B, 1.0 / math.sqrt(w.K), w.name)


@pytest.mark.parametrize("N", [1, 127, 128, 129, 1000, 1024])
def test_equal_scores_exact(N):
    """All scores equal: row_max = scale K exactly and row_sum = N exactly
    (every term is exp(0) = 1, every partial sum an integer below 2^24), so a
    lost or repeated column shows as an integer difference."""
    M, K = 300, 64
    A = synth.f64_to_fp16(np.ones(M * K)); B = synth.f64_to_fp16(np.ones(N * K))
    got_c, got_max, got_sum = run_stats(M, N, K, A, B, 0.25)
    assert np.all(got_max == 16.0)
    assert np.all(got_sum == N)
    assert np.all(got_c == np.float16(16.0).view(np.uint16))


def test_integer_scores_exact_max():
    """+-1 operands with scale 1: every score is an integer, exact in FP32 and
    fp16 (|s| <= K = 512 < 2048), so C and row_max are bit-exact."""
    M, N, K = 640, 700, 512
    A = synth.sign_fp16(M * K, 31); B = synth.sign_fp16(N * K, 32)
    got_c, got_max, _ = check(M, N, K, A, B, 1.0, "pm1")
    c_ref, mx_ref, _, _ = oracle.gemm_f16_tn_softmax_stats(M, N, K, A, K, B, K, 1.0)
    assert np.array_equal(got_c, oracle.c_as_nm(c_ref, M, N, M))
    assert np.array_equal(got_max, mx_ref)


@pytest.fixture
def force_group():
    import dense_gemm_tn_gb300 as g
    yield g.gemm_debug_force_cta_group
    g.gemm_debug_force_cta_group(0)


@pytest.mark.parametrize("cta_group", [1, 2])
def test_every_tile_shape(force_group, cta_group):
    force_group(cta_group)
    M, N, K = 1100, 900, 200
    A = synth.gauss_fp16(M * K, 41); B = synth.gauss_fp16(N * K, 42)
    check(M, N, K, A, B, 0.0625, f"cta group {cta_group}")


def test_large_grid_deterministic():
    """More tiles than CTA slots (the persistent loop, several tile rows
    finishing in any order); two calls give identical bits."""
    M, N, K = 4096, 4096, 128
    A = synth.gauss_fp16(M * K, 51); B = synth.gauss_fp16(N * K, 52)
    c1, m1, s1 = check(M, N, K, A, B, 1.0 / math.sqrt(K), "4096x4096x128")
    c2, m2, s2 = run_stats(M, N, K, A, B, 1.0 / math.sqrt(K))
    assert np.array_equal(c1, c2) and np.array_equal(m1, m2) and np.array_equal(s1, s2)


def test_k_zero_negative_scale_and_empty():
    A = synth.gauss_fp16(64, 1); B = synth.gauss_fp16(64, 2)
    got_c, got_max, got_sum = run_stats(5, 7, 0, A, B, -0.5)
    assert np.all(got_max == 0.0) and np.all(got_sum == 7.0)
    assert np.all(got_c == 0x8000)                       # scale * (+0) = -0
    import dense_gemm_tn_gb300 as g
    row = torch.full((4,), float("nan"), device="cuda")
    g.gemm_f16_tn_softmax_stats(4, 0, 3, 0, 3, 0, 3, 0, 4, 1.0, row, row)     # N = 0: nothing written
    g.gemm_poll_device_status()
    assert torch.isnan(row).all().item()


def test_side_stream():
    side = torch.cuda.Stream()
    M, N, K = 700, 900, 96
    A = synth.gauss_fp16(M * K, 61); B = synth.gauss_fp16(N * K, 62)
    got_c, got_max, got_sum = run_stats(M, N, K, A, B, 0.1, stream=side)
    c_ref, mx_ref, sm_ref, S = oracle.gemm_f16_tn_softmax_stats(M, N, K, A, K, B, K, 0.1)
    assert np.allclose(got_max, mx_ref, rtol=0, atol=1e-3) and np.allclose(got_sum, sm_ref, rtol=1e-3)


def test_invalid_arguments():
    import dense_gemm_tn_gb300 as g
    x = torch.zeros(64, dtype=torch.float16, device="cuda")
    r = torch.zeros(8, device="cuda")
    with pytest.raises(g.GemmError):
        g.gemm_f16_tn_softmax_stats(8, 8, 8, x, 8, x, 8, x, 8, 1.0, None, r)
    with pytest.raises(g.GemmError):
        g.gemm_f16_tn_softmax_stats(8, 8, 8, x, 8, x, 8, x, 8, float("inf"), r, r)


def test_cuda_graph_replay():
    """The statistics' tile-row tickets return to zero after each launch, so a
    captured launch replays correctly (replays give the direct call's bits)."""
    import dense_gemm_tn_gb300 as g
    M, N, K = 2048, 2048, 128
    A = synth.gauss_fp16(M * K, 71); B = synth.gauss_fp16(N * K, 72)
    dA, dB = to_dev_u16(A), to_dev_u16(B)
    s = torch.cuda.Stream()
    out = []
    for _ in range(2):
        out.append((torch.empty((N, M), dtype=torch.float16, device="cuda"),
                    torch.empty(M, device="cuda"), torch.empty(M, device="cuda")))
    C0, mx0, sm0 = out[0]
    g.gemm_f16_tn_softmax_stats(M, N, K, dA, K, dB, K, C0, M, 0.1, mx0, sm0, s)     # warm-up
    g.gemm_poll_device_status(s)
    C1, mx1, sm1 = out[1]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.gemm_f16_tn_softmax_stats(M, N, K, dA, K, dB, K, C1, M, 0.1, mx1, sm1, s)
    for _ in range(3):
        mx1.fill_(float("nan")); sm1.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        g.gemm_poll_device_status(s)
        assert torch.equal(C1.view(torch.int16), C0.view(torch.int16))
        assert torch.equal(mx1, mx0) and torch.equal(sm1, sm0)
