"""The kernel for few columns n (N <= 64): 128 rows m of A on the MMA's M side,
the N columns on its N side, k ranges of a tile meeting in a per-stream
workspace where the grid has room for them.  gemm_debug_set_skinny_mode(2)
runs it for every N <= 64, so these cases cover it whatever the library's own
choice.  +-1 inputs must give the oracle's bits; Gaussian inputs stay within
the FP16 / FP8 tolerances and give the same bits on every run (the ranges
are added in a fixed order, whichever unit arrives last)."""
import re

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import (F8_TOL, F16_TOL, GuardedC, assert_tol, bf16_values, f16_values, run_f8, run_f16,
                               sample_positions, to_dev_u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    g.gemm_debug_set_skinny_mode(2)
    yield g
    g.gemm_debug_set_skinny_mode(0)


def record(g):
    return {k: int(v) for k, v in re.findall(r"(\w+)=(\d+)", g.last_launch())}


# (M, N, K, k ranges per tile)
SHAPES = [
    (8192, 16, 8192, 2),     # the skinny workload: 64 tiles x 2 ranges
    (8192, 1, 4096, 2),      # one column
    (1000, 5, 1000, 4),      # ragged m, n and K (a zero-filled last k block)
    (4096, 64, 8192, 4),     # the widest N
    (4096, 33, 2048, 4),     # MMA N = 48
    (300, 16, 136, 1),       # too few k blocks to cut
    (128, 64, 64, 1),
    (8192, 48, 4097, 2),     # K % 8 != 0: both operands copied to a padded stride first
    (100, 3, 7, 1),
    (1, 1, 1, 1),
    (65536, 8, 256, 1),      # 512 tiles on 152 CTAs: both accumulators in turn
]


@pytest.mark.parametrize("M,N,K,parts", SHAPES)
def test_skinny_pm1_exact(g, M, N, K, parts):
    A = synth.sign_fp16(M * K, 9800 + M % 97)
    B = synth.sign_fp16(N * K, 9801 + N % 97)
    got = run_f16(M, N, K, A, K, B, K)
    rec = record(g)
    assert rec["skinny"] == 1 and rec["split_parts"] == parts, g.last_launch()
    Cref, _, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    ref = oracle.c_as_nm(Cref, M, N, M)
    assert np.array_equal(got, ref), f"{np.sum(got != ref)} outputs differ"


@pytest.mark.parametrize("M,N,K,parts", [s for s in SHAPES if s[0] * s[2] <= 8192 * 8192])
def test_skinny_gauss_within_tolerance_and_repeatable(g, M, N, K, parts):
    A = synth.gauss_fp16(M * K, 9810 + K % 89)
    B = synth.gauss_fp16(N * K, 9811 + K % 89)
    got = run_f16(M, N, K, A, K, B, K)
    assert record(g)["skinny"] == 1
    Cref, S, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    assert_tol(f16_values(got), f16_values(oracle.c_as_nm(Cref, M, N, M)), S, F16_TOL, f"skinny {M}x{N}x{K}")
    again = run_f16(M, N, K, A, K, B, K)
    assert np.array_equal(got, again)


@pytest.mark.parametrize("M,N,K", [(8192, 16, 8192), (1000, 5, 1000), (4096, 64, 2048), (512, 40, 300)])
def test_skinny_e4m3(g, M, N, K):
    A, _ = synth.gauss_e4m3(M * K, 9820 + M % 7)
    B, _ = synth.gauss_e4m3(N * K, 9821 + N % 7)
    sa, sb = 0.75, 1.25
    got = run_f8(M, N, K, A, K, B, K, sa, sb)
    assert record(g)["skinny"] == 1
    Cref, S, _ = oracle.gemm_f8e4m3_tn(M, N, K, A, K, B, K, sa, sb)
    assert_tol(bf16_values(got), bf16_values(oracle.c_as_nm(Cref, M, N, M)), S, F8_TOL, f"skinny e4m3 {M}x{N}x{K}")


def test_skinny_unaligned_c_and_padded_ldc(g):
    """C one element off 16-byte alignment with ldc > M: direct stores only
    into the M x N block (the guard bands and ldc padding stay intact)."""
    M, N, K = 1500, 12, 1024
    A = synth.sign_fp16(M * K, 9830)
    B = synth.sign_fp16(N * K, 9831)
    got = run_f16(M, N, K, A, K, B, K, ldc=M + 3, c_offset=1)
    Cref, _, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    assert np.array_equal(got, oracle.c_as_nm(Cref, M, N, M))


def test_skinny_noalloc_runs_one_range(g):
    """The no-allocation entry point has no workspace: one range per tile."""
    M, N, K = 8192, 16, 2048
    A = synth.sign_fp16(M * K, 9840)
    B = synth.sign_fp16(N * K, 9841)
    dA, dB = to_dev_u16(A), to_dev_u16(B)
    C = GuardedC(M, N, M)
    g.gemm_f16_tn_noalloc(M, N, K, dA, K, dB, K, C.ptr, M)
    g.gemm_poll_device_status(None)
    rec = record(g)
    assert rec["skinny"] == 1 and rec["split_parts"] == 1, g.last_launch()
    Cref, _, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    assert np.array_equal(C.nm(), oracle.c_as_nm(Cref, M, N, M))


def test_skinny_back_to_back_and_graph_replay(g):
    """Sixteen launches with no synchronisation in between (the tile tickets
    go back to 0 after each launch), then the same launches replayed twice
    from a CUDA graph: every output is the oracle's."""
    M, N, K = 8192, 16, 4096
    A = synth.sign_fp16(M * K, 9850)
    B = synth.sign_fp16(N * K, 9851)
    dA, dB = to_dev_u16(A), to_dev_u16(B)
    Cref, _, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    ref = oracle.c_as_nm(Cref, M, N, M)
    outs = [GuardedC(M, N, M) for _ in range(16)]
    torch.cuda.synchronize()
    for C in outs:
        g.gemm_f16_tn(M, N, K, dA, K, dB, K, C.ptr, M)
    assert record(g)["split_parts"] == 2
    g.gemm_poll_device_status(None)
    for i, C in enumerate(outs):
        assert np.array_equal(C.nm(), ref), f"launch {i}"
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    outs = [GuardedC(M, N, M) for _ in range(4)]
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.gemm_f16_tn(M, N, K, dA, K, dB, K, outs[0].ptr, M, s.cuda_stream)    # the stream's workspace
        s.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for C in outs:
                g.gemm_f16_tn(M, N, K, dA, K, dB, K, C.ptr, M, s.cuda_stream)
    for _ in range(2):
        for C in outs:
            C.buf[C.off: C.off + C.n] = np.int16(0x7E00)
        graph.replay()
        torch.cuda.synchronize()
        g.gemm_poll_device_status(None)
        for i, C in enumerate(outs):
            assert np.array_equal(C.nm(), ref), f"replayed launch {i}"


def test_skinny_not_used_beyond_64_columns_or_with_statistics(g):
    M, N, K = 4096, 65, 512
    A = synth.sign_fp16(M * K, 9860)
    B = synth.sign_fp16(N * K, 9861)
    run_f16(M, N, K, A, K, B, K)
    assert record(g)["skinny"] == 0, g.last_launch()
    M, N, K = 1024, 16, 128
    dA = to_dev_u16(synth.gauss_fp16(M * K, 9862))
    dB = to_dev_u16(synth.gauss_fp16(N * K, 9863))
    C = GuardedC(M, N, M)
    mx = torch.empty(M, device="cuda")
    sm = torch.empty(M, device="cuda")
    g.gemm_f16_tn_softmax_stats(M, N, K, dA, K, dB, K, C.ptr, M, 0.1, mx, sm)
    g.gemm_poll_device_status(None)
    assert record(g)["skinny"] == 0, g.last_launch()


@pytest.mark.parametrize("M,N,K,want", [
    (8192, 16, 2048, 1),      # 32 k blocks
    (1024, 64, 4096, 1),      # 64 k blocks
    (8192, 16, 8192, 0),      # 128 k blocks: the cluster reduce of the general kernel
    (4096, 65, 512, 0),       # more than 64 columns
])
def test_default_choice(g, M, N, K, want):
    A = synth.sign_fp16(M * K, 9870)
    B = synth.sign_fp16(N * K, 9871)
    g.gemm_debug_set_skinny_mode(0)
    try:
        got = run_f16(M, N, K, A, K, B, K)
        assert record(g)["skinny"] == want, g.last_launch()
    finally:
        g.gemm_debug_set_skinny_mode(2)
    Cref, _, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    assert np.array_equal(got, oracle.c_as_nm(Cref, M, N, M))


def test_workload_skinny_8192x16x2048(g):
    """The bench workload of the kernel, with the library's own choice, on
    sampled outputs against the oracle, and identical run to run."""
    w = synth.WORKLOADS["skinny_8192x16x2048"]
    A, B, _, _ = synth.make_inputs(w, 0)
    g.gemm_debug_set_skinny_mode(0)
    try:
        got = run_f16(w.M, w.N, w.K, A, w.K, B, w.K)
        assert record(g)["skinny"] == 1, g.last_launch()
        again = run_f16(w.M, w.N, w.K, A, w.K, B, w.K)
    finally:
        g.gemm_debug_set_skinny_mode(2)
    assert np.array_equal(got, again)
    mi, ni = sample_positions(w.M, w.N, 20000, seed=7)
    c, s, _ = oracle.gemm_f16_tn_at(w.M, w.N, w.K, A, w.K, B, w.K, mi, ni)
    assert_tol(f16_values(got[ni, mi]), f16_values(c), s, F16_TOL, "skinny_8192x16x2048")


def test_skinny_fp8_device_scales(g):
    """bf16 operands quantised to E4M3 on the device, then the GEMM with the
    scales read by the kernel (gemm_f8e4m3_tn_dscale) at N = 16: codes and
    scales as the oracle's quantiser gives them, C within the FP8 tolerance."""
    M, N, K = 4096, 16, 1024
    xa = synth.gauss_bf16(M * K, 9880)
    xb = synth.gauss_bf16(N * K, 9881)
    da = torch.from_numpy(xa.view(np.int16)).cuda()
    db = torch.from_numpy(xb.view(np.int16)).cuda()
    qa = torch.zeros(M * K, dtype=torch.uint8, device="cuda")
    qb = torch.zeros(N * K, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(2, dtype=torch.float32, device="cuda")
    g.gemm_quantize_e4m3(da, g.GEMM_IN_BF16, M, K, K, qa, K, sc.data_ptr())
    g.gemm_quantize_e4m3(db, g.GEMM_IN_BF16, N, K, K, qb, K, sc.data_ptr() + 4)
    C = GuardedC(M, N, M)
    g.gemm_f8e4m3_tn_dscale(M, N, K, qa, K, qb, K, C.ptr, M, sc.data_ptr(), sc.data_ptr() + 4)
    g.gemm_poll_device_status(None)
    assert record(g)["skinny"] == 1, g.last_launch()
    ref_qa, ref_sa = oracle.quantize_e4m3(xa, "bf16", M, K)
    ref_qb, ref_sb = oracle.quantize_e4m3(xb, "bf16", N, K)
    assert np.array_equal(qa.cpu().numpy(), ref_qa) and np.array_equal(qb.cpu().numpy(), ref_qb)
    scales = sc.cpu().numpy()
    assert scales[0] == np.float32(ref_sa) and scales[1] == np.float32(ref_sb)
    Cref, S, _ = oracle.gemm_f8e4m3_tn(M, N, K, ref_qa, K, ref_qb, K, float(scales[0]), float(scales[1]))
    assert_tol(bf16_values(C.nm()), bf16_values(oracle.c_as_nm(Cref, M, N, M)), S, F8_TOL, "skinny dscale")
