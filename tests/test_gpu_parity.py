"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bit-exact on +-1 inputs (every partial sum is an integer below 2^24, so FP32
accumulation is exact in any order and both sides round the same integer
once); within |C - C_ref| <= 2^-10 |C_ref| + 2^-12 sum_k|a b| for FP16 and
2^-7 |C_ref| + 2^-8 sum_k|a b| for FP8 with bf16 output on Gaussian inputs.
Every output buffer is NaN-poisoned and fenced by canary bands.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import (F8_TOL, F16_TOL, assert_tol, bf16_values, check_f8_full,
                               check_f16_full, f16_values, pad_rows, run_f8, run_f16, sample_positions,
                               to_dev_u8, to_dev_u16, GuardedC)

pytestmark = pytest.mark.gpu

EDGE_SHAPES = [(1, 1, 1), (3, 5, 7), (15, 17, 19), (17, 19, 23), (31, 33, 29)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    return g


def f16(vals):
    return np.asarray(vals, np.float64).astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------- page values
def test_worked_example():
    """hello-gpu ch.11 section 11.1: [[1,2,3],[4,5,6]] x [[1,0],[2,1],[0,2]]."""
    A = f16([1, 2, 3, 4, 5, 6])
    B = f16([1, 2, 0, 0, 1, 2])
    got = run_f16(2, 2, 3, A, 3, B, 3)
    assert f16_values(got).T.tolist() == [[5, 8], [14, 17]]


@pytest.mark.parametrize("M,N,K", EDGE_SHAPES)
def test_edge_shapes_gaussian(M, N, K):
    A = synth.gauss_fp16(M * K, 1000 + K)
    B = synth.gauss_fp16(N * K, 2000 + K)
    check_f16_full(M, N, K, A, B, what=f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", EDGE_SHAPES)
def test_edge_shapes_pm1_exact(M, N, K):
    A = synth.sign_fp16(M * K, 3000 + K)
    B = synth.sign_fp16(N * K, 4000 + K)
    check_f16_full(M, N, K, A, B, exact=True, what=f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", EDGE_SHAPES)
def test_edge_shapes_e4m3(M, N, K):
    A, sa = synth.gauss_e4m3(M * K, 5000 + K)
    B, sb = synth.gauss_e4m3(N * K, 6000 + K)
    check_f8_full(M, N, K, A, B, sa, sb, what=f"e4m3 {M}x{N}x{K}")


# ---------------------------------------------------------------- tile boundaries
BOUNDARY = [(255, 127, 64), (256, 128, 64), (257, 129, 65), (511, 383, 63), (513, 257, 200),
            (128, 640, 1), (300, 200, 136), (1000, 300, 1000), (64, 64, 8)]


@pytest.mark.parametrize("M,N,K", BOUNDARY)
def test_tile_boundaries_pm1_exact(M, N, K):
    A = synth.sign_fp16(M * K, 7 + M)
    B = synth.sign_fp16(N * K, 8 + N)
    check_f16_full(M, N, K, A, B, exact=True, what=f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", BOUNDARY)
def test_tile_boundaries_gaussian(M, N, K):
    A = synth.gauss_fp16(M * K, 9 + M)
    B = synth.gauss_fp16(N * K, 10 + N)
    check_f16_full(M, N, K, A, B, what=f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(257, 129, 130), (300, 200, 256), (513, 384, 1000)])
def test_tile_boundaries_e4m3(M, N, K):
    A, sa = synth.gauss_e4m3(M * K, 11 + M)
    B, sb = synth.gauss_e4m3(N * K, 12 + N)
    check_f8_full(M, N, K, A, B, sa, sb, what=f"e4m3 {M}x{N}x{K}")


# ---------------------------------------------------------------- layouts
@pytest.mark.parametrize("lda,ldb,ldc,c_off", [
    (136, 136, 304, 0),     # padded, all 16-byte aligned: TMA everywhere
    (141, 137, 303, 0),     # odd strides: repack A and B, direct C stores
    (136, 136, 300, 1),     # C base off 16-byte alignment: direct C stores
    (144, 144, 312, 0),     # K, lda, ldb, ldc aligned, M ragged: TMA stores + direct tail
])
def test_leading_dimensions(lda, ldb, ldc, c_off):
    M, N, K = 300, 200, 130
    A = synth.gauss_fp16(M * K, 21)
    B = synth.gauss_fp16(N * K, 22)
    check_f16_full(M, N, K, A, B, lda=lda, ldb=ldb, ldc=ldc, c_offset=c_off, what="ld")


@pytest.mark.parametrize("M,ldc", [(5, 8), (13, 16), (8, 8), (70, 72)])
def test_small_m_with_aligned_ldc(M, ldc):
    N, K = 40, 64
    A = synth.sign_fp16(M * K, 27)
    B = synth.sign_fp16(N * K, 28)
    check_f16_full(M, N, K, A, B, exact=True, ldc=ldc, what=f"M={M} ldc={ldc}")


def test_unaligned_operand_bases():
    M, N, K = 200, 150, 64
    A = synth.gauss_fp16(M * K, 23)
    B = synth.gauss_fp16(N * K, 24)
    check_f16_full(M, N, K, A, B, a_offset=3, b_offset=5, what="offset bases")
    A8, sa = synth.gauss_e4m3(M * K, 25)
    B8, sb = synth.gauss_e4m3(N * K, 26)
    check_f8_full(M, N, K, A8, B8, sa, sb, a_offset=7, b_offset=1, what="e4m3 offset bases")


@pytest.mark.parametrize("pad", [1, 3, 8])
@pytest.mark.parametrize("off", [0, 1, 3, 7])
def test_repack_every_row_offset_f16(pad, off):
    """Operands the TMA cannot address (K = 2100 is not a 16-byte multiple),
    with strides and bases that start rows at every 2-byte offset from 16-byte
    alignment; rows of 263 chunks span three copy segments.  The padding
    holds +-Inf, which must never reach a product."""
    M, N, K = 40, 36, 2100
    A = synth.sign_fp16(M * K, 31 + pad)
    B = synth.sign_fp16(N * K, 32 + off)
    check_f16_full(M, N, K, A, B, exact=True, lda=K + pad, ldb=K + pad + 2, a_offset=off, b_offset=(off + 5) % 8,
                   what=f"repack f16 pad {pad} off {off}")


@pytest.mark.parametrize("pad", [1, 5, 16])
@pytest.mark.parametrize("off", [0, 1, 5, 15])
def test_repack_every_row_offset_e4m3(pad, off):
    """As above for E4M3 rows (K = 2100 bytes): every byte offset occurs.
    The padding holds NaN codes."""
    M, N, K = 40, 36, 2100
    A, sa = synth.gauss_e4m3(M * K, 41 + pad)
    B, sb = synth.gauss_e4m3(N * K, 42 + off)
    check_f8_full(M, N, K, A, B, sa, sb, lda=K + pad, ldb=K + pad + 3, a_offset=off, b_offset=(off + 9) % 16,
                  what=f"repack e4m3 pad {pad} off {off}")


def test_k_zero_writes_zeros_and_empty_is_noop():
    import dense_gemm_tn_gb300 as g
    got = run_f16(5, 3, 0, np.zeros(1, np.uint16), 1, np.zeros(1, np.uint16), 1)
    assert np.all(got == 0)
    C = GuardedC(4, 1, 4)
    g.gemm_f16_tn(0, 1, 8, 0, 8, 0, 8, C.ptr, 4)
    g.gemm_f16_tn(4, 0, 8, 0, 8, 0, 8, C.ptr, 4)
    torch.cuda.synchronize()
    assert np.all(C.host() == 0x7E00)           # untouched


def test_identity_returns_b_exactly():
    K, N = 192, 160
    Bc = synth.gauss_fp16(N * K, 31)
    A = f16(np.eye(K).reshape(-1))
    got = run_f16(K, N, K, A, K, Bc, K)
    assert np.array_equal(got, Bc.reshape(N, K))


def test_all_ones_closed_form():
    """C == fp16_rne(K): 4097 rounds to 4096 (the wide workload's K)."""
    M, N, K = 260, 130, 4097
    got = run_f16(M, N, K, f16(np.ones(M * K)), K, f16(np.ones(N * K)), K)
    assert np.all(f16_values(got) == 4096.0)


def test_deterministic_and_side_stream():
    M, N, K = 700, 500, 300
    A = synth.gauss_fp16(M * K, 41)
    B = synth.gauss_fp16(N * K, 42)
    s = torch.cuda.Stream()
    g1 = run_f16(M, N, K, A, K, B, K, stream=s)
    g2 = run_f16(M, N, K, A, K, B, K)
    assert np.array_equal(g1, g2)


# ---------------------------------------------------------------- the five workloads
def test_workload_pm1_512_exact():
    w = synth.WORKLOADS["pm1_512"]
    A, B, _, _ = synth.make_inputs(w)
    check_f16_full(w.M, w.N, w.K, A, B, exact=True, what=w.name)


def test_workload_qk_1024():
    w = synth.WORKLOADS["qk_1024"]
    A, B, _, _ = synth.make_inputs(w)
    check_f16_full(w.M, w.N, w.K, A, B, what=w.name)


def _sampled_f16(w, A, B, got, exact, count=20000):
    mi, ni = sample_positions(w.M, w.N, count, seed=w.seed_a)
    c, s, _ = oracle.gemm_f16_tn_at(w.M, w.N, w.K, A, w.K, B, w.K, mi, ni)
    g = got[ni, mi]
    if exact:
        assert np.array_equal(g, c), f"{w.name}: {np.sum(g != c)} sampled outputs differ"
    else:
        assert_tol(f16_values(g), f16_values(c), s, F16_TOL, w.name)


@pytest.mark.parametrize("name", ["wide_pm1", "wide_gauss"])
def test_workload_wide(name):
    w = synth.WORKLOADS[name]
    A, B, _, _ = synth.make_inputs(w)
    got = run_f16(w.M, w.N, w.K, A, w.K, B, w.K)
    _sampled_f16(w, A, B, got, exact=(w.values == "pm1"))
    vals = f16_values(got)
    assert not np.isnan(vals).any()
    if w.values == "pm1":
        # at every output: an integer of K's parity with |C| <= K (|C| < 2048 here)
        assert np.all(np.abs(vals) <= w.K) and np.all(vals == np.round(vals))
        small = np.abs(vals) < 2048
        assert np.all((vals[small].astype(np.int64) - w.K) % 2 == 0)


def test_workload_sq_8192_sampled():
    w = synth.WORKLOADS["sq_8192"]
    A, B, _, _ = synth.make_inputs(w, 0)
    got = run_f16(w.M, w.N, w.K, A, w.K, B, w.K)
    _sampled_f16(w, A, B, got, exact=False, count=8000)
    assert not np.isnan(f16_values(got)).any()


def test_workload_ffn_8192_sampled():
    """The wide, N-heavy feed-forward shape of the ROCm blog's "Where we are"
    section (Table 16): M=8192, N=28672, K=8192."""
    w = synth.WORKLOADS["ffn_8192"]
    A, B, _, _ = synth.make_inputs(w, 0)
    got = run_f16(w.M, w.N, w.K, A, w.K, B, w.K)
    _sampled_f16(w, A, B, got, exact=False, count=8000)
    assert not np.any((got & 0x7C00) == 0x7C00), "Inf or NaN in C"


@pytest.mark.parametrize("name", ["longk_4096x512", "skinny_8192x16"])
def test_workload_long_k_sampled(name):
    """The long-K benchmark workloads (k ranges reduced in clusters) against
    the oracle on sampled outputs, within tolerance, and identical run to run."""
    w = synth.WORKLOADS[name]
    A, B, _, _ = synth.make_inputs(w, 0)
    got = run_f16(w.M, w.N, w.K, A, w.K, B, w.K)
    _sampled_f16(w, A, B, got, exact=False, count=20000)
    assert np.array_equal(got, run_f16(w.M, w.N, w.K, A, w.K, B, w.K))


def test_workload_e4m3_8192_sampled():
    w = synth.WORKLOADS["e4m3_8192"]
    A, B, sa, sb = synth.make_inputs(w, 0)
    got = run_f8(w.M, w.N, w.K, A, w.K, B, w.K, sa, sb)
    mi, ni = sample_positions(w.M, w.N, 8000, seed=w.seed_a)
    c, s, _ = oracle.gemm_f8e4m3_tn_at(w.M, w.N, w.K, A, w.K, B, w.K, sa, sb, mi, ni)
    assert_tol(bf16_values(got[ni, mi]), bf16_values(c), s, F8_TOL, w.name)
    assert not np.isnan(bf16_values(got)).any()


# ---------------------------------------------------------------- both tile shapes
@pytest.fixture
def force_group():
    import dense_gemm_tn_gb300 as g
    yield g.gemm_debug_force_cta_group
    g.gemm_debug_force_cta_group(0)


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (31, 33, 29), (257, 129, 65), (300, 200, 136), (513, 640, 520),
                                   (1000, 300, 1000), (64, 600, 64), (1100, 700, 300)])
def test_forced_cta_group_pm1_exact(force_group, cta_group, M, N, K):
    force_group(cta_group)
    A = synth.sign_fp16(M * K, 50 + M)
    B = synth.sign_fp16(N * K, 60 + N)
    check_f16_full(M, N, K, A, B, exact=True, what=f"group {cta_group} {M}x{N}x{K}")


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("M,N,K", [(300, 200, 136), (513, 640, 520), (200, 1030, 4096), (1300, 900, 700)])
def test_forced_cta_group_gaussian(force_group, cta_group, M, N, K):
    force_group(cta_group)
    A = synth.gauss_fp16(M * K, 70 + M)
    B = synth.gauss_fp16(N * K, 80 + N)
    check_f16_full(M, N, K, A, B, what=f"group {cta_group} {M}x{N}x{K}")
    A8, sa = synth.gauss_e4m3(M * K, 90 + M)
    B8, sb = synth.gauss_e4m3(N * K, 91 + N)
    check_f8_full(M, N, K, A8, B8, sa, sb, what=f"e4m3 group {cta_group} {M}x{N}x{K}")


# ---------------------------------------------------------------- split tail wave
def _launch_record():
    import re
    import dense_gemm_tn_gb300 as g
    rec = g.last_launch()
    fields = dict(re.findall(r"(\w+)=(\d+)", rec))
    return {k: int(v) for k, v in fields.items()}


@pytest.mark.parametrize("cta_group,M,N,K", [
    (2, 2000, 3000, 200),      # 8 x 12 = 96 pair tiles: one full wave + a short one
    (2, 8192, 8192, 192),      # the headline shape's 1024 tiles (13 waves + 36)
    (1, 2000, 2560, 136),      # 8 x 20 = 160 one-CTA tiles
    (2, 3000, 1700, 136),      # 12 x 7 = 84 pair tiles (one wave + 8), ragged m, n
])
def test_tail_wave_split_into_half_units(force_group, force_wide, cta_group, M, N, K):
    force_group(cta_group)
    force_wide(-1)                # the split tail of 256 x 256 tiles
    A = synth.sign_fp16(M * K, 77 + M)
    B = synth.sign_fp16(N * K, 78 + N)
    got = run_f16(M, N, K, A, K, B, K)
    rec = _launch_record()
    tiles, clusters = rec["tiles"], rec["clusters"]
    waves, rem = divmod(tiles, clusters)
    split = waves >= 1 and 0 < rem and 2 * rem <= clusters
    assert rec["units"] == (tiles + rem if split else tiles)
    if M * N <= 8_000_000:
        Cref, _, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
        assert np.array_equal(got, oracle.c_as_nm(Cref, M, N, M))
    else:
        mi, ni = sample_positions(M, N, 20000, seed=M)
        c, _, _ = oracle.gemm_f16_tn_at(M, N, K, A, K, B, K, mi, ni)
        assert np.array_equal(got[ni, mi], c)
    # with the measured 76 pair / 152 single slots of a GB300 these shapes split
    if clusters in (76, 152):
        assert split


@pytest.mark.parametrize("cta_group,M,N,K", [
    (2, 8192, 8192, 512),      # 1024 pair tiles: the 36 of the last wave split along K
    (2, 2000, 3000, 520),      # 96 pair tiles, odd k-block count (zero-padded half)
    (1, 2000, 2560, 700),      # one-CTA tiles
])
def test_split_k_tail_exact_and_deterministic(force_group, force_wide, cta_group, M, N, K):
    force_group(cta_group)
    force_wide(-1)                # the split tail of 256 x 256 tiles
    A = synth.sign_fp16(M * K, 88 + M)
    B = synth.sign_fp16(N * K, 89 + N)
    got = run_f16(M, N, K, A, K, B, K)
    rec = _launch_record()
    if rec["clusters"] in (76, 152):
        assert rec["tail_mode"] == 2, rec
    if M * N <= 8_000_000:
        Cref, _, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
        assert np.array_equal(got, oracle.c_as_nm(Cref, M, N, M))
    else:
        mi, ni = sample_positions(M, N, 20000, seed=K)
        c, _, _ = oracle.gemm_f16_tn_at(M, N, K, A, K, B, K, mi, ni)
        assert np.array_equal(got[ni, mi], c)
    # Gaussian inputs: within tolerance, and the same bits on every run
    Ag = synth.gauss_fp16(M * K, 90 + M)
    Bg = synth.gauss_fp16(N * K, 91 + N)
    g1 = run_f16(M, N, K, Ag, K, Bg, K)
    g2 = run_f16(M, N, K, Ag, K, Bg, K)
    assert np.array_equal(g1, g2)
    mi, ni = sample_positions(M, N, 20000, seed=K + 1)
    c, s, _ = oracle.gemm_f16_tn_at(M, N, K, Ag, K, Bg, K, mi, ni)
    assert_tol(f16_values(g1[ni, mi]), f16_values(c), s, F16_TOL, "split-K tail")


@pytest.mark.parametrize("wide", [-1, 1])
def test_cuda_graph_capture_and_replay(force_wide, wide):
    """After one warm-up call (which sets the kernel attributes and allocates
    the split-K buffer of the stream), the calls enqueue only kernel launches,
    so a stream can be captured into a CUDA graph and replayed; the replays
    give the same bits as direct calls.  256 x 256 tiles: 32 x 9 = 288 pair
    tiles with a split-K last wave (its tickets reset within each launch);
    256 x 512 tiles: 16 x 9 = 144."""
    import dense_gemm_tn_gb300 as g
    force_wide(wide)
    M, N, K = 8192, 2304, 1024
    A = synth.gauss_fp16(M * K, 5); B = synth.gauss_fp16(N * K, 6)
    dA, dB = to_dev_u16(A), to_dev_u16(B)
    s = torch.cuda.Stream()
    C_direct = torch.empty((N, M), dtype=torch.float16, device="cuda")
    C_graph = torch.empty((N, M), dtype=torch.float16, device="cuda")
    g.gemm_f16_tn(M, N, K, dA, K, dB, K, C_direct, M, s)        # warm-up
    g.gemm_poll_device_status(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.gemm_f16_tn(M, N, K, dA, K, dB, K, C_graph, M, s)
    for _ in range(2):
        C_graph.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        g.gemm_poll_device_status(s)
        assert torch.equal(C_graph.view(torch.int16), C_direct.view(torch.int16))


@pytest.mark.parametrize("cta_group,M,N,K,parts", [
    (0, 1024, 1024, 8192, 4),    # 32 one-CTA tiles on 152 slots: four k ranges each
    (1, 2000, 700, 4100, 3),     # ragged m, n and k (repacked): 8 x 6 = 48 tiles, three ranges
    (2, 512, 2048, 16384, 4),    # 16 pair tiles of a long K
])
def test_split_reduce_long_k(force_group, long_k_mode, cta_group, M, N, K, parts):
    """Grids of at most half the slots with a long K: every tile is cut into k
    ranges whose FP32 partials a second kernel sums in order.  +-1 inputs are
    bit-exact, Gaussian inputs within tolerance and identical run to run."""
    force_group(cta_group)
    long_k_mode(1)
    A = synth.sign_fp16(M * K, 95 + M)
    B = synth.sign_fp16(N * K, 96 + N)
    got = run_f16(M, N, K, A, K, B, K)
    rec = _launch_record()
    if rec["slots"] in (76, 152):
        assert rec["tail_mode"] == 3 and rec["split_parts"] == parts, rec
    mi, ni = sample_positions(M, N, 20000, seed=K)
    c, _, _ = oracle.gemm_f16_tn_at(M, N, K, A, K, B, K, mi, ni)
    assert np.array_equal(got[ni, mi], c)
    Ag = synth.gauss_fp16(M * K, 97 + M)
    Bg = synth.gauss_fp16(N * K, 98 + N)
    g1 = run_f16(M, N, K, Ag, K, Bg, K)
    g2 = run_f16(M, N, K, Ag, K, Bg, K)
    assert np.array_equal(g1, g2)
    c, s, _ = oracle.gemm_f16_tn_at(M, N, K, Ag, K, Bg, K, mi, ni)
    assert_tol(f16_values(g1[ni, mi]), f16_values(c), s, F16_TOL, "split-reduce")


@pytest.mark.parametrize("M,N,K,parts", [
    (512, 2048, 16384, 8),      # 8 wide tiles: eight k ranges each
    (1000, 300, 8199, 8),       # ragged m, n, k (repacked to 129 stages): 2 x 2 = 4 tiles
    (4096, 16, 8192, 8),        # a skinny problem: 8 tiles, 16 valid columns of 256
])
def test_split_reduce_on_wide_tiles(force_group, force_wide, M, N, K, parts):
    """The split-reduce of a small grid with a long K, run on 256 x 512 pair
    tiles (each part stores both halves of its partial).  +-1 inputs
    bit-exact; Gaussian inputs within tolerance and identical run to run;
    E4M3 within its tolerance."""
    force_group(2)
    force_wide(1)
    A = synth.sign_fp16(M * K, 97 + M)
    B = synth.sign_fp16(N * K, 98 + N)
    got = run_f16(M, N, K, A, K, B, K)
    rec = _launch_record()
    assert rec["wide"] == 1, rec
    if rec["slots"] == 76:
        assert rec["tail_mode"] == 3 and rec["split_parts"] == parts, rec
    mi, ni = sample_positions(M, N, 20000, seed=K + 1)
    c, _, _ = oracle.gemm_f16_tn_at(M, N, K, A, K, B, K, mi, ni)
    assert np.array_equal(got[ni, mi], c)
    Ag = synth.gauss_fp16(M * K, 99 + M)
    Bg = synth.gauss_fp16(N * K, 100 + N)
    g1 = run_f16(M, N, K, Ag, K, Bg, K)
    assert np.array_equal(g1, run_f16(M, N, K, Ag, K, Bg, K))
    c, s, _ = oracle.gemm_f16_tn_at(M, N, K, Ag, K, Bg, K, mi, ni)
    assert_tol(f16_values(g1[ni, mi]), f16_values(c), s, F16_TOL, "wide split-reduce")
    qa, sa = synth.gauss_e4m3(M * K, 101 + M)
    qb, sb = synth.gauss_e4m3(N * K, 102 + N)
    got8 = run_f8(M, N, K, qa, K, qb, K, sa, sb)
    c, s, _ = oracle.gemm_f8e4m3_tn_at(M, N, K, qa, K, qb, K, sa, sb, mi, ni)
    assert_tol(bf16_values(got8[ni, mi]), bf16_values(c), s, F8_TOL, "wide split-reduce e4m3")


def test_split_reduce_e4m3_host_and_device_scales(long_k_mode):
    import dense_gemm_tn_gb300 as g
    long_k_mode(1)
    M, N, K = 1024, 1024, 8192
    qa, sa = synth.gauss_e4m3(M * K, 81)
    qb, sb = synth.gauss_e4m3(N * K, 82)
    got = run_f8(M, N, K, qa, K, qb, K, sa, sb)
    rec = _launch_record()
    if rec["slots"] in (76, 152):
        assert rec["tail_mode"] == 3, rec
    mi, ni = sample_positions(M, N, 20000, seed=3)
    c, s, _ = oracle.gemm_f8e4m3_tn_at(M, N, K, qa, K, qb, K, sa, sb, mi, ni)
    assert_tol(bf16_values(got[ni, mi]), bf16_values(c), s, F8_TOL, "split-reduce e4m3")
    dA, dB = to_dev_u8(qa), to_dev_u8(qb)
    scales = torch.tensor([sa, sb], dtype=torch.float32, device="cuda")
    C = GuardedC(M, N, M)
    g.gemm_f8e4m3_tn_dscale(M, N, K, dA, K, dB, K, C.ptr, M, scales.data_ptr(), scales.data_ptr() + 4)
    g.gemm_poll_device_status()
    assert np.array_equal(C.nm(), got)


@pytest.mark.parametrize("cta_group,M,N,K,parts", [
    (0, 1024, 1024, 128, 4),     # 32 one-CTA tiles on 152 slots: each cut into four 64-row m ranges
    (0, 2048, 1024, 256, 2),     # 64 one-CTA tiles: two 128-row m ranges each
    (0, 900, 300, 77, 4),        # ragged m (the last range of the last tile row lies past M), repacked K
    (0, 1, 1000, 40, 4),         # one row m: three of each tile's four ranges are empty
    (2, 1024, 1024, 128, 4),     # forced CTA pairs: 32 A rows per CTA, MMA N = 64
    (2, 700, 1000, 136, 4),      # forced CTA pairs, ragged m and n
])
def test_small_grid_m_parts(force_group, cta_group, M, N, K, parts):
    """Grids of at most half the slots with a short K: every tile's m range is
    cut into 2 or 4 units.  +-1 inputs are bit-exact, Gaussian inputs within
    tolerance, and E4M3 runs the same cut."""
    force_group(cta_group)
    A = synth.sign_fp16(M * K, 60 + M)
    B = synth.sign_fp16(N * K, 61 + N)
    check_f16_full(M, N, K, A, B, exact=True, what=f"m parts {M}x{N}x{K}")
    rec = _launch_record()
    if rec["slots"] in (76, 152):
        assert rec["tail_mode"] == 1 and rec["split_parts"] == parts and rec["tail_start"] == 0, rec
        assert rec["units"] == rec["tiles"] * parts, rec
    Ag = synth.gauss_fp16(M * K, 62 + M)
    Bg = synth.gauss_fp16(N * K, 63 + N)
    check_f16_full(M, N, K, Ag, Bg, what=f"m parts gaussian {M}x{N}x{K}")
    qa, sa = synth.gauss_e4m3(M * K, 64 + M)
    qb, sb = synth.gauss_e4m3(N * K, 65 + N)
    check_f8_full(M, N, K, qa, qb, sa, sb, what=f"m parts e4m3 {M}x{N}x{K}")


# ---------------------------------------------------------------- 256 x 512 pair tiles
@pytest.fixture
def force_wide():
    import dense_gemm_tn_gb300 as g
    yield g.gemm_debug_force_wide_tiles
    g.gemm_debug_force_wide_tiles(0)
    g.gemm_debug_force_cta_group(0)


@pytest.mark.parametrize("M,N,K,cut", [
    (1, 1, 1, False),
    (257, 129, 65, False),       # one ragged tile
    (513, 640, 520, False),      # ragged m across the two halves, ragged k
    (300, 1000, 4097, False),    # K not a 16-byte multiple: repacked operands
    (4096, 2560, 136, True),     # 8 x 10 = 80 tiles: the last 4 cut into m halves
    (3000, 12289, 136, False),   # 6 x 49 = 294 tiles: a last wave too full to cut
])
def test_wide_tiles_pm1_exact(force_group, force_wide, M, N, K, cut):
    """CTA pairs computing 256 x 512 tiles (two N = 256 halves), forced on shapes
    the library would give other tiles: +-1 inputs bit-exact, Gaussian inputs
    within tolerance, E4M3 too."""
    import dense_gemm_tn_gb300 as g
    force_group(2)
    force_wide(1)
    A = synth.sign_fp16(M * K, 66 + M)
    B = synth.sign_fp16(N * K, 67 + N)
    if M * N <= 4_000_000:
        check_f16_full(M, N, K, A, B, exact=True, what=f"wide {M}x{N}x{K}")
    else:
        got = run_f16(M, N, K, A, K, B, K)
        mi, ni = sample_positions(M, N, 20000, seed=M + K)
        c, _, _ = oracle.gemm_f16_tn_at(M, N, K, A, K, B, K, mi, ni)
        assert np.array_equal(got[ni, mi], c)
    rec = _launch_record()
    assert rec["wide"] == 1 and rec["ctas_per_cluster"] == 2, rec
    if rec["slots"] == 76:
        assert (rec["tail_mode"] == 1) == cut, rec
        if cut:
            assert rec["units"] == rec["tiles"] + rec["tiles"] % 76, rec
    if M * N <= 4_000_000:
        Ag = synth.gauss_fp16(M * K, 68 + M)
        Bg = synth.gauss_fp16(N * K, 69 + N)
        check_f16_full(M, N, K, Ag, Bg, what=f"wide gaussian {M}x{N}x{K}")
        qa, sa = synth.gauss_e4m3(M * K, 70 + M)
        qb, sb = synth.gauss_e4m3(N * K, 71 + N)
        check_f8_full(M, N, K, qa, qb, sa, sb, what=f"wide e4m3 {M}x{N}x{K}")
        assert _launch_record()["wide"] == 1


@pytest.mark.parametrize("rows", [2, 6, 16])
def test_raster_group_heights_exact(rows):
    """Other raster group heights reorder the tiles only: +-1 inputs give the
    same bits (a short last group included: 11 tile rows)."""
    import dense_gemm_tn_gb300 as g
    M, N, K = 2816, 1536, 192
    A = synth.sign_fp16(M * K, 111)
    B = synth.sign_fp16(N * K, 112)
    g.gemm_debug_set_raster_group(rows)
    try:
        check_f16_full(M, N, K, A, B, exact=True, what=f"raster group {rows}")
    finally:
        g.gemm_debug_set_raster_group(0)


def test_wide_tiles_chosen_by_estimate():
    """The library picks 256 x 512 tiles where its estimate of the launch's
    length says they are faster (a long K: the wide tile's exposed epilogue is
    a small part of it) and 256 x 256 tiles elsewhere (a short K, or a grid
    whose wide tiles would leave most of a wave idle), on 76 pair slots."""
    import dense_gemm_tn_gb300 as g
    cases = [((8192, 8192, 2048), 1), ((3072, 3072, 8192), 1), ((8192, 8192, 256), 0), ((2048, 3072, 64), 0)]
    for (M, N, K), want in cases:
        A = synth.sign_fp16(M * K, 5)
        B = synth.sign_fp16(N * K, 6)
        got = run_f16(M, N, K, A, K, B, K)
        rec = _launch_record()
        if rec["slots"] == 76 and rec["ctas_per_cluster"] == 2:
            assert rec["wide"] == want, (M, N, K, rec)
        mi, ni = sample_positions(M, N, 5000, seed=K)
        c, _, _ = oracle.gemm_f16_tn_at(M, N, K, A, K, B, K, mi, ni)
        assert np.array_equal(got[ni, mi], c)


LAYOUTS = [(136, 136, 304, 0, 0, 0), (141, 137, 303, 0, 0, 0), (136, 136, 300, 1, 0, 0), (144, 144, 312, 0, 0, 0),
           (130, 130, 300, 0, 3, 5)]      # lda, ldb, ldc, C offset, A offset, B offset (elements)


@pytest.mark.parametrize("cta_group,wide", [(1, -1), (2, -1), (2, 1)])
def test_layouts_on_every_tile_shape(force_group, force_wide, cta_group, wide):
    """Padded, odd and unaligned leading dimensions and bases (TMA in place,
    repacked operands, direct C stores) on each tile shape, FP16 and E4M3."""
    force_group(cta_group)
    force_wide(wide)
    M, N, K = 300, 700, 130
    A = synth.gauss_fp16(M * K, 31)
    B = synth.gauss_fp16(N * K, 32)
    A8, sa = synth.gauss_e4m3(M * K, 33)
    B8, sb = synth.gauss_e4m3(N * K, 34)
    for lda, ldb, ldc, c_off, a_off, b_off in LAYOUTS:
        what = f"group {cta_group} wide {wide} ld {lda},{ldb},{ldc} offsets {c_off},{a_off},{b_off}"
        check_f16_full(M, N, K, A, B, lda=lda, ldb=ldb, ldc=ldc, c_offset=c_off, a_offset=a_off, b_offset=b_off,
                       what=what)
        if cta_group == 2:
            assert _launch_record()["wide"] == (1 if wide == 1 else 0)
        check_f8_full(M, N, K, A8, B8, sa, sb, lda=lda, ldb=ldb, ldc=ldc, c_offset=c_off, a_offset=a_off,
                      b_offset=b_off, what="e4m3 " + what)


# ---------------------------------------------------------------- k order by wave
@pytest.fixture
def k_order():
    import dense_gemm_tn_gb300 as g
    yield g.gemm_debug_set_k_order
    g.gemm_debug_set_k_order(0)


@pytest.mark.parametrize("cta_group,wide,M,N,K", [
    (2, 1, 8192, 8192, 1000),    # 512 wide tiles: 6 waves + 56; a ragged last k block read first
    (2, -1, 4096, 4096, 520),    # 256 pair tiles: 3 waves + 28, the last 28 split along K (forward)
    (1, -1, 2048, 3000, 136),    # one-CTA tiles, 8 x 24 = 192 on 152 slots
])
def test_k_order_reversed_on_odd_waves(force_group, force_wide, k_order, cta_group, wide, M, N, K):
    """Whole tiles of odd waves walking their k blocks backwards: the same
    bits on +-1 inputs as the oracle; Gaussian inputs within tolerance,
    identical run to run, and within tolerance of the forward order."""
    force_group(cta_group)
    force_wide(wide)
    A = synth.sign_fp16(M * K, 300 + M)
    B = synth.sign_fp16(N * K, 301 + N)
    mi, ni = sample_positions(M, N, 20000, seed=M + K)
    c, _, _ = oracle.gemm_f16_tn_at(M, N, K, A, K, B, K, mi, ni)
    for mode in (2, 1):
        k_order(mode)
        got = run_f16(M, N, K, A, K, B, K)
        assert np.array_equal(got[ni, mi], c), f"k order {mode}"
    Ag = synth.gauss_fp16(M * K, 302 + M)
    Bg = synth.gauss_fp16(N * K, 303 + N)
    k_order(2)
    g1 = run_f16(M, N, K, Ag, K, Bg, K)
    assert np.array_equal(g1, run_f16(M, N, K, Ag, K, Bg, K))
    c, s, _ = oracle.gemm_f16_tn_at(M, N, K, Ag, K, Bg, K, mi, ni)
    assert_tol(f16_values(g1[ni, mi]), f16_values(c), s, F16_TOL, "k order 2")
    qa, sa = synth.gauss_e4m3(M * K, 304 + M)
    qb, sb = synth.gauss_e4m3(N * K, 305 + N)
    got8 = run_f8(M, N, K, qa, K, qb, K, sa, sb)
    c8, s8, _ = oracle.gemm_f8e4m3_tn_at(M, N, K, qa, K, qb, K, sa, sb, mi, ni)
    assert_tol(bf16_values(got8[ni, mi]), bf16_values(c8), s8, F8_TOL, "k order 2 e4m3")


# ---------------------------------------------------------------- k ranges reduced in a cluster
@pytest.fixture
def long_k_mode():
    import dense_gemm_tn_gb300 as g
    yield g.gemm_debug_set_long_k_mode
    g.gemm_debug_set_long_k_mode(0)


@pytest.mark.parametrize("M,N,K,parts", [
    (1024, 1024, 8192, (4,)),      # 32 one-CTA tiles: clusters of four k ranges
    (4096, 512, 8192, (2,)),       # 64 tiles: clusters of two
    (2000, 700, 4100, (2, 3)),     # ragged m, n, k (repacked): 8 x 6 = 48 tiles; clusters of three if 48 fit
    (8192, 16, 8192, (4,)),        # skinny: 16 valid columns n of 128 per tile, only those exchanged
    (4096, 40, 8192, (4,)),        # 40 columns n: one warp whole, one in part, two with none (they skip)
    (300, 100, 16384, (4,)),       # 2 tiles: the split-reduce would take 8 ranges, a cluster 4
    (1280, 1024, 8192, (2, 3)),    # 5 x 8 = 40 tiles: clusters of three where 40 of them fit at once
])
@pytest.mark.parametrize("group", [1, 2])
def test_cluster_reduce_long_k(force_group, long_k_mode, M, N, K, parts, group):
    """Small grids with a long K, on single CTAs (group 1) or CTA pairs (group
    2), the k ranges of each tile in one cluster that adds the FP32 partials
    through distributed shared memory: +-1 inputs bit-exact against the
    oracle, Gaussian inputs within tolerance and identical run to run, E4M3
    with host and device scales."""
    import dense_gemm_tn_gb300 as g
    force_group(group)
    long_k_mode(2)
    if group == 2:
        parts = (2, 3, 4)      # as many ranges as pair clusters fit (up to 8 CTAs per cluster)
    A = synth.sign_fp16(M * K, 400 + M)
    B = synth.sign_fp16(N * K, 401 + N)
    got = run_f16(M, N, K, A, K, B, K)
    rec = _launch_record()
    if rec["slots"] == 152 // group and rec["tail_mode"] == 4:
        assert rec["split_parts"] in parts, rec
        assert rec["ctas_per_cluster"] == group * rec["split_parts"], rec
        assert rec["grid"] == group * rec["split_parts"] * rec["tiles"], rec
    elif group == 1 and rec["slots"] == 152:
        assert rec["tail_mode"] == 4, rec
    if M * N <= 2_000_000:
        Cref, _, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
        assert np.array_equal(got, oracle.c_as_nm(Cref, M, N, M))
    else:
        mi, ni = sample_positions(M, N, 20000, seed=K + M)
        c, _, _ = oracle.gemm_f16_tn_at(M, N, K, A, K, B, K, mi, ni)
        assert np.array_equal(got[ni, mi], c)
    mi, ni = sample_positions(M, N, 20000, seed=K + N)
    Ag = synth.gauss_fp16(M * K, 402 + M)
    Bg = synth.gauss_fp16(N * K, 403 + N)
    g1 = run_f16(M, N, K, Ag, K, Bg, K)
    assert np.array_equal(g1, run_f16(M, N, K, Ag, K, Bg, K))
    c, s, _ = oracle.gemm_f16_tn_at(M, N, K, Ag, K, Bg, K, mi, ni)
    assert_tol(f16_values(g1[ni, mi]), f16_values(c), s, F16_TOL, "cluster reduce")
    qa, sa = synth.gauss_e4m3(M * K, 404 + M)
    qb, sb = synth.gauss_e4m3(N * K, 405 + N)
    got8 = run_f8(M, N, K, qa, K, qb, K, sa, sb)
    c8, s8, _ = oracle.gemm_f8e4m3_tn_at(M, N, K, qa, K, qb, K, sa, sb, mi, ni)
    assert_tol(bf16_values(got8[ni, mi]), bf16_values(c8), s8, F8_TOL, "cluster reduce e4m3")
    dA, dB = to_dev_u8(qa), to_dev_u8(qb)
    scales = torch.tensor([sa, sb], dtype=torch.float32, device="cuda")
    C = GuardedC(M, N, M)
    g.gemm_f8e4m3_tn_dscale(M, N, K, dA, K, dB, K, C.ptr, M, scales.data_ptr(), scales.data_ptr() + 4)
    g.gemm_poll_device_status()
    assert np.array_equal(C.nm(), got8)


def test_cluster_reduce_matches_split_reduce_on_pm1(force_group, long_k_mode):
    """The two ways of adding up k ranges give the same bits on +-1 inputs."""
    force_group(1)
    M, N, K = 1024, 1024, 8192
    A = synth.sign_fp16(M * K, 410)
    B = synth.sign_fp16(N * K, 411)
    long_k_mode(1)
    a = run_f16(M, N, K, A, K, B, K)
    assert _launch_record()["tail_mode"] in (3, 0, 1)
    long_k_mode(2)
    b = run_f16(M, N, K, A, K, B, K)
    assert np.array_equal(a, b)



def test_clock_probe_counts_launches_and_leaves_results_alone():
    """The measurement hook: each launch adds its first CTA's SM cycles and
    nanoseconds and one launch to the counters; results are unchanged."""
    import dense_gemm_tn_gb300 as g
    M, N, K = 2048, 2048, 1024
    A = synth.sign_fp16(M * K, 600)
    B = synth.sign_fp16(N * K, 601)
    ref = run_f16(M, N, K, A, K, B, K)
    counters = torch.zeros(3, dtype=torch.int64, device="cuda")
    g.gemm_debug_set_clock_probe(counters.data_ptr())
    try:
        got = [run_f16(M, N, K, A, K, B, K) for _ in range(3)]
    finally:
        g.gemm_debug_set_clock_probe(None)
    cycles, ns, launches = (int(x) for x in counters.tolist())
    assert launches == 3 and cycles > 0 and ns > 0
    assert 300.0 < cycles / ns * 1e3 < 2500.0, cycles / ns
    for x in got:
        assert np.array_equal(x, ref)
    run_f16(M, N, K, A, K, B, K)                 # off again: the counters stay
    assert int(counters[2].item()) == 3



def test_long_k_small_grid_tile_choice():
    """Small grids with a long K: CTA pairs in k-range clusters where they keep
    at least as many SMs busy as single CTAs would, single CTAs otherwise
    (checked on a GB300's 152 / 76 slots); +-1 inputs bit-exact on samples."""
    cases = [((4096, 512, 8192), 2), ((2048, 1024, 8192), 2), ((1024, 1024, 8192), 1), ((8192, 16, 8192), 1)]
    for (M, N, K), want in cases:
        A = synth.sign_fp16(M * K, 620 + M)
        B = synth.sign_fp16(N * K, 621 + N)
        got = run_f16(M, N, K, A, K, B, K)
        rec = _launch_record()
        if rec["slots"] in (76, 152) and rec["tail_mode"] == 4:
            assert rec["ctas_per_cluster"] == want * rec["split_parts"], ((M, N, K), rec)
        mi, ni = sample_positions(M, N, 10000, seed=M + N)
        c, _, _ = oracle.gemm_f16_tn_at(M, N, K, A, K, B, K, mi, ni)
        assert np.array_equal(got[ni, mi], c), (M, N, K)
