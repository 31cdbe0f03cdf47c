"""The lean single-CTA configurations: launches whose units are all quarter-m
or half-m units (grids of few tiles with a short K) can run a variant compiled
for two CTAs per SM, with a ring sized for such a unit (three stages for
quarters, two for halves) and 128 or 256 TMEM columns.  The library picks it
for such launches of more units than half the slots with at most 8 (halves:
4) k blocks; gemm_debug_set_lean_mode(2) forces it wherever the units allow,
(1) forbids it.  Its arithmetic is the full configuration's (the same MMAs in
the same k order), so:
  - +-1 inputs give the oracle's bits on every output;
  - Gaussian inputs give the full configuration's bits and stay within the
    FP16 / FP8 tolerances of the oracle;
  - launches issued back to back, whose CTAs share SMs with the previous
    launch's, leave each output intact.
"""
import re

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import (F8_TOL, F16_TOL, GuardedC, assert_tol, bf16_values, f16_values, run_f8, run_f16,
                               to_dev_u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    g.gemm_debug_set_skinny_mode(1)      # (shapes with N <= 64 would go to the skinny kernel)
    yield g
    g.gemm_debug_set_lean_mode(0)
    g.gemm_debug_set_skinny_mode(0)


def record(g):
    return {k: int(v) for k, v in re.findall(r"(\w+)=(\d+)", g.last_launch())}


# (M, N, K, m parts): grids of at most a quarter (half) of the slots'
# single-CTA tiles with fewer than 32 k blocks, so every tile is cut into four
# (two) m parts; run lean by mode 2 whatever their unit and k block counts
LEAN_SHAPES = [
    (1024, 1024, 128, 4),    # the QK^T block
    (512, 512, 512, 4),      # 8 k blocks through a 3-stage ring
    (256, 256, 256, 4),
    (1000, 700, 136, 4),     # ragged m, n and a zero-filled last k block
    (700, 300, 40, 4),
    (64, 8, 8, 4),
    (1024, 1024, 1984, 4),   # 31 k blocks: the 3-stage ring wraps ten times
    (300, 1, 24, 4),         # one column n
    (2048, 1024, 128, 2),    # half-m units: 2 k blocks through a 2-stage ring
    (1024, 2048, 256, 2),
    (1536, 1480, 200, 2),    # ragged n, a zero-filled last k block
]


@pytest.mark.parametrize("M,N,K,parts", LEAN_SHAPES)
def test_lean_pm1_exact(g, M, N, K, parts):
    A = synth.sign_fp16(M * K, 9700 + M % 89)
    B = synth.sign_fp16(N * K, 9701 + N % 89)
    g.gemm_debug_set_lean_mode(2)
    try:
        got = run_f16(M, N, K, A, K, B, K)
        rec = record(g)
    finally:
        g.gemm_debug_set_lean_mode(0)
    assert rec["lean"] == parts and rec["tail_mode"] == 1 and rec["split_parts"] == parts, g.last_launch()
    Cref, _, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    ref = oracle.c_as_nm(Cref, M, N, M)
    assert np.array_equal(got, ref), f"{np.sum(got != ref)} outputs differ"


@pytest.mark.parametrize("M,N,K,parts", LEAN_SHAPES)
def test_lean_gauss_equals_full_configuration(g, M, N, K, parts):
    A = synth.gauss_fp16(M * K, 9710 + K % 83)
    B = synth.gauss_fp16(N * K, 9711 + K % 83)
    g.gemm_debug_set_lean_mode(2)
    try:
        lean = run_f16(M, N, K, A, K, B, K)
        assert record(g)["lean"] == parts, g.last_launch()
    finally:
        g.gemm_debug_set_lean_mode(0)
    g.gemm_debug_set_lean_mode(1)
    try:
        full = run_f16(M, N, K, A, K, B, K)
        assert record(g)["lean"] == 0, g.last_launch()
    finally:
        g.gemm_debug_set_lean_mode(0)
    assert np.array_equal(lean, full), f"{np.sum(lean != full)} outputs differ from the full configuration"
    Cref, S, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    assert_tol(f16_values(lean), f16_values(oracle.c_as_nm(Cref, M, N, M)), S, F16_TOL, f"lean {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,parts", [(1024, 1024, 256, 4), (520, 260, 160, 4), (128, 64, 3968, 4),
                                         (2048, 1024, 512, 2)])
def test_lean_e4m3_equals_full_configuration(g, M, N, K, parts):
    A, _ = synth.gauss_e4m3(M * K, 9720 + M % 7)
    B, _ = synth.gauss_e4m3(N * K, 9721 + N % 7)
    sa, sb = 0.5, 1.5
    g.gemm_debug_set_lean_mode(2)
    try:
        lean = run_f8(M, N, K, A, K, B, K, sa, sb)
        assert record(g)["lean"] == parts, g.last_launch()
    finally:
        g.gemm_debug_set_lean_mode(0)
    g.gemm_debug_set_lean_mode(1)
    try:
        full = run_f8(M, N, K, A, K, B, K, sa, sb)
    finally:
        g.gemm_debug_set_lean_mode(0)
    assert np.array_equal(lean, full)
    Cref, S, _ = oracle.gemm_f8e4m3_tn(M, N, K, A, K, B, K, sa, sb)
    assert_tol(bf16_values(lean), bf16_values(oracle.c_as_nm(Cref, M, N, M)), S, F8_TOL, f"lean e4m3 {M}x{N}x{K}")


def test_softmax_stats_keep_the_full_configuration(g):
    """The statistics epilogue ran slower in the lean configuration: those
    launches keep the full one."""
    M, N, K = 1024, 1024, 128
    dA = to_dev_u16(synth.gauss_fp16(M * K, 9730))
    dB = to_dev_u16(synth.gauss_fp16(N * K, 9731))
    C = GuardedC(M, N, M)
    mx = torch.empty(M, device="cuda")
    sm = torch.empty(M, device="cuda")
    g.gemm_debug_set_lean_mode(0)
    g.gemm_f16_tn_softmax_stats(M, N, K, dA, K, dB, K, C.ptr, M, 0.1, mx, sm)
    g.gemm_poll_device_status(None)
    rec = record(g)
    assert rec["lean"] == 0 and rec["split_parts"] == 4, g.last_launch()


def test_lean_back_to_back_outputs_intact(g):
    """Sixteen launches issued with no synchronisation between them, each into
    its own C: a launch's CTAs become resident beside the previous launch's
    and wait for it; every output must still be the oracle's."""
    M, N, K = 1024, 1024, 128
    A = synth.sign_fp16(M * K, 9740)
    B = synth.sign_fp16(N * K, 9741)
    dA, dB = to_dev_u16(A), to_dev_u16(B)
    g.gemm_debug_set_lean_mode(0)
    outs = [GuardedC(M, N, M) for _ in range(16)]
    torch.cuda.synchronize()
    for C in outs:
        g.gemm_f16_tn(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, C.ptr, M)
    assert record(g)["lean"] == 4
    g.gemm_poll_device_status(None)
    Cref, _, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    ref = oracle.c_as_nm(Cref, M, N, M)
    for i, C in enumerate(outs):
        got = C.nm()
        assert np.array_equal(got, ref), f"launch {i}: {np.sum(got != ref)} outputs differ"


@pytest.mark.parametrize("M,N,K,want", [
    (1024, 1024, 128, 4),     # 128 quarter units, 2 k blocks
    (1024, 1024, 512, 4),     # 8 k blocks
    (2048, 1024, 128, 2),     # 128 half units
    (2048, 1024, 256, 2),     # 4 k blocks
    (1024, 1024, 1984, 0),    # 31 k blocks: the full ring's depth pays
    (2048, 1024, 512, 0),     # halves with 8 k blocks
    (512, 512, 512, 0),       # 32 units leave room beside them for the next launch
    (1024, 512, 1024, 0),     # 64 units
    (4096, 4096, 128, 0),     # a full grid of pair tiles
    (1024, 1024, 8192, 0),    # k ranges reduced in clusters
])
def test_default_choice(g, M, N, K, want):
    A = synth.sign_fp16(M * K, 9750)
    B = synth.sign_fp16(N * K, 9751)
    g.gemm_debug_set_lean_mode(0)
    got = run_f16(M, N, K, A, K, B, K)
    assert record(g)["lean"] == want, g.last_launch()
    Cref, _, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    assert np.array_equal(got, oracle.c_as_nm(Cref, M, N, M))


@pytest.mark.parametrize("M,N,K,parts", [(2048, 1024, 1024, 2), (2048, 1024, 520, 2), (1024, 1024, 1000, 4)])
def test_forced_lean_long_k_equals_full_configuration(g, M, N, K, parts):
    """Mode 2 runs half-m units lean at any K: 16 k blocks through the 2-stage
    ring (and a quarter-m grid with a zero-filled last block) give the full
    configuration's bits, and the oracle's on +-1 inputs."""
    A = synth.sign_fp16(M * K, 9760)
    B = synth.sign_fp16(N * K, 9761)
    g.gemm_debug_set_lean_mode(2)
    try:
        lean = run_f16(M, N, K, A, K, B, K)
        assert record(g)["lean"] == parts, g.last_launch()
    finally:
        g.gemm_debug_set_lean_mode(0)
    Cref, _, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    assert np.array_equal(lean, oracle.c_as_nm(Cref, M, N, M))
    Ag = synth.gauss_fp16(M * K, 9762)
    Bg = synth.gauss_fp16(N * K, 9763)
    g.gemm_debug_set_lean_mode(2)
    try:
        lean = run_f16(M, N, K, Ag, K, Bg, K)
    finally:
        g.gemm_debug_set_lean_mode(0)
    g.gemm_debug_set_lean_mode(1)
    try:
        full = run_f16(M, N, K, Ag, K, Bg, K)
        assert record(g)["lean"] == 0, g.last_launch()
    finally:
        g.gemm_debug_set_lean_mode(0)
    assert np.array_equal(lean, full)
