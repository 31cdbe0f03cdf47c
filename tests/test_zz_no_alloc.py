"""gemm_f16_tn_noalloc: the FP16 entry point for callers that cannot let the
library allocate device memory -- programs that hand out all device memory
from their own pool or fixed budget, or hot paths where the implicit device
synchronisation of cudaMalloc / cudaFree is not acceptable.  Instead of a
cudaMalloc'd workspace it copies unaligned operands into a fixed array in
the library's device image.

Its results must match gemm_f16_tn's within the FP16 tolerance of the other
tests, on two calls in a row (the second reuses the array the first wrote).
This file is named so pytest collects it last."""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_helpers import F16_TOL, assert_tol, f16_values, pad_rows, to_dev_u16

pytestmark = pytest.mark.gpu


def _run(entry, M, N, K, dA, a_off, lda, dB, b_off, ldb):
    C = torch.full((N, M), float("nan"), dtype=torch.float16, device="cuda")
    entry(M, N, K, dA.data_ptr() + 2 * a_off, lda, dB.data_ptr() + 2 * b_off, ldb, C.data_ptr(), M)
    return C


@pytest.mark.parametrize("tiles", ["auto", "256x512 pairs"])
def test_noalloc_matches_gemm_f16_tn_on_two_calls(tiles):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    if tiles != "auto":
        g.gemm_debug_force_cta_group(2)
        g.gemm_debug_force_wide_tiles(1)
    try:
        _compare_two_calls(g)
    finally:
        g.gemm_debug_force_cta_group(0)
        g.gemm_debug_force_wide_tiles(0)


def _compare_two_calls(g):
    cases = [
        # M, N, K, lda, ldb, a_off, b_off: every case needs an operand copy
        (300, 200, 130, 141, 137, 0, 0),     # K and strides not 16-byte multiples
        (257, 129, 72, 72, 72, 3, 5),        # aligned K and strides, unaligned bases
    ]
    for i, (M, N, K, lda, ldb, a_off, b_off) in enumerate(cases):
        A = synth.gauss_fp16(M * K, 900 + i)
        B = synth.gauss_fp16(N * K, 950 + i)
        Ap = np.concatenate([np.zeros(a_off, np.uint16), pad_rows(A, M, K, lda, 0x7C00)])
        Bp = np.concatenate([np.zeros(b_off, np.uint16), pad_rows(B, N, K, ldb, 0xFC00)])
        dA, dB = to_dev_u16(Ap), to_dev_u16(Bp)
        ref = _run(g.gemm_f16_tn, M, N, K, dA, a_off, lda, dB, b_off, ldb)
        got = _run(g.gemm_f16_tn_noalloc, M, N, K, dA, a_off, lda, dB, b_off, ldb)
        g.gemm_poll_device_status()
        r = ref.float().cpu().numpy().astype(np.float64)
        o = got.float().cpu().numpy().astype(np.float64)
        Am = f16_values(A).reshape(M, K)
        Bn = f16_values(B).reshape(N, K)
        S = np.abs(Bn) @ np.abs(Am).T                      # (N, M): sum_k |a b|
        assert_tol(o, r, S, F16_TOL, f"noalloc call {i + 1}")


def test_noalloc_rejects_copies_beyond_its_array():
    import dense_gemm_tn_gb300 as g
    # 2 operands x 4096 rows x roundup(4097, 8) x 2 bytes = 64 MiB > 32 MiB;
    # rejected before anything touches the (dummy, never dereferenced) pointers
    st = g.lib.gemm_f16_tn_noalloc(4096, 4096, 4097, 0x1000, 4097, 0x2000, 4097, 0x3000, 4096, None)
    assert st == g.GEMM_ERR_INVALID_ARG
    assert "scratch" in g.last_error()
