"""The CPython-API binding (dense_gemm_tn_gb300.fast) against the ctypes one
(dense_gemm_tn_gb300.lib): the same C functions behind both, so every output
must be bit-identical, and equal to the oracle where it is exact (+-1 inputs)
or within the FP16 / FP8 tolerances (Gaussian inputs)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import F16_TOL, GuardedC, assert_tol, f16_values, to_dev_u16, to_dev_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    if g.fast is None:
        pytest.skip("the CPython-API binding was not built (no Python.h)")
    return g


def both_f16(g, fn_name, M, N, K, A, B):
    """Runs the call through both bindings into guarded C buffers; returns both (N, M) results."""
    dA, dB = to_dev_u16(A), to_dev_u16(B)
    s = torch.cuda.current_stream().cuda_stream
    outs = []
    for binding in (g.fast, g.lib):
        C = GuardedC(M, N, M)
        st = getattr(binding, fn_name)(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, C.ptr, M, s)
        assert st == g.GEMM_OK, g.last_error()
        g.gemm_poll_device_status(None)
        outs.append(C.nm())
    return outs


@pytest.mark.parametrize("fn_name", ["gemm_f16_tn", "gemm_f16_tn_noalloc"])
@pytest.mark.parametrize("M,N,K,values", [(512, 384, 256, "pm1"), (300, 200, 136, "gauss"), (1024, 1024, 128, "gauss")])
def test_f16_calls_match_ctypes_and_oracle(g, fn_name, M, N, K, values):
    gen = synth.sign_fp16 if values == "pm1" else synth.gauss_fp16
    A, B = gen(M * K, 9101), gen(N * K, 9102)
    fast, ref_binding = both_f16(g, fn_name, M, N, K, A, B)
    assert np.array_equal(fast, ref_binding), f"{np.sum(fast != ref_binding)} outputs differ between bindings"
    Cref, S, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    ref = oracle.c_as_nm(Cref, M, N, M)
    if values == "pm1":
        assert np.array_equal(fast, ref)
    else:
        assert_tol(f16_values(fast), f16_values(ref), S, F16_TOL, fn_name)


def test_fp8_pipeline_matches_ctypes(g):
    """bf16 -> E4M3 quantisation of both operands, then the GEMM with device
    scales, once through each binding: codes, scales and C bit-identical."""
    M, N, K = 640, 384, 320
    xa = torch.from_numpy(synth.gauss_bf16(M * K, 9201).view(np.int16)).cuda()
    xb = torch.from_numpy(synth.gauss_bf16(N * K, 9202).view(np.int16)).cuda()
    s = torch.cuda.current_stream().cuda_stream
    results = []
    for binding in (g.fast, g.lib):
        qa = torch.zeros(M * K, dtype=torch.uint8, device="cuda")
        qb = torch.zeros(N * K, dtype=torch.uint8, device="cuda")
        sc = torch.zeros(2, dtype=torch.float32, device="cuda")
        assert binding.gemm_quantize_e4m3(xa.data_ptr(), g.GEMM_IN_BF16, M, K, K, qa.data_ptr(), K,
                                          sc.data_ptr(), s) == g.GEMM_OK
        assert binding.gemm_quantize_e4m3(xb.data_ptr(), g.GEMM_IN_BF16, N, K, K, qb.data_ptr(), K,
                                          sc.data_ptr() + 4, s) == g.GEMM_OK
        C = GuardedC(M, N, M)
        assert binding.gemm_f8e4m3_tn_dscale(M, N, K, qa.data_ptr(), K, qb.data_ptr(), K, C.ptr, M,
                                             sc.data_ptr(), sc.data_ptr() + 4, s) == g.GEMM_OK
        g.gemm_poll_device_status(None)
        results.append((qa.cpu().numpy(), qb.cpu().numpy(), sc.cpu().numpy(), C.nm()))
    for a, b in zip(*results):
        assert np.array_equal(a, b)


def test_fp8_scales_by_value_match_ctypes(g):
    M, N, K = 384, 256, 256
    A = synth.gauss_e4m3(M * K, 9301)[0]
    B = synth.gauss_e4m3(N * K, 9302)[0]
    dA, dB = to_dev_u8(A), to_dev_u8(B)
    s = torch.cuda.current_stream().cuda_stream
    outs = []
    for binding in (g.fast, g.lib):
        C = GuardedC(M, N, M)
        assert binding.gemm_f8e4m3_tn(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, C.ptr, M, 0.75, 1.25, s) == \
            g.GEMM_OK
        g.gemm_poll_device_status(None)
        outs.append(C.nm())
    assert np.array_equal(outs[0], outs[1])


def test_softmax_stats_match_ctypes(g):
    M, N, K = 512, 640, 128
    A, B = synth.gauss_fp16(M * K, 9401), synth.gauss_fp16(N * K, 9402)
    dA, dB = to_dev_u16(A), to_dev_u16(B)
    s = torch.cuda.current_stream().cuda_stream
    outs = []
    for binding in (g.fast, g.lib):
        C = GuardedC(M, N, M)
        mx = torch.full((M,), float("nan"), device="cuda")
        sm = torch.full((M,), float("nan"), device="cuda")
        assert binding.gemm_f16_tn_softmax_stats(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, C.ptr, M,
                                                 K ** -0.5, mx.data_ptr(), sm.data_ptr(), s) == g.GEMM_OK
        g.gemm_poll_device_status(None)
        outs.append((C.nm(), mx.cpu().numpy().view(np.uint32), sm.cpu().numpy().view(np.uint32)))
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


def test_errors_match_ctypes(g):
    """A bad argument gives the same status and message through both bindings."""
    assert g.fast.gemm_f16_tn(64, 64, 64, 0x1000, 32, 0x2000, 64, 0x3000, 64, None) == g.GEMM_ERR_INVALID_ARG
    msg = g.last_error()
    assert g.lib.gemm_f16_tn(64, 64, 64, 0x1000, 32, 0x2000, 64, 0x3000, 64, None) == g.GEMM_ERR_INVALID_ARG
    assert g.last_error() == msg
