"""The torch-level helpers of the binding: argument checks on the host (CPU),
and, on a GPU, results on strided views and every helper against the oracle."""
import numpy as np
import pytest
import torch

import dense_gemm_tn_gb300 as g


def test_helpers_reject_wrong_tensors_before_any_call():
    a = torch.zeros((4, 8), dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA"):
        g.f16_tn(a, a)
    with pytest.raises(ValueError, match="float16"):
        g.f16_tn(a.float(), a)
    with pytest.raises(ValueError, match="2-D"):
        g.f16_tn(a.reshape(-1), a)
    with pytest.raises(ValueError, match="unit stride"):
        g.f16_tn(torch.zeros((8, 4), dtype=torch.float16).t(), a)
    with pytest.raises(ValueError, match="uint8"):
        g.f8e4m3_tn(a, a, 1.0, 1.0)
    with pytest.raises(ValueError, match="second dimensions"):
        g.f16_tn(a, torch.zeros((4, 9), dtype=torch.float16))
    with pytest.raises(ValueError, match="shape"):
        g._output(torch.zeros((5, 4), dtype=torch.float16), 4, 4, torch.float16, None)
    with pytest.raises(ValueError, match="CUDA"):
        g.quantize_e4m3(torch.zeros((4, 8), dtype=torch.bfloat16))


@pytest.mark.gpu
def test_helpers_on_strided_views_match_the_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import oracle
    import synth
    from tests.gpu_helpers import F16_TOL, F8_TOL, assert_tol, bf16_values, f16_values
    M, N, K = 300, 520, 136
    A = synth.gauss_fp16(M * K, 81)
    B = synth.gauss_fp16(N * K, 82)
    # row-contiguous views with padded rows: lda = ldb = K + 24
    wideA = torch.zeros((M, K + 24), dtype=torch.int16, device="cuda")
    wideB = torch.zeros((N, K + 24), dtype=torch.int16, device="cuda")
    wideA[:, :K] = torch.from_numpy(A.view(np.int16).reshape(M, K)).cuda()
    wideB[:, :K] = torch.from_numpy(B.view(np.int16).reshape(N, K)).cuda()
    Av, Bv = wideA[:, :K].view(torch.float16), wideB[:, :K].view(torch.float16)
    Cref, S, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    C = g.f16_tn(Av, Bv)
    assert_tol(f16_values(C.view(torch.int16).cpu().numpy().view(np.uint16)),
               f16_values(oracle.c_as_nm(Cref, M, N, M)), S, F16_TOL, "f16_tn on views")
    Cs, mx, sm = g.f16_tn_softmax_stats(Av, Bv, 0.125)
    c_ref, mx_ref, sm_ref, S2 = oracle.gemm_f16_tn_softmax_stats(M, N, K, A, K, B, K, 0.125)
    assert_tol(f16_values(Cs.view(torch.int16).cpu().numpy().view(np.uint16)),
               f16_values(oracle.c_as_nm(c_ref, M, N, M)), S2, F16_TOL, "f16_tn_softmax_stats")
    assert np.allclose(mx.cpu().numpy(), mx_ref, rtol=0, atol=1e-3)
    assert np.allclose(sm.cpu().numpy(), sm_ref, rtol=1e-3)
    qa, sa = synth.gauss_e4m3(M * K, 83)
    qb, sb = synth.gauss_e4m3(N * K, 84)
    C8ref, S8, _ = oracle.gemm_f8e4m3_tn(M, N, K, qa, K, qb, K, sa, sb)
    dqa = torch.from_numpy(qa.reshape(M, K)).cuda()
    dqb = torch.from_numpy(qb.reshape(N, K)).cuda()
    C8 = g.f8e4m3_tn(dqa, dqb, sa, sb)
    ref8 = bf16_values(oracle.c_as_nm(C8ref, M, N, M))
    assert_tol(bf16_values(C8.view(torch.int16).cpu().numpy().view(np.uint16)), ref8, S8, F8_TOL, "f8e4m3_tn")
    scales = torch.tensor([sa, sb], dtype=torch.float32, device="cuda")
    C8d = g.f8e4m3_tn_dscale(dqa, dqb, scales[0:1], scales[1:2])
    assert torch.equal(C8d.view(torch.int16), C8.view(torch.int16))
