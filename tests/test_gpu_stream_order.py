"""Stream order across back-to-back launches.

Every GEMM launch is a programmatic dependent of the previous kernel on its
stream: its CTAs may start while that kernel still runs, and it lets the next
kernel start early too.  These tests chain calls through each other's buffers
with no host synchronisation in between and check every result bit for bit
against the oracle:
  - read after write: each GEMM's C is the next GEMM's A;
  - write after read: a GEMM overwrites the operand the previous GEMM reads;
  - the same through the split-reduce pair of kernels and through small grids
    whose CTAs leave most SMs free for the next launch to start on.
Operands are small integers (signs, and sparse sign matrices that keep the
sums bounded), so every sum is exact in FP32 and both sides round the same
integer once.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import to_dev_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    return g


def f16(vals):
    return np.asarray(vals, np.float64).astype(np.float16).view(np.uint16)


def sparse_signs(rows, K, per_row, seed):
    """rows x K codes with `per_row` entries of +-1 per row, the rest 0."""
    rng = np.random.default_rng(seed)
    out = np.zeros((rows, K), np.float64)
    for r in range(rows):
        cols = rng.choice(K, size=min(per_row, K), replace=False)
        out[r, cols] = rng.choice([-1.0, 1.0], size=cols.size)
    return f16(out.reshape(-1))


def ref_nm(M, N, K, A, B):
    C, _, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    return oracle.c_as_nm(C, M, N, M)        # (N, M): row-major, the next GEMM's A


# (M, N, K) of each link: link j's A is link j-1's C viewed as (N_{j-1}) x (M_{j-1}) row-major,
# so M_j = N_{j-1} and K_j = M_{j-1}.
CHAINS = {
    "small grids": [(1024, 1024, 64), (1024, 512, 1024), (512, 768, 1024), (768, 256, 512), (256, 1024, 768)],
    # 96 pair tiles (a half-m tail), 96 pair tiles (a split-K tail), then a split-reduce grid
    "pairs and split tails": [(2048, 3072, 128), (3072, 2048, 2048), (2048, 1024, 3072)],
    "split-reduce": [(512, 512, 8192), (512, 1024, 512), (1024, 512, 512)],
}


@pytest.mark.parametrize("name", sorted(CHAINS))
def test_read_after_write_chain(name):
    import dense_gemm_tn_gb300 as g
    links = CHAINS[name]
    M0, _, K0 = links[0]
    A = synth.sign_fp16(M0 * K0, 7001)
    Bs = []
    for j, (M, N, K) in enumerate(links):
        Bs.append(synth.sign_fp16(N * K, 7100 + j) if j == 0 else sparse_signs(N, K, 6, 7100 + j))
    refs = []
    a = A
    for (M, N, K), B in zip(links, Bs):
        r = ref_nm(M, N, K, a, B)
        refs.append(r)
        a = r.reshape(-1)
    s = torch.cuda.Stream()
    dB = [to_dev_u16(B) for B in Bs]
    for rep in range(3):
        outs = [torch.empty((N, M), dtype=torch.int16, device="cuda") for (M, N, K) in links]
        for o in outs:
            o.fill_(0x7E00)                                     # NaN poison
        dA = to_dev_u16(A)
        torch.cuda.synchronize()                                # uploads done before the side stream starts
        src = dA
        with torch.cuda.stream(s):
            for (M, N, K), b, o in zip(links, dB, outs):         # no host synchronisation in the chain
                g.gemm_f16_tn(M, N, K, src, K, b, K, o, M, s)
                src = o
        g.gemm_poll_device_status(s)
        for j, (o, r) in enumerate(zip(outs, refs)):
            got = o.cpu().numpy().view(np.uint16)
            assert np.array_equal(got, r), f"{name}: link {j} (rep {rep}): {np.sum(got != r)} outputs differ"


def test_write_after_read():
    """GEMM 1 reads X as A; GEMM 2, launched right behind it, writes its C into
    X.  GEMM 1 must see X as it was; X must end up holding GEMM 2's C."""
    import dense_gemm_tn_gb300 as g
    M1, N1, K1 = 1024, 1024, 256          # small grid: most SMs free for GEMM 2 to start on
    M2, N2, K2 = 512, 512, 64             # its C (512 x 512) fits in X (1024 x 256)
    X0 = synth.sign_fp16(M1 * K1, 7201)
    B1 = synth.sign_fp16(N1 * K1, 7202)
    A2 = synth.sign_fp16(M2 * K2, 7203)
    B2 = synth.sign_fp16(N2 * K2, 7204)
    ref1 = ref_nm(M1, N1, K1, X0, B1)
    ref2 = ref_nm(M2, N2, K2, A2, B2)
    s = torch.cuda.Stream()
    dB1, dA2, dB2 = to_dev_u16(B1), to_dev_u16(A2), to_dev_u16(B2)
    for rep in range(5):
        X = to_dev_u16(X0)
        C1 = torch.full((N1, M1), 0x7E00, dtype=torch.int16, device="cuda")
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.gemm_f16_tn(M1, N1, K1, X, K1, dB1, K1, C1, M1, s)
            g.gemm_f16_tn(M2, N2, K2, dA2, K2, dB2, K2, X, M2, s)     # overwrites GEMM 1's A
        g.gemm_poll_device_status(s)
        got1 = C1.cpu().numpy().view(np.uint16)
        got2 = X.cpu().numpy().view(np.uint16)[: M2 * N2].reshape(N2, M2)
        assert np.array_equal(got1, ref1), f"rep {rep}: GEMM 1 saw X after GEMM 2 wrote it"
        assert np.array_equal(got2, ref2), f"rep {rep}: GEMM 2's C"


def test_softmax_stats_then_gemm_on_its_scores():
    """The scaled scores of gemm_f16_tn_softmax_stats feed the next GEMM at once."""
    import dense_gemm_tn_gb300 as g
    M, N, K = 512, 640, 128
    A = synth.sign_fp16(M * K, 7301)
    B = synth.sign_fp16(N * K, 7302)
    C_ref, mx_ref, sm_ref, _ = oracle.gemm_f16_tn_softmax_stats(M, N, K, A, K, B, K, 0.5)
    scores = oracle.c_as_nm(C_ref, M, N, M)                  # (N, M) = the next A (M' = N, K' = M)
    B2 = sparse_signs(256, M, 6, 7303)
    ref2 = ref_nm(N, 256, M, scores.reshape(-1), B2)
    s = torch.cuda.Stream()
    dA, dB, dB2 = to_dev_u16(A), to_dev_u16(B), to_dev_u16(B2)
    for rep in range(3):
        C = torch.full((N, M), 0x7E00, dtype=torch.int16, device="cuda")
        C2 = torch.full((256, N), 0x7E00, dtype=torch.int16, device="cuda")
        row_max = torch.full((M,), float("nan"), device="cuda")
        row_sum = torch.full((M,), float("nan"), device="cuda")
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.gemm_f16_tn_softmax_stats(M, N, K, dA, K, dB, K, C, M, 0.5, row_max, row_sum, s)
            g.gemm_f16_tn(N, 256, M, C, M, dB2, M, C2, N, s)
        g.gemm_poll_device_status(s)
        assert np.array_equal(C.cpu().numpy().view(np.uint16), scores)
        assert np.array_equal(row_max.cpu().numpy().astype(np.float64), mx_ref)     # integer scores x 0.5: exact
        assert np.array_equal(C2.cpu().numpy().view(np.uint16), ref2), f"rep {rep}"


def test_gemm_then_quantise_then_fp8_gemm():
    """An FP16 GEMM's C is quantised to E4M3 on the device and fed, with its
    device-resident scale, to an FP8 GEMM: three programmatic dependents back
    to back.  C and the codes are bit-exact (integer sums, the same binary32
    quantisation arithmetic), the FP8 result within the FP8 tolerance."""
    import dense_gemm_tn_gb300 as g
    from tests.gpu_helpers import F8_TOL, assert_tol, bf16_values
    M, N, K = 1024, 768, 64
    A = synth.sign_fp16(M * K, 7401)
    B = synth.sign_fp16(N * K, 7402)
    C1 = ref_nm(M, N, K, A, B)                                # (N, M) fp16 codes
    q_ref, s_ref = oracle.quantize_e4m3(C1.reshape(-1), "f16", N, M)
    N2 = 512
    qb, sb = synth.gauss_e4m3(N2 * M, 7403)                   # the second GEMM: M' = N, K' = M
    C2_ref, S2, _ = oracle.gemm_f8e4m3_tn(N, N2, M, q_ref, M, qb, M, s_ref, sb)
    s = torch.cuda.Stream()
    dA, dB = to_dev_u16(A), to_dev_u16(B)
    dqb = torch.from_numpy(qb).cuda()
    scales = torch.tensor([0.0, sb], dtype=torch.float32, device="cuda")
    for rep in range(3):
        C = torch.full((N, M), 0x7E00, dtype=torch.int16, device="cuda")
        q = torch.zeros((N, M), dtype=torch.uint8, device="cuda")
        C2 = torch.full((N2, N), 0x7FC0, dtype=torch.int16, device="cuda")
        scales[0] = float("nan")
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.gemm_f16_tn(M, N, K, dA, K, dB, K, C, M, s)
            g.gemm_quantize_e4m3(C, g.GEMM_IN_F16, N, M, M, q, M, scales.data_ptr(), s)
            g.gemm_f8e4m3_tn_dscale(N, N2, M, q, M, dqb, M, C2, N, scales.data_ptr(), scales.data_ptr() + 4, s)
        g.gemm_poll_device_status(s)
        assert np.array_equal(C.cpu().numpy().view(np.uint16), C1), f"rep {rep}: C"
        assert np.array_equal(q.cpu().numpy().reshape(-1), q_ref[: N * M]), f"rep {rep}: codes"
        assert scales[0].item() == s_ref, f"rep {rep}: scale"
        got2 = C2.cpu().numpy().view(np.uint16)
        ref2 = oracle.c_as_nm(C2_ref, N, N2, N)
        assert_tol(bf16_values(got2), bf16_values(ref2), S2, F8_TOL, f"rep {rep}: FP8 GEMM")
