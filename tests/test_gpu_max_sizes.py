"""Operands and results of more than 2^31 elements.

Every element offset on the path must be 64-bit: row offsets of A and B (in
the tensor maps, and in the repack of unaligned rows), column offsets of C (in
the TMA store and in the plain stores used when C is not TMA-addressable),
the quantiser's element indices, and the scores the softmax-statistics path
writes.  A 32-bit offset would wrap at 2^31 elements (or 2^32 bytes) and
alias a row or column far from the right one.

Inputs are +-1 (E4M3 +-1 for the FP8 case), so every output is an integer
below 2^24 and must be bit-exact.  The large operands are built on the
device from seeded sign blocks: row r is block row r mod 4099 with its sign
flipped by a per-row sign, both drawn by `synth`.  4099 divides no power of
two, so a row aliased by a wrapped offset differs from the right one.  The
oracle gets the same rows, built on the host by the same sign flips, and
computes sampled outputs.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import POISON, f16_values, to_dev_u16

pytestmark = pytest.mark.gpu

BLOCK = 4099
CANARY = 0x5A5A
TAIL = 4096            # canary elements after a large output


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    return g


@pytest.fixture(autouse=True)
def _free():
    yield
    import dense_gemm_tn_gb300 as g
    g.gemm_debug_force_cta_group(0)
    g.gemm_debug_force_wide_tiles(0)
    g.gemm_release_workspace()
    torch.cuda.empty_cache()


class TallSigns:
    """A rows x K sign operand (fp16 codes) and its host rows on demand."""

    def __init__(self, rows, K, seed):
        self.rows, self.K = rows, K
        self.block = synth.sign_fp16(BLOCK * K, seed).reshape(BLOCK, K)
        self.flip = synth.sign_fp16(rows, seed + 1) & np.uint16(0x8000)

    def host_rows(self, r):
        r = np.asarray(r, np.int64)
        return (self.block[r % BLOCK] ^ self.flip[r][:, None]).astype(np.uint16)

    def device(self, ld, pad_code=0x7C00):
        """rows x ld int16 on the device; columns K..ld-1 hold `pad_code`."""
        blk = to_dev_u16(self.block)
        flip = to_dev_u16(self.flip)
        out = torch.empty((self.rows, ld), dtype=torch.int16, device="cuda")
        step = 1 << 16
        for r0 in range(0, self.rows, step):
            r1 = min(self.rows, r0 + step)
            idx = torch.arange(r0, r1, device="cuda") % BLOCK
            out[r0:r1, : self.K] = torch.bitwise_xor(blk.index_select(0, idx), flip[r0:r1, None])
        if ld > self.K:
            out[:, self.K:] = as_i16(pad_code)
        return out


def as_i16(code):
    """A 16-bit code as the int16 value torch stores for it."""
    return int(np.array(code, np.uint16).view(np.int16))


def big_output(rows, ld, dtype=torch.int16, poison=POISON, canary=CANARY):
    """A rows x ld output (flat, plus a canary tail), poisoned."""
    conv = as_i16 if dtype == torch.int16 else int
    buf = torch.empty((rows * ld + TAIL,), dtype=dtype, device="cuda")
    buf[: rows * ld] = conv(poison)
    buf[rows * ld:] = conv(canary)
    return buf


def check_tail(buf, n, canary=CANARY):
    tail = buf[n:].cpu().numpy().view(np.uint16 if buf.dtype == torch.int16 else np.uint8)
    assert np.all(tail == canary), "store past the end of the output"


SHAPES = ["auto", "cta1", "wide"]


def set_shape(shape):
    """auto: the library's choice; cta1: one CTA per 128 x 256 tile; wide:
    CTA pairs on 256 x 512 tiles."""
    import dense_gemm_tn_gb300 as g
    g.gemm_debug_force_cta_group(1 if shape == "cta1" else 2 if shape == "wide" else 0)
    g.gemm_debug_force_wide_tiles(1 if shape == "wide" else 0)


def picks(count, n, seed, must):
    rng = np.random.default_rng(seed)
    m = [x for x in must if 0 <= x < n]
    return np.unique(np.concatenate([np.array(m, np.int64), rng.integers(0, n, count)]))


def e4m3_signs(codes16):
    """+-1 fp16 codes -> +-1 E4M3 codes (0x38 / 0xB8)."""
    return (((codes16 >> 8) & 0x80) | 0x38).astype(np.uint8)


@pytest.mark.parametrize("kind", ["f16", "e4m3"])
@pytest.mark.parametrize("pad", [0, 1])
@pytest.mark.parametrize("shape", SHAPES)
def test_c_beyond_2_31_elements(kind, pad, shape):
    """C of 65536 x 40960 (2.68e9 elements, 5.4 GB) with ldc = M (TMA stores)
    or M + 1 (plain stores): columns on both sides of element 2^31."""
    import dense_gemm_tn_gb300 as g
    set_shape(shape)
    M, N, K = 65536, 40960, 64
    ldc = M + pad
    A = synth.sign_fp16(M * K, 811)
    B = synth.sign_fp16(N * K, 812)
    C = big_output(N, ldc)
    if kind == "f16":
        g.gemm_f16_tn(M, N, K, to_dev_u16(A), K, to_dev_u16(B), K, C, ldc, None)
    else:
        dA = torch.from_numpy(e4m3_signs(A)).cuda()
        dB = torch.from_numpy(e4m3_signs(B)).cuda()
        g.gemm_f8e4m3_tn(M, N, K, dA, K, dB, K, C, ldc, 1.0, 1.0, None)
    g.gemm_poll_device_status()
    wrap = (1 << 31) // ldc
    ns = picks(9, N, 813, [0, 1, wrap - 1, wrap, wrap + 1, (1 << 32) // (2 * ldc), N - 2, N - 1])
    got = C[: N * ldc].view(N, ldc)[torch.from_numpy(ns).cuda()].cpu().numpy().view(np.uint16)
    Bs = B.reshape(N, K)[ns].reshape(-1)
    if kind == "f16":
        ref, _, _ = oracle.gemm_f16_tn(M, ns.size, K, A, K, Bs, K)
    else:
        ref, _, _ = oracle.gemm_f8e4m3_tn(M, ns.size, K, e4m3_signs(A), K, e4m3_signs(Bs), K, 1.0, 1.0)
    ref = oracle.c_as_nm(ref, M, ns.size, M)
    bad = np.flatnonzero((got[:, :M] != ref).any(axis=1))
    assert bad.size == 0, f"columns {ns[bad][:8]} differ"
    if pad:
        assert np.all(got[:, M:] == POISON), "store into ldc padding"
    check_tail(C, N * ldc)


@pytest.mark.parametrize("pad", [0, 1])
@pytest.mark.parametrize("shape", SHAPES)
def test_a_beyond_2_31_elements(pad, shape):
    """A of 270000 x 8192 (2.2e9 elements) with lda = K (TMA in place) or
    K + 1 (the repack): rows on both sides of element 2^31 and the ragged
    last tile row."""
    import dense_gemm_tn_gb300 as g
    set_shape(shape)
    M, N, K = 270000, 384, 8192
    lda = K + pad
    tall = TallSigns(M, K, 821)
    dA = tall.device(lda)
    B = synth.sign_fp16(N * K, 823)
    C = big_output(N, M)
    g.gemm_f16_tn(M, N, K, dA, lda, to_dev_u16(B), K, C, M, None)
    g.gemm_poll_device_status()
    del dA
    wrap = (1 << 31) // lda
    ms = picks(48, M, 824, [0, 1, wrap - 1, wrap, wrap + 1, (1 << 32) // (2 * lda), 269823, 269824, M - 2, M - 1])
    got = C[: N * M].view(N, M)[:, torch.from_numpy(ms).cuda()].cpu().numpy().view(np.uint16).T    # (S, N)
    ref, _, _ = oracle.gemm_f16_tn(ms.size, N, K, tall.host_rows(ms).reshape(-1), K, B, K)
    ref = oracle.c_as_nm(ref, ms.size, N, ms.size).T                                                 # (S, N)
    bad = np.flatnonzero((got != ref).any(axis=1))
    assert bad.size == 0, f"rows {ms[bad][:8]} differ"
    check_tail(C, N * M)


@pytest.mark.parametrize("pad", [0, 1])
def test_b_beyond_2_31_elements(pad):
    """B of 270000 x 8192 (N x K, 2.2e9 elements) with ldb = K or K + 1."""
    import dense_gemm_tn_gb300 as g
    M, N, K = 384, 270000, 8192
    ldb = K + pad
    tall = TallSigns(N, K, 831)
    dB = tall.device(ldb, pad_code=0xFC00)
    A = synth.sign_fp16(M * K, 833)
    C = big_output(N, M)
    g.gemm_f16_tn(M, N, K, to_dev_u16(A), K, dB, ldb, C, M, None)
    g.gemm_poll_device_status()
    del dB
    wrap = (1 << 31) // ldb
    ns = picks(48, N, 834, [0, 1, wrap - 1, wrap, wrap + 1, (1 << 32) // (2 * ldb), N - 2, N - 1])
    got = C[: N * M].view(N, M)[torch.from_numpy(ns).cuda()].cpu().numpy().view(np.uint16)          # (S, M)
    ref, _, _ = oracle.gemm_f16_tn(M, ns.size, K, A, K, tall.host_rows(ns).reshape(-1), K)
    ref = oracle.c_as_nm(ref, M, ns.size, M)
    bad = np.flatnonzero((got != ref).any(axis=1))
    assert bad.size == 0, f"columns {ns[bad][:8]} differ"
    check_tail(C, N * M)


def test_quantize_beyond_2_31_elements():
    """A 65536 x 40960 bfloat16 tensor (2.68e9 elements) whose largest
    magnitude sits past element 2^31: the scale and sampled codes on both
    sides of 2^31 must match the oracle's."""
    import dense_gemm_tn_gb300 as g
    rows, cols = 65536, 40960
    blk_rows = 1031
    blk = synth.gauss_bf16(blk_rows * cols, 841).reshape(blk_rows, cols)
    flip = synth.sign_fp16(rows, 842) & np.uint16(0x8000)
    d_blk, d_flip = to_dev_u16(blk), to_dev_u16(flip)
    x = torch.empty((rows, cols), dtype=torch.int16, device="cuda")
    for r0 in range(0, rows, 8192):
        idx = torch.arange(r0, r0 + 8192, device="cuda") % blk_rows
        x[r0:r0 + 8192] = torch.bitwise_xor(d_blk.index_select(0, idx), d_flip[r0:r0 + 8192, None])
    r_max, c_max = 60000, 12345                            # flat index 2.46e9
    x[r_max, c_max] = as_i16(0xC47A)                       # bf16 -1000.0
    q = big_output(rows, cols, dtype=torch.uint8, poison=0x7F, canary=0xA5)
    scale = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    g.gemm_quantize_e4m3(x, g.GEMM_IN_BF16, rows, cols, cols, q, cols, scale, None)
    g.gemm_poll_device_status()
    wrap_r = (1 << 31) // cols
    rs = picks(40, rows, 843, [0, wrap_r - 1, wrap_r, wrap_r + 1, r_max, rows - 1])
    cs = np.random.default_rng(844).integers(0, cols, 64)
    cs = np.unique(np.concatenate([cs, [0, c_max, cols - 1]]))
    rr, cc = np.meshgrid(rs, cs, indexing="ij")
    host_x = (blk[rr % blk_rows, cc] ^ flip[rr]).astype(np.uint16)
    host_x[(rr == r_max) & (cc == c_max)] = 0xC47A
    q_ref, s_ref = oracle.quantize_e4m3(host_x.reshape(-1), "bf16", 1, host_x.size)
    got_q = q[: rows * cols].view(rows, cols)[torch.from_numpy(rs).cuda()][:, torch.from_numpy(cs).cuda()]
    got_q = got_q.cpu().numpy().reshape(-1)
    assert float(scale.item()) == s_ref
    assert np.array_equal(got_q, q_ref[: host_x.size]), f"{np.sum(got_q != q_ref[:host_x.size])} codes differ"
    assert got_q[np.flatnonzero(((rr == r_max) & (cc == c_max)).reshape(-1))[0]] == 0xFE      # -448
    check_tail(q, rows * cols, canary=0xA5)


def test_softmax_stats_scores_beyond_2_31_elements():
    """Scores of 8192 x 270000 (C of 2.2e9 elements): sampled rows' scores and
    statistics over all 270000 columns."""
    import dense_gemm_tn_gb300 as g
    M, N, K = 8192, 270000, 64
    scale = 0.125
    A = synth.sign_fp16(M * K, 851)
    B = synth.sign_fp16(N * K, 852)
    C = big_output(N, M)
    row_max = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    row_sum = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    g.gemm_f16_tn_softmax_stats(M, N, K, to_dev_u16(A), K, to_dev_u16(B), K, C, M, scale, row_max, row_sum, None)
    g.gemm_poll_device_status()
    ms = picks(6, M, 853, [0, M - 1])
    As = A.reshape(M, K)[ms].reshape(-1)
    c_ref, mx_ref, sm_ref, S = oracle.gemm_f16_tn_softmax_stats(ms.size, N, K, As, K, B, K, scale)
    got_c = C[: N * M].view(N, M)[:, torch.from_numpy(ms).cuda()].cpu().numpy().view(np.uint16)    # (N, S)
    ref_c = oracle.c_as_nm(c_ref, ms.size, N, ms.size)                                               # (N, S)
    assert np.array_equal(got_c, ref_c), f"{np.sum(got_c != ref_c)} scores differ"
    got_max = row_max.cpu().numpy()[ms].astype(np.float64)
    got_sum = row_sum.cpu().numpy()[ms].astype(np.float64)
    assert np.array_equal(got_max, mx_ref)                 # integer scores x 1/8: exact
    Y = np.abs(f16_values(ref_c))
    E = (2.0 ** -16 * S + 2.0 ** -23 * Y).max(axis=0)
    rel = 2.0 * E + 2.0 ** -19 + (4 * ((N + 127) // 128) + 8) * 2.0 ** -22
    err = np.abs(got_sum - sm_ref) / sm_ref
    assert np.all(err <= rel), f"row_sum rel error {err.max()} > {rel[np.argmax(err)]}"
    check_tail(C, N * M)


@pytest.mark.parametrize("pad", [0, 1])
def test_skinny_kernel_a_beyond_2_31_elements(pad):
    """The kernel for few columns (forced) on A of 270000 x 8192 (2.2e9
    elements) with lda = K or K + 1: rows m on both sides of element 2^31,
    2110 tiles walked by 152 CTAs in turn."""
    import dense_gemm_tn_gb300 as g
    M, N, K = 270000, 16, 8192
    lda = K + pad
    tall = TallSigns(M, K, 841)
    dA = tall.device(lda)
    B = synth.sign_fp16(N * K, 843)
    C = big_output(N, M)
    g.gemm_debug_set_skinny_mode(2)
    try:
        g.gemm_f16_tn(M, N, K, dA, lda, to_dev_u16(B), K, C, M, None)
        g.gemm_poll_device_status()
        assert "skinny=1" in g.last_launch(), g.last_launch()
    finally:
        g.gemm_debug_set_skinny_mode(0)
    del dA
    wrap = (1 << 31) // lda
    ms = picks(48, M, 844, [0, 1, wrap - 1, wrap, wrap + 1, (1 << 32) // (2 * lda), 269951, 269952, M - 2, M - 1])
    got = C[: N * M].view(N, M)[:, torch.from_numpy(ms).cuda()].cpu().numpy().view(np.uint16).T    # (S, N)
    ref, _, _ = oracle.gemm_f16_tn(ms.size, N, K, tall.host_rows(ms).reshape(-1), K, B, K)
    ref = oracle.c_as_nm(ref, ms.size, N, ms.size).T                                                 # (S, N)
    bad = np.flatnonzero((got != ref).any(axis=1))
    assert bad.size == 0, f"rows {ms[bad][:8]} differ"
    check_tail(C, N * M)
