"""GPU parity of the FP8 front end: per-tensor E4M3 quantisation on the device
(gemm_quantize_e4m3) and the FP8 GEMM with device-resident scales
(gemm_f8e4m3_tn_dscale), against the CPU oracle.

Codes and scales are integers / binary32 values decided by floating point in
binary32 on both sides, so they must be bit-identical.  The GEMM on quantised
operands is held to the FP8 tolerance 2^-7 |C_ref| + 2^-8 sum_k |a b|.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import F8_TOL, GuardedC, assert_tol, bf16_values, run_f8, to_dev_u8

pytestmark = pytest.mark.gpu

QGUARD = 4096
QCANARY = 0xA5
QPOISON = 0x7F         # the E4M3 NaN code, never produced from finite input


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    return g


def values(rows, cols, seed, spread=True):
    """rows x cols N(0,1) draws (float64), optionally times e^U(-5,5) so the
    codes span the subnormal and normal ranges of E4M3."""
    x = synth.gauss_f64(rows * cols, seed).reshape(rows, cols) if rows * cols else np.zeros((rows, cols))
    if spread and x.size:
        u = synth.gauss_f64(rows * cols, seed + 7777).reshape(rows, cols)
        x = x * np.exp(np.clip(u, -2.5, 2.5) * 2.0)
    return x


def host_input(x64, x_type):
    """The harness's input tensor of one type: (numpy array for the oracle, torch CPU tensor)."""
    t32 = torch.from_numpy(np.ascontiguousarray(x64, np.float32))
    if x_type == "f32":
        return t32.numpy(), t32
    if x_type == "f16":
        t = t32.to(torch.float16)
        return t.view(torch.int16).numpy().view(np.uint16), t
    t = t32.to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16), t


TYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}
ESZ = {"f32": 4, "f16": 2, "bf16": 2}


class GuardedQ:
    def __init__(self, rows, ldq, offset=0):
        self.n = max(rows * ldq, 1)
        self.off = QGUARD + offset
        self.buf = torch.full((self.off + self.n + QGUARD,), QCANARY, dtype=torch.uint8, device="cuda")
        self.buf[self.off: self.off + self.n] = QPOISON
        self.rows, self.ldq = rows, ldq

    @property
    def ptr(self):
        return self.buf.data_ptr() + self.off

    def host(self):
        h = self.buf.cpu().numpy()
        assert np.all(h[: self.off] == QCANARY), "store before q"
        assert np.all(h[self.off + self.n:] == QCANARY), "store after q"
        return h[self.off: self.off + self.n].copy()


def run_quant(xt, x_type, rows, cols, ldx, ldq, x_off=0, q_off=0, stream=None):
    """Quantise the torch CPU tensor xt (rows x ldx after padding) on the GPU.
    Returns (q as rows x ldq host bytes, scale as a Python float)."""
    import dense_gemm_tn_gb300 as g
    esz = ESZ[x_type]
    flat = xt.reshape(-1)
    dev = torch.zeros(x_off + max(flat.numel(), 1), dtype=xt.dtype, device="cuda")
    if flat.numel():
        dev[x_off: x_off + flat.numel()] = flat.cuda()
    q = GuardedQ(rows, ldq, q_off)
    scale = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    g.gemm_quantize_e4m3(dev.data_ptr() + esz * x_off, TYPE_CODE[x_type], rows, cols, ldx, q.ptr, ldq, scale,
                         stream)
    g.gemm_poll_device_status(stream)
    return q.host(), float(scale.item())


def padded(x64, ldx):
    rows, cols = x64.shape
    out = np.zeros((rows, ldx))
    out[:, :cols] = x64
    out[:, cols:] = 1e30 if ldx > cols else 0     # huge padding must not enter amax
    return out


SHAPES = [(1, 1), (3, 5), (7, 4100), (300, 136), (1000, 1000), (33, 8195)]


@pytest.mark.parametrize("x_type", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_quantize_matches_oracle(x_type, rows, cols):
    x64 = values(rows, cols, 1000 + rows + cols)
    xn, xt = host_input(x64, x_type)
    q, scale = run_quant(xt, x_type, rows, cols, cols, cols)
    q_ref, s_ref = oracle.quantize_e4m3(xn, x_type, rows, cols)
    assert scale == s_ref
    assert np.array_equal(q, q_ref[: rows * cols]), f"{np.sum(q != q_ref[:rows * cols])} codes differ"


@pytest.mark.parametrize("x_type", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols,ldx,ldq,x_off,q_off", [
    (17, 4097, 4120, 4105, 0, 0),      # padded rows (16-byte aligned f32 / bf16 rows? ldx*esz decides)
    (9, 300, 301, 300, 0, 0),          # odd row stride: unaligned rows
    (64, 512, 512, 520, 1, 0),         # unaligned x base
    (64, 512, 600, 512, 0, 3),         # unaligned q base
    (5, 9000, 9000, 9001, 0, 0),       # contiguous x, padded q
])
def test_quantize_strided_and_unaligned(x_type, rows, cols, ldx, ldq, x_off, q_off):
    x64 = values(rows, cols, 77 + cols)
    xn, xt = host_input(padded(x64, ldx), x_type)
    # padding of 1e30 would overflow f16; this test uses f32 / bf16 only
    q, scale = run_quant(xt, x_type, rows, cols, ldx, ldq, x_off, q_off)
    q_ref, s_ref = oracle.quantize_e4m3(xn, x_type, rows, cols, ldx, ldq)
    assert scale == s_ref
    q2 = q[: rows * ldq].reshape(rows, ldq)
    assert np.array_equal(q2[:, :cols], q_ref.reshape(rows, ldq)[:, :cols])
    assert np.all(q2[:, cols:] == QPOISON), "store into q's row padding"


def test_quantize_full_size_bf16():
    """An 8192 x 8192 bfloat16 operand (the FP8 GEMM's operand size), all codes."""
    rows = cols = 8192
    x64 = synth.gauss_f64(rows * cols, 555).reshape(rows, cols)
    xn, xt = host_input(x64, "bf16")
    q, scale = run_quant(xt, "bf16", rows, cols, cols, cols)
    q_ref, s_ref = oracle.quantize_e4m3(xn, "bf16", rows, cols)
    assert scale == s_ref
    assert np.array_equal(q, q_ref)


def test_quantize_zero_and_empty():
    x = torch.zeros((40, 70), dtype=torch.float32)
    x[3, 4] = -0.0
    q, scale = run_quant(x, "f32", 40, 70, 70, 70)
    assert scale == 0.0
    assert np.all((q & 0x7F) == 0) and q[3 * 70 + 4] == 0x80
    q, scale = run_quant(torch.zeros((0, 5)), "f32", 0, 5, 5, 5)
    assert scale == 0.0 and np.all(q == QPOISON)


def test_quantize_bf16_subnormals_flt_max_path():
    bits = np.array([0x0001, 0x8003, 0x0002, 0x0000] * 300, np.uint16)
    xt = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    q, scale = run_quant(xt, "bf16", 1, bits.size, bits.size, bits.size)
    q_ref, s_ref = oracle.quantize_e4m3(bits, "bf16", 1, bits.size)
    assert scale == s_ref and np.array_equal(q, q_ref)


def test_quantize_back_to_back_and_side_stream():
    """Calls on one stream reuse its slot array with a new epoch each, queued
    without a host synchronisation in between; a side stream has its own
    array.  Every result must be its own call's."""
    import dense_gemm_tn_gb300 as g
    side = torch.cuda.Stream()
    streams = [torch.cuda.current_stream(), torch.cuda.current_stream(), side, torch.cuda.current_stream(), side]
    rows, cols = 200, 3000
    jobs = []
    for i in range(len(streams)):
        xn, xt = host_input(values(rows, cols, 40 + i) * (1.0 + i), "bf16")
        q = torch.full((rows, cols), QPOISON, dtype=torch.uint8, device="cuda")
        scale = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
        jobs.append((xn, xt.cuda(), q, scale))
    torch.cuda.synchronize()
    for (xn, x, q, scale), stream in zip(jobs, streams):
        g.gemm_quantize_e4m3(x, TYPE_CODE["bf16"], rows, cols, cols, q, cols, scale, stream)
    g.gemm_poll_device_status(side)
    g.gemm_poll_device_status()
    for i, (xn, x, q, scale) in enumerate(jobs):
        q_ref, s_ref = oracle.quantize_e4m3(xn, "bf16", rows, cols)
        assert float(scale.item()) == s_ref, f"call {i}"
        assert np.array_equal(q.cpu().numpy().reshape(-1), q_ref), f"call {i}"


@pytest.mark.parametrize("M,N,K", [(300, 200, 136), (1000, 700, 520), (4096, 4096, 1024)])
def test_dscale_gemm_equals_host_scale_gemm(M, N, K):
    """Device-resident scales give bit-identical C to the same scales passed by value."""
    import dense_gemm_tn_gb300 as g
    qa, sa = synth.gauss_e4m3(M * K, 61)
    qb, sb = synth.gauss_e4m3(N * K, 62)
    ref = run_f8(M, N, K, qa, K, qb, K, sa, sb)
    dA, dB = to_dev_u8(qa), to_dev_u8(qb)
    scales = torch.tensor([sa, sb], dtype=torch.float32, device="cuda")
    C = GuardedC(M, N, M)
    g.gemm_f8e4m3_tn_dscale(M, N, K, dA, K, dB, K, C.ptr, M, scales.data_ptr(), scales.data_ptr() + 4)
    g.gemm_poll_device_status()
    assert np.array_equal(C.nm(), ref)


@pytest.mark.parametrize("M,N,K", [(257, 300, 520), (2048, 2048, 1024)])
def test_fp8_pipeline_matches_oracle(M, N, K):
    """bf16 X (M x K) and W (N x K) -> device quantisation -> FP8 GEMM with the
    device scales, with no host round trip; codes and scales bit-exact, C
    within the FP8 tolerance of the oracle GEMM on the oracle's codes."""
    import dense_gemm_tn_gb300 as g
    xn, xt = host_input(values(M, K, 91, spread=False), "bf16")
    wn, wt = host_input(values(N, K, 92, spread=False), "bf16")
    X, W = xt.cuda(), wt.cuda()
    qx, sx = g.quantize_e4m3(X)
    qw, sw = g.quantize_e4m3(W)
    C = g.f8e4m3_tn_dscale(qx, qw, sx, sw)
    g.gemm_poll_device_status()
    qx_ref, sx_ref = oracle.quantize_e4m3(xn, "bf16", M, K)
    qw_ref, sw_ref = oracle.quantize_e4m3(wn, "bf16", N, K)
    assert float(sx.item()) == sx_ref and float(sw.item()) == sw_ref
    assert np.array_equal(qx.cpu().numpy().reshape(-1), qx_ref)
    assert np.array_equal(qw.cpu().numpy().reshape(-1), qw_ref)
    c_ref, S, _ = oracle.gemm_f8e4m3_tn(M, N, K, qx_ref, K, qw_ref, K, sx_ref, sw_ref)
    got = C.view(torch.int16).cpu().numpy().view(np.uint16)
    assert_tol(bf16_values(got), bf16_values(oracle.c_as_nm(c_ref, M, N, M)), S, F8_TOL, "fp8 pipeline")
