"""Shared helpers of the GPU tests: upload TN operands, run the C ABI into a
NaN-poisoned output with guard bands, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle

GUARD = 2048          # elements of canary on each side of C
CANARY = 0x5A5A
POISON = 0x7E00       # binary16 / bf16-ish NaN pattern written into C before the call

F16_TOL = (2.0 ** -10, 2.0 ** -12)    # |C - C_ref| <= rel |C_ref| + abs * sum_k |a b|
F8_TOL = (2.0 ** -7, 2.0 ** -8)


def to_dev_u16(codes: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(codes).view(np.int16)).cuda()


def to_dev_u8(codes: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(codes)).cuda()


def pad_rows(codes: np.ndarray, rows: int, K: int, ld: int, fill) -> np.ndarray:
    """Dense rows x K codes -> rows x ld with the padding set to `fill`."""
    out = np.full(rows * ld if rows else 1, fill, dtype=codes.dtype)
    if rows and K:
        out[: rows * ld].reshape(rows, ld)[:, :K] = codes.reshape(rows, K)
    return out


class GuardedC:
    """A C buffer (ldc*N 16-bit elements) with canary bands on both sides and
    the payload poisoned with NaN.  `offset_elems` shifts C off 16-byte
    alignment when odd."""

    def __init__(self, M, N, ldc, offset_elems=0):
        self.M, self.N, self.ldc = M, N, ldc
        self.n = max(ldc * N, 1)
        self.off = GUARD + offset_elems
        self.buf = torch.full((self.off + self.n + GUARD,), CANARY, dtype=torch.int16, device="cuda")
        self.buf[self.off: self.off + self.n] = np.int16(POISON)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr() + 2 * self.off

    def host(self) -> np.ndarray:
        h = self.buf.cpu().numpy().view(np.uint16)
        assert np.all(h[: self.off] == CANARY), "store before C"
        assert np.all(h[self.off + self.n:] == CANARY), "store after C"
        return h[self.off: self.off + self.n].copy()

    def nm(self) -> np.ndarray:
        """(N, M) codes: row n = column n of C; padding rows must be intact."""
        h = self.host()
        full = h[: self.ldc * self.N].reshape(self.N, self.ldc)
        if self.ldc > self.M:
            assert np.all(full[:, self.M:] == POISON), "store into ldc padding"
        return full[:, : self.M]


def f16_values(codes):
    return np.asarray(codes, np.uint16).view(np.float16).astype(np.float64)


def bf16_values(codes):
    c = np.ascontiguousarray(np.asarray(codes, np.uint16)).view(np.int16)
    return torch.from_numpy(c).view(torch.bfloat16).double().numpy()


def assert_tol(got_vals, ref_vals, S, tol, what=""):
    rel, absf = tol
    assert not np.isnan(got_vals).any(), f"{what}: NaN in output (unwritten?)"
    D = np.abs(got_vals - ref_vals)
    bound = rel * np.abs(ref_vals) + absf * S
    bad = D > bound
    if bad.any():
        i = np.flatnonzero(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} outside tolerance; first at {i}: got "
                             f"{got_vals.flat[i]} want {ref_vals.flat[i]} bound {bound.flat[i]}")


def sample_positions(M, N, count, seed, tile_m=256, tile_n=128):
    """Random positions plus the corners and both sides of every tile edge
    (capped), so ragged tails are always sampled."""
    rng = np.random.default_rng(seed)
    ms = [0, M - 1] + [x for t in range(tile_m, M, tile_m) for x in (t - 1, t)][:64]
    ns = [0, N - 1] + [x for t in range(tile_n, N, tile_n) for x in (t - 1, t)][:64]
    edge_m = np.array([m for m in ms for _ in ns[:8]] + [M - 1] * len(ns), np.int64)
    edge_n = np.array([n for _ in ms for n in ns[:8]] + ns, np.int64)
    rm = rng.integers(0, M, count)
    rn = rng.integers(0, N, count)
    return np.concatenate([edge_m, rm]), np.concatenate([edge_n, rn])


def run_f16(M, N, K, A, lda, B, ldb, ldc=None, c_offset=0, a_offset=0, b_offset=0, stream=None):
    """A, B: codes already laid out with lda / ldb.  Returns the (N, M) codes."""
    import dense_gemm_tn_gb300 as g
    ldc = M if ldc is None else ldc
    dA = to_dev_u16(np.concatenate([np.zeros(a_offset, np.uint16), A]))
    dB = to_dev_u16(np.concatenate([np.zeros(b_offset, np.uint16), B]))
    C = GuardedC(M, N, ldc, c_offset)
    g.gemm_f16_tn(M, N, K, dA.data_ptr() + 2 * a_offset, lda, dB.data_ptr() + 2 * b_offset, ldb,
                  C.ptr, ldc, stream)
    g.gemm_poll_device_status(stream)
    return C.nm()


def run_f8(M, N, K, A, lda, B, ldb, sa, sb, ldc=None, c_offset=0, a_offset=0, b_offset=0, stream=None):
    import dense_gemm_tn_gb300 as g
    ldc = M if ldc is None else ldc
    dA = to_dev_u8(np.concatenate([np.zeros(a_offset, np.uint8), A]))
    dB = to_dev_u8(np.concatenate([np.zeros(b_offset, np.uint8), B]))
    C = GuardedC(M, N, ldc, c_offset)
    g.gemm_f8e4m3_tn(M, N, K, dA.data_ptr() + a_offset, lda, dB.data_ptr() + b_offset, ldb,
                     C.ptr, ldc, sa, sb, stream)
    g.gemm_poll_device_status(stream)
    return C.nm()


def check_f16_full(M, N, K, A, B, exact=False, what="", **kw):
    lda = kw.pop("lda", K)
    ldb = kw.pop("ldb", K)
    Ap = pad_rows(A, M, K, lda, 0x7C00) if lda != K else A     # +Inf in padding must be ignored
    Bp = pad_rows(B, N, K, ldb, 0xFC00) if ldb != K else B
    got = run_f16(M, N, K, Ap, lda, Bp, ldb, **kw)
    Cref, S, _ = oracle.gemm_f16_tn(M, N, K, A, K, B, K)
    ref = oracle.c_as_nm(Cref, M, N, M)
    if exact:
        assert np.array_equal(got, ref), f"{what}: not bit-exact ({np.sum(got != ref)} differ)"
    else:
        assert_tol(f16_values(got), f16_values(ref), S, F16_TOL, what)
    return got


def check_f8_full(M, N, K, A, B, sa, sb, what="", **kw):
    lda = kw.pop("lda", K)
    ldb = kw.pop("ldb", K)
    Ap = pad_rows(A, M, K, lda, 0x7F) if lda != K else A       # NaN codes in padding must be ignored
    Bp = pad_rows(B, N, K, ldb, 0xFF) if ldb != K else B
    got = run_f8(M, N, K, Ap, lda, Bp, ldb, sa, sb, **kw)
    Cref, S, _ = oracle.gemm_f8e4m3_tn(M, N, K, A, K, B, K, sa, sb)
    ref = oracle.c_as_nm(Cref, M, N, M)
    assert_tol(bf16_values(got), bf16_values(ref), S, F8_TOL, what)
    return got
