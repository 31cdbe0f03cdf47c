"""CPU oracle for the TN GEMM (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm import this package.  The product library never
does, and the two share no code: this package wraps ``oracle.c``, a plain
fp64 triple loop with its own binary16 / bfloat16 / E4M3 codecs written from
the format definitions.

The computation is the plain definition C[m,n] = sum_k A[m,k] B[k,n]
(hello-gpu ch.11 "GEMM-Like", section 11.1) in the TN storage of the AMD ROCm
blog "FP16 GEMM optimization on AMD RDNA 3 and RDNA 4" (section "What we
compute"): A row-major M x K, B column-major K x N, C column-major with
leading dimension M.  Accumulation is sequential in k in double, rounded once
to the output type with round-to-nearest-even.

Also: the scaled-score GEMM with the softmax's row statistics (row maximum and
sum of exponentials), and per-tensor E4M3 quantisation (amax, scale to 448, one RNE rounding),
the step that produces the F8 GEMM's operands.

Pins (tests/test_oracle.py): the worked example and its partial sums, the
outer-product intermediates, closed forms (all-ones, identity, permutation),
exact rational brute force on the edge shapes of section 11.4, and exhaustive
codec checks against numpy / torch CPU conversions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build_cmd() -> list[str]:
    return ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC",
            "-o", _LIB, _SRC, "-lm"]


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (if missing or stale)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(build_cmd())
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_fp16_decode.restype = ctypes.c_double
    lib.oracle_fp16_decode.argtypes = [ctypes.c_uint16]
    lib.oracle_fp16_encode.restype = ctypes.c_uint16
    lib.oracle_fp16_encode.argtypes = [ctypes.c_double]
    lib.oracle_bf16_encode.restype = ctypes.c_uint16
    lib.oracle_bf16_encode.argtypes = [ctypes.c_double]
    lib.oracle_bf16_decode.restype = ctypes.c_double
    lib.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
    lib.oracle_e4m3_decode.restype = ctypes.c_double
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_gemm_f16_tn.restype = ctypes.c_int
    lib.oracle_gemm_f16_tn.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64, p, p]
    lib.oracle_gemm_f16_tn_at.restype = ctypes.c_int
    lib.oracle_gemm_f16_tn_at.argtypes = [i64, i64, i64, p, i64, p, i64, i64, p, p, p, p, p]
    lib.oracle_gemm_f8e4m3_tn.restype = ctypes.c_int
    lib.oracle_gemm_f8e4m3_tn.argtypes = [i64, i64, i64, p, i64, p, i64,
                                          ctypes.c_float, ctypes.c_float, p, i64, p, p]
    lib.oracle_gemm_f8e4m3_tn_at.restype = ctypes.c_int
    lib.oracle_gemm_f8e4m3_tn_at.argtypes = [i64, i64, i64, p, i64, p, i64,
                                             ctypes.c_float, ctypes.c_float,
                                             i64, p, p, p, p, p]
    lib.oracle_gemm_f16_tn_softmax_stats.restype = ctypes.c_int
    lib.oracle_gemm_f16_tn_softmax_stats.argtypes = [i64, i64, i64, p, i64, p, i64, ctypes.c_double,
                                                     p, i64, p, p, p]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
    lib.oracle_quantize_e4m3.restype = ctypes.c_int
    lib.oracle_quantize_e4m3.argtypes = [p, ctypes.c_int, i64, i64, i64, p, i64, p]
    lib.oracle_num_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# --- codecs (scalar; the tests sweep them) ---------------------------------
def fp16_decode(h: int) -> float:
    return _load().oracle_fp16_decode(h)


def fp16_encode(x: float) -> int:
    return _load().oracle_fp16_encode(x)


def bf16_encode(x: float) -> int:
    return _load().oracle_bf16_encode(x)


def bf16_decode(h: int) -> float:
    return _load().oracle_bf16_decode(h)


def e4m3_decode(q: int) -> float:
    return _load().oracle_e4m3_decode(q)


def e4m3_encode(x: float) -> int:
    return _load().oracle_e4m3_encode(x)


# --- per-tensor E4M3 quantisation -------------------------------------------
QUANT_IN = {"f32": (0, np.float32), "f16": (1, np.uint16), "bf16": (2, np.uint16)}


def quantize_e4m3(x: np.ndarray, x_type: str, rows: int, cols: int, ldx: int | None = None,
                  ldq: int | None = None):
    """amax over the tensor, s_q = 448 / amax (binary32), q = E4M3(x * s_q),
    scale = amax / 448.  x: float32 values ("f32") or binary16 / bfloat16
    codes ("f16" / "bf16"), rows x cols with row stride ldx.  Returns
    (q uint8 flat array with row stride ldq, scale as a Python float that is
    exactly a binary32 value)."""
    code, dt = QUANT_IN[x_type]
    ldx = max(cols, 1) if ldx is None else ldx
    ldq = max(cols, 1) if ldq is None else ldq
    x = np.ascontiguousarray(x, dtype=dt).reshape(-1)
    if rows > 0 and cols > 0 and x.size < (rows - 1) * ldx + cols:
        raise ValueError("x is smaller than (rows-1)*ldx + cols elements")
    q = np.zeros(max(rows * ldq, 1), dtype=np.uint8)
    scale = np.zeros(1, dtype=np.float32)
    rc = _load().oracle_quantize_e4m3(_ptr(x), code, rows, cols, ldx, _ptr(q), ldq, _ptr(scale))
    if rc != 0:
        raise ValueError("oracle_quantize_e4m3 rejected its arguments")
    return q, float(scale[0])


# --- GEMM -------------------------------------------------------------------
def _check_operands(A, B, M, N, K, lda, ldb, dtype):
    A = np.ascontiguousarray(A, dtype=dtype).reshape(-1)
    B = np.ascontiguousarray(B, dtype=dtype).reshape(-1)
    if M > 0 and K > 0 and A.size < (M - 1) * lda + K:
        raise ValueError("A is smaller than (M-1)*lda + K elements")
    if N > 0 and K > 0 and B.size < (N - 1) * ldb + K:
        raise ValueError("B is smaller than (N-1)*ldb + K elements")
    return A, B


def gemm_f16_tn(M, N, K, A, lda, B, ldb, ldc=None):
    """Full F16 oracle.  A, B: uint16 binary16 codes in TN storage.

    Returns (C, S, X): C uint16 codes, column-major with ldc (flat array of
    ldc*N elements, untouched padding rows are 0); S, X float64 (N, M) arrays
    (row n holds column n of the column-major result)."""
    ldc = M if ldc is None else ldc
    A, B = _check_operands(A, B, M, N, K, lda, ldb, np.uint16)
    C = np.zeros(max(ldc * N, 1), dtype=np.uint16)
    S = np.zeros((N, M), dtype=np.float64)
    X = np.zeros((N, M), dtype=np.float64)
    rc = _load().oracle_gemm_f16_tn(M, N, K, _ptr(A), lda, _ptr(B), ldb,
                                    _ptr(C), ldc, _ptr(S), _ptr(X))
    if rc != 0:
        raise ValueError("oracle_gemm_f16_tn rejected its arguments")
    return C, S, X


def gemm_f16_tn_at(M, N, K, A, lda, B, ldb, m_idx, n_idx):
    """F16 oracle at chosen output positions.  Returns (c, s, x) per position."""
    A, B = _check_operands(A, B, M, N, K, lda, ldb, np.uint16)
    m_idx = np.ascontiguousarray(m_idx, dtype=np.int64)
    n_idx = np.ascontiguousarray(n_idx, dtype=np.int64)
    cnt = m_idx.size
    c = np.zeros(cnt, dtype=np.uint16)
    s = np.zeros(cnt, dtype=np.float64)
    x = np.zeros(cnt, dtype=np.float64)
    rc = _load().oracle_gemm_f16_tn_at(M, N, K, _ptr(A), lda, _ptr(B), ldb, cnt,
                                       _ptr(m_idx), _ptr(n_idx), _ptr(c), _ptr(s), _ptr(x))
    if rc != 0:
        raise ValueError("oracle_gemm_f16_tn_at rejected its arguments")
    return c, s, x


def gemm_f16_tn_softmax_stats(M, N, K, A, lda, B, ldb, scale, ldc=None):
    """Scaled scores Y = scale * A B (C = binary16(Y), column-major with ldc)
    and per row m: row_max = max_n Y[m,n], row_sum = sum_n exp(Y[m,n] - row_max).
    Returns (C flat codes, row_max (M,), row_sum (M,), S (N, M))."""
    ldc = M if ldc is None else ldc
    A, B = _check_operands(A, B, M, N, K, lda, ldb, np.uint16)
    C = np.zeros(max(ldc * N, 1), dtype=np.uint16)
    row_max = np.full(M, np.nan)
    row_sum = np.full(M, np.nan)
    S = np.zeros((N, M), dtype=np.float64)
    rc = _load().oracle_gemm_f16_tn_softmax_stats(M, N, K, _ptr(A), lda, _ptr(B), ldb, float(scale),
                                                  _ptr(C), ldc, _ptr(row_max), _ptr(row_sum), _ptr(S))
    if rc != 0:
        raise ValueError("oracle_gemm_f16_tn_softmax_stats rejected its arguments")
    return C, row_max, row_sum, S


def gemm_f8e4m3_tn(M, N, K, A, lda, B, ldb, scale_a, scale_b, ldc=None):
    """Full F8 oracle.  A, B: uint8 E4M3 codes; returns (C bf16 codes, S, X)."""
    ldc = M if ldc is None else ldc
    A, B = _check_operands(A, B, M, N, K, lda, ldb, np.uint8)
    C = np.zeros(max(ldc * N, 1), dtype=np.uint16)
    S = np.zeros((N, M), dtype=np.float64)
    X = np.zeros((N, M), dtype=np.float64)
    rc = _load().oracle_gemm_f8e4m3_tn(M, N, K, _ptr(A), lda, _ptr(B), ldb,
                                       float(scale_a), float(scale_b),
                                       _ptr(C), ldc, _ptr(S), _ptr(X))
    if rc != 0:
        raise ValueError("oracle_gemm_f8e4m3_tn rejected its arguments")
    return C, S, X


def gemm_f8e4m3_tn_at(M, N, K, A, lda, B, ldb, scale_a, scale_b, m_idx, n_idx):
    A, B = _check_operands(A, B, M, N, K, lda, ldb, np.uint8)
    m_idx = np.ascontiguousarray(m_idx, dtype=np.int64)
    n_idx = np.ascontiguousarray(n_idx, dtype=np.int64)
    cnt = m_idx.size
    c = np.zeros(cnt, dtype=np.uint16)
    s = np.zeros(cnt, dtype=np.float64)
    x = np.zeros(cnt, dtype=np.float64)
    rc = _load().oracle_gemm_f8e4m3_tn_at(M, N, K, _ptr(A), lda, _ptr(B), ldb,
                                          float(scale_a), float(scale_b), cnt,
                                          _ptr(m_idx), _ptr(n_idx), _ptr(c), _ptr(s), _ptr(x))
    if rc != 0:
        raise ValueError("oracle_gemm_f8e4m3_tn_at rejected its arguments")
    return c, s, x


def c_as_nm(C: np.ndarray, M: int, N: int, ldc: int) -> np.ndarray:
    """View a flat column-major C (ldc*N codes) as an (N, M) array: row n is
    output column n, entry m is C[m + n*ldc]."""
    return C[: ldc * N].reshape(N, ldc)[:, :M] if N > 0 else np.zeros((0, M), C.dtype)
