"""Seeded synthetic inputs for the TN GEMM workloads.

Shared by the tests and ``bench.py``; it holds none of the GEMM's arithmetic
(see ``synth.c`` for the generator's definition: SplitMix64 per element index,
Box-Muller in double, one round-to-nearest-even cast to binary16 or a
saturating cast to OCP E4M3FN).

Operands are produced in the TN storage of the AMD ROCm blog "FP16 GEMM
optimization on AMD RDNA 3 and RDNA 4" (section "What we compute"):
A row-major M x K (element index m*K + k), B column-major K x N (element index
k + n*K), i.e. B is handed over as an (N, K) row-major array.

Workloads (shapes and value distributions of the pages' benchmarks).  The
benchmark cycles through `rotating` input sets, enough that together they are
larger than the GPU's L2 (129 MB), so every step reads its operands from HBM:
  pm1_512      M=N=K=512, entries uniform {-1,+1}, 160 sets of 1 MiB (exact case)
  qk_1024      M=N=1024, K=128, N(0,1) cast to fp16, 320 sets of 0.5 MiB
               (QK^T-shaped block)
  sq_8192      M=N=K=8192, N(0,1) cast to fp16, 4 rotating sets (headline)
  wide_pm1     M=3000, N=12289, K=4097, uniform {-1,+1}, 2 sets    (tails)
  wide_gauss   M=3000, N=12289, K=4097, N(0,1) cast to fp16, 2 sets (tails)
  e4m3_8192    M=N=K=8192, N(0,1) scaled per tensor to max|x| = 448 and
               cast to E4M3, 4 rotating sets
  ffn_8192     M=8192, N=28672, K=8192, N(0,1) cast to fp16, 2 rotating
               sets (the wide feed-forward projection shape)
  qk_stats_1024  qk_1024's inputs (320 sets) through the fused attention-score
               epilogue (scale 1/sqrt(K), softmax row statistics)
  fp8_pipeline_8192  M=N=K=8192, N(0,1) cast to bfloat16, 2 rotating sets;
               each step quantises both operands to E4M3 on the device
               before the FP8 GEMM
  longk_4096x512  M=4096, N=512, K=8192, N(0,1) cast to fp16, 2 rotating
               sets: a grid of fewer tiles than half the GPU with a long K
               (its k ranges are reduced inside clusters)
  skinny_8192x16  M=8192, N=16, K=8192, N(0,1) cast to fp16, 2 rotating sets:
               a decode-like product, bound by the read of A
  skinny_8192x16x2048  M=8192, N=16, K=2048, N(0,1) cast to fp16, 6 rotating
               sets: the same product with a shorter K (the kernel for few
               columns n)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None


def build_cmd() -> list[str]:
    return ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC",
            "-o", _LIB, _SRC, "-lm"]


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(build_cmd())
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    p, i64, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64
    for name in ("synth_sign_fp16", "synth_gauss_f64", "synth_gauss_fp16", "synth_gauss_bf16", "synth_raw"):
        getattr(lib, name).argtypes = [p, i64, u64]
        getattr(lib, name).restype = None
    lib.synth_gauss_absmax.argtypes = [i64, u64]
    lib.synth_gauss_absmax.restype = ctypes.c_double
    lib.synth_gauss_e4m3.argtypes = [p, i64, u64, ctypes.c_double]
    lib.synth_gauss_e4m3.restype = None
    lib.synth_f64_to_fp16.argtypes = [p, p, i64]
    lib.synth_f64_to_e4m3.argtypes = [p, p, i64]
    lib.synth_f64_to_bf16.argtypes = [p, p, i64]
    _lib = lib
    return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def raw(n: int, seed: int) -> np.ndarray:
    out = np.empty(n, np.uint64)
    _load().synth_raw(_p(out), n, seed)
    return out


def sign_fp16(n: int, seed: int, out: np.ndarray | None = None) -> np.ndarray:
    """n binary16 codes, each +1 (0x3C00) or -1 (0xBC00)."""
    out = np.empty(n, np.uint16) if out is None else out
    _load().synth_sign_fp16(_p(out), n, seed)
    return out


def gauss_f64(n: int, seed: int) -> np.ndarray:
    out = np.empty(n, np.float64)
    _load().synth_gauss_f64(_p(out), n, seed)
    return out


def gauss_fp16(n: int, seed: int, out: np.ndarray | None = None) -> np.ndarray:
    """n N(0,1) draws rounded to binary16 codes."""
    out = np.empty(n, np.uint16) if out is None else out
    _load().synth_gauss_fp16(_p(out), n, seed)
    return out


def gauss_bf16(n: int, seed: int, out: np.ndarray | None = None) -> np.ndarray:
    """n N(0,1) draws rounded to bfloat16 codes."""
    out = np.empty(n, np.uint16) if out is None else out
    _load().synth_gauss_bf16(_p(out), n, seed)
    return out


def gauss_e4m3(n: int, seed: int, out: np.ndarray | None = None):
    """n N(0,1) draws quantised per tensor to E4M3.

    The quantisation multiplier is s_q = 448 / max|x| (fp32), so the largest
    draw maps to 448; the returned dequantisation factor is
    scale = max|x| / 448 (fp32), the value the GEMM multiplies its
    accumulator by.  Returns (codes uint8, scale float)."""
    lib = _load()
    amax = lib.synth_gauss_absmax(n, seed)
    amax32 = np.float32(amax)
    s_q = np.float32(448.0) / amax32
    scale = amax32 / np.float32(448.0)
    out = np.empty(n, np.uint8) if out is None else out
    lib.synth_gauss_e4m3(_p(out), n, seed, float(s_q))
    return out, float(scale)


def f64_to_fp16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty(x.size, np.uint16)
    _load().synth_f64_to_fp16(_p(out), _p(x), x.size)
    return out


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty(x.size, np.uint16)
    _load().synth_f64_to_bf16(_p(out), _p(x), x.size)
    return out


def f64_to_e4m3(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty(x.size, np.uint8)
    _load().synth_f64_to_e4m3(_p(out), _p(x), x.size)
    return out


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    values: str          # "pm1", "gauss", "e4m3", or "bf16" (quantised to E4M3 on the device)
    seed_a: int
    seed_b: int
    rotating: int = 1    # input sets cycled by the benchmark
    op: str = "gemm"     # "gemm", or "softmax_stats": scaled scores plus softmax row statistics

    @property
    def dtype(self) -> str:
        """Element type of the GEMM's operands."""
        return "e4m3" if self.values in ("e4m3", "bf16") else "f16"

    def seeds(self, i: int) -> tuple[int, int]:
        """Seeds of rotating input set i (sets differ by 2 per step)."""
        return self.seed_a + 2 * i, self.seed_b + 2 * i


WORKLOADS = {
    w.name: w for w in [
        Workload("pm1_512", 512, 512, 512, "pm1", 101, 102, rotating=160),
        Workload("qk_1024", 1024, 1024, 128, "gauss", 201, 202, rotating=320),
        Workload("sq_8192", 8192, 8192, 8192, "gauss", 301, 302, rotating=4),
        Workload("wide_pm1", 3000, 12289, 4097, "pm1", 401, 402, rotating=2),
        Workload("wide_gauss", 3000, 12289, 4097, "gauss", 403, 404, rotating=2),
        Workload("e4m3_8192", 8192, 8192, 8192, "e4m3", 501, 502, rotating=4),
        Workload("ffn_8192", 8192, 28672, 8192, "gauss", 601, 602, rotating=2),
        Workload("fp8_pipeline_8192", 8192, 8192, 8192, "bf16", 701, 702, rotating=2),
        Workload("qk_stats_1024", 1024, 1024, 128, "gauss", 201, 202, rotating=320, op="softmax_stats"),
        Workload("longk_4096x512", 4096, 512, 8192, "gauss", 801, 802, rotating=2),
        Workload("skinny_8192x16", 8192, 16, 8192, "gauss", 803, 804, rotating=2),
        Workload("skinny_8192x16x2048", 8192, 16, 2048, "gauss", 805, 806, rotating=6),
    ]
}


def operand(values: str, rows: int, K: int, seed: int):
    """One K-contiguous operand (rows x K, dense) as a flat code array.

    Returns (codes, scale); scale is 1.0 except for E4M3 operands."""
    n = rows * K
    if values == "pm1":
        return sign_fp16(n, seed), 1.0
    if values == "gauss":
        return gauss_fp16(n, seed), 1.0
    if values == "e4m3":
        return gauss_e4m3(n, seed)
    if values == "bf16":
        return gauss_bf16(n, seed), 1.0
    raise ValueError(values)


def make_inputs(w: Workload, i: int = 0):
    """Rotating set i of workload w: (A codes (M*K), B codes (N*K), scale_a, scale_b)."""
    sa_seed, sb_seed = w.seeds(i)
    A, sa = operand(w.values, w.M, w.K, sa_seed)
    B, sb = operand(w.values, w.N, w.K, sb_seed)
    return A, B, sa, sb
