"""Builds libdense_gemm_tn.so in-tree with nvcc for sm_103a (no torch
extension machinery: the library is a plain C-ABI shared object)."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libdense_gemm_tn.so")
SOURCES = [os.path.join(CSRC, "tn_gemm.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("tn_gemm_kernel.cuh", "sm103_ptx.cuh", "quant_e4m3_kernel.cuh", "repack_kernel.cuh",
                                                     "aux_kernels.cuh")] + [
    os.path.join(INCLUDE, "tn_gemm.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def build_cmd(verbose_ptxas: bool = False) -> list[str]:
    cmd = [nvcc(), "-std=c++17", "-O3", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
           "-diag-suppress", "1160", "-I", INCLUDE, "-o", LIB, *SOURCES]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in DEPENDS)


def build(force: bool = False) -> str:
    if force or stale():
        subprocess.check_call(build_cmd())
    return LIB
