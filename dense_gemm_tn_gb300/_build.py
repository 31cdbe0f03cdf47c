"""Builds libdense_gemm_tn.so in-tree with nvcc for sm_103a (no torch
extension machinery: the library is a plain C-ABI shared object), and the
CPython-API binding of its compute calls (_tn_fast, gcc) where the Python
headers are installed."""
from __future__ import annotations

import os
import shutil
import subprocess
import sysconfig

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libdense_gemm_tn.so")
SOURCES = [os.path.join(CSRC, "tn_gemm.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("tn_gemm_kernel.cuh", "sm103_ptx.cuh", "quant_e4m3_kernel.cuh", "repack_kernel.cuh",
                                                     "aux_kernels.cuh", "skinny_kernel.cuh")] + [
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


FAST_SRC = os.path.join(CSRC, "pyfast.c")
FAST = os.path.join(PKG, "_tn_fast" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))


def fast_build_cmd() -> list[str] | None:
    """gcc command for the CPython-API binding, or None without Python.h.  It
    links libdense_gemm_tn.so by an $ORIGIN run path, so the process shares the
    one copy of the library that the ctypes binding loads."""
    inc = sysconfig.get_paths().get("include", "")
    if not inc or not os.path.exists(os.path.join(inc, "Python.h")):
        return None
    cc = shutil.which("gcc") or shutil.which("cc") or "gcc"
    return [cc, "-O2", "-std=c11", "-shared", "-fPIC", "-Wall", "-I", INCLUDE, "-I", inc, "-o", FAST, FAST_SRC,
            "-L", PKG, "-ldense_gemm_tn", "-Wl,-rpath,$ORIGIN"]


def fast_stale() -> bool:
    if not os.path.exists(FAST):
        return True
    t = os.path.getmtime(FAST)
    return any(os.path.getmtime(f) > t for f in (FAST_SRC, os.path.join(INCLUDE, "tn_gemm.h"), LIB))


def build_fast(force: bool = False) -> str | None:
    """Builds the binding after the library; returns its path, or None when the
    Python headers are missing (the ctypes binding of the same calls remains)."""
    cmd = fast_build_cmd()
    if cmd is None:
        return None
    if force or fast_stale():
        subprocess.check_call(cmd)
    return FAST
