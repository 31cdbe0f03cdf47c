"""Python binding of libdense_gemm_tn.so (the C ABI in include/tn_gemm.h).

Argument marshalling only: every step of the GEMM runs in the library's CUDA
kernels.  There is no CPU or PyTorch fallback -- importing this package
without the built library raises ImportError.

The same names as the C ABI:

    gemm_f16_tn(M, N, K, A, lda, B, ldb, C, ldc, stream=None)
    gemm_f8e4m3_tn(M, N, K, A, lda, B, ldb, C, ldc, scale_a, scale_b, stream=None)
    gemm_f8e4m3_tn_dscale(M, N, K, A, lda, B, ldb, C, ldc, scale_a_ptr, scale_b_ptr, stream=None)
    gemm_quantize_e4m3(x, x_type, rows, cols, ldx, q, ldq, scale_ptr, stream=None)
    gemm_f16_tn_softmax_stats(M, N, K, A, lda, B, ldb, C, ldc, scale, row_max, row_sum, stream=None)
    gemm_poll_device_status(stream=None)

A, B and C are device pointers given as ints or as CUDA torch tensors (their
data_ptr() is passed; the tensor's shape is NOT consulted).

Two bindings of the same C functions: `lib` (ctypes) and, where build()
found the Python headers, `fast` (the CPython-API module _tn_fast, built from
csrc/pyfast.c: the same names and argument order, ints for pointers, about a
tenth of the per-call host time).  `calls` is `fast` when present, else
`lib`; the wrappers below go through it.  `stream` is an
int handle, a torch.cuda.Stream, or None for torch's current stream.  A
status other than GEMM_OK raises GemmError.

Convenience wrappers over torch tensors in TN storage:
    f16_tn(A (M,K) fp16, Bt (N,K) fp16, C=None) -> C^T as an (N, M) fp16 tensor
    f8e4m3_tn(A (M,K) uint8/float8_e4m3fn, Bt (N,K), scale_a, scale_b, C=None) -> (N, M) bf16
The (N, M) row-major result IS the column-major M x N matrix C with ldc = M.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_UNSUPPORTED = 2
GEMM_ERR_CUDA = 3
GEMM_ERR_TIMEOUT = 4

LIB_PATH = _build.LIB

#: C symbols the header declares (checked by the test suite).
EXPORTS = (
    "gemm_f16_tn", "gemm_f8e4m3_tn", "gemm_status_string", "gemm_last_error",
    "gemm_poll_device_status", "gemm_release_workspace", "gemm_tile_coord",
    "gemm_set_wait_limit_ns", "gemm_debug_inject_stall", "gemm_build_info",
    "gemm_f16_tn_noalloc", "gemm_debug_force_cta_group", "gemm_debug_force_wide_tiles", "gemm_debug_last_launch",
    "gemm_debug_set_raster_group", "gemm_debug_set_k_order", "gemm_debug_set_long_k_mode", "gemm_debug_set_lean_mode",
    "gemm_debug_set_skinny_mode",
    "gemm_debug_set_clock_probe",
    "gemm_f8e4m3_tn_dscale", "gemm_quantize_e4m3", "gemm_f16_tn_softmax_stats",
)

GEMM_IN_F32 = 0
GEMM_IN_F16 = 1
GEMM_IN_BF16 = 2


class GemmError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{status_string(status)}: {detail}" if detail else status_string(status))


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
            "(nvcc for sm_103a); there is no fallback path")
    lib = ctypes.CDLL(LIB_PATH)
    i64, vp, st = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.gemm_f16_tn.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp]
    lib.gemm_f16_tn.restype = st
    lib.gemm_f8e4m3_tn.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64,
                                   ctypes.c_float, ctypes.c_float, vp]
    lib.gemm_f8e4m3_tn.restype = st
    lib.gemm_f8e4m3_tn_dscale.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, vp, vp]
    lib.gemm_f8e4m3_tn_dscale.restype = st
    lib.gemm_f16_tn_softmax_stats.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ctypes.c_float, vp, vp, vp]
    lib.gemm_f16_tn_softmax_stats.restype = st
    lib.gemm_quantize_e4m3.argtypes = [vp, st, i64, i64, i64, vp, i64, vp, vp]
    lib.gemm_quantize_e4m3.restype = st
    lib.gemm_f16_tn_noalloc.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp]
    lib.gemm_f16_tn_noalloc.restype = st
    lib.gemm_status_string.argtypes = [st]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_last_error.argtypes = []
    lib.gemm_last_error.restype = ctypes.c_char_p
    lib.gemm_poll_device_status.argtypes = [vp]
    lib.gemm_poll_device_status.restype = st
    lib.gemm_release_workspace.argtypes = []
    lib.gemm_release_workspace.restype = None
    lib.gemm_tile_coord.argtypes = [i64, i64, i64, i64, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    lib.gemm_tile_coord.restype = ctypes.c_int
    lib.gemm_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.gemm_set_wait_limit_ns.restype = None
    lib.gemm_debug_inject_stall.argtypes = [ctypes.c_int]
    lib.gemm_debug_inject_stall.restype = None
    lib.gemm_debug_force_cta_group.argtypes = [ctypes.c_int]
    lib.gemm_debug_force_cta_group.restype = ctypes.c_int
    lib.gemm_debug_force_wide_tiles.argtypes = [ctypes.c_int]
    lib.gemm_debug_force_wide_tiles.restype = ctypes.c_int
    lib.gemm_debug_set_raster_group.argtypes = [ctypes.c_int]
    lib.gemm_debug_set_raster_group.restype = ctypes.c_int
    lib.gemm_debug_set_clock_probe.argtypes = [ctypes.c_void_p]
    lib.gemm_debug_set_clock_probe.restype = None
    lib.gemm_debug_set_long_k_mode.argtypes = [ctypes.c_int]
    lib.gemm_debug_set_long_k_mode.restype = ctypes.c_int
    lib.gemm_debug_set_lean_mode.argtypes = [ctypes.c_int]
    lib.gemm_debug_set_lean_mode.restype = ctypes.c_int
    lib.gemm_debug_set_skinny_mode.argtypes = [ctypes.c_int]
    lib.gemm_debug_set_skinny_mode.restype = ctypes.c_int
    lib.gemm_debug_set_k_order.argtypes = [ctypes.c_int]
    lib.gemm_debug_set_k_order.restype = ctypes.c_int
    lib.gemm_debug_last_launch.argtypes = []
    lib.gemm_debug_last_launch.restype = ctypes.c_char_p
    lib.gemm_build_info.argtypes = []
    lib.gemm_build_info.restype = ctypes.c_char_p
    return lib


_lib = _load()
lib = _lib

try:
    # loads after _lib: it links the same library file, which the dynamic
    # loader then shares with the ctypes binding (one device state)
    from . import _tn_fast as fast
except ImportError:
    fast = None
calls = fast if fast is not None else _lib


def status_string(status: int) -> str:
    return _lib.gemm_status_string(int(status)).decode()


def last_error() -> str:
    return _lib.gemm_last_error().decode()


def last_launch() -> str:
    return _lib.gemm_debug_last_launch().decode()


def build_info() -> str:
    return _lib.gemm_build_info().decode()


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(status: int) -> int:
    if status != GEMM_OK:
        detail = last_error()
        if status == GEMM_ERR_CUDA and last_launch():
            detail += f" (last launch: {last_launch()})"
        raise GemmError(status, detail)
    return status


def gemm_f16_tn(M, N, K, A, lda, B, ldb, C, ldc, stream=None) -> int:
    return _check(calls.gemm_f16_tn(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, _stream(stream)))


def gemm_f8e4m3_tn(M, N, K, A, lda, B, ldb, C, ldc, scale_a, scale_b, stream=None) -> int:
    return _check(calls.gemm_f8e4m3_tn(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc,
                                       float(scale_a), float(scale_b), _stream(stream)))


def gemm_f8e4m3_tn_dscale(M, N, K, A, lda, B, ldb, C, ldc, scale_a, scale_b, stream=None) -> int:
    """gemm_f8e4m3_tn with scale_a / scale_b as device pointers (one fp32 each)."""
    return _check(calls.gemm_f8e4m3_tn_dscale(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc,
                                              _ptr(scale_a), _ptr(scale_b), _stream(stream)))


def gemm_f16_tn_softmax_stats(M, N, K, A, lda, B, ldb, C, ldc, scale, row_max, row_sum, stream=None) -> int:
    """Scaled scores C = fp16(scale * A B) with the softmax row statistics
    (row_max, row_sum: device float arrays of M)."""
    return _check(calls.gemm_f16_tn_softmax_stats(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, float(scale),
                                                  _ptr(row_max), _ptr(row_sum), _stream(stream)))


def gemm_quantize_e4m3(x, x_type, rows, cols, ldx, q, ldq, scale, stream=None) -> int:
    """Per-tensor E4M3 quantisation on the device: codes into q, amax / 448 into *scale."""
    return _check(calls.gemm_quantize_e4m3(_ptr(x), int(x_type), rows, cols, ldx, _ptr(q), ldq, _ptr(scale),
                                           _stream(stream)))


def gemm_f16_tn_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream=None) -> int:
    """gemm_f16_tn for callers that cannot let the library allocate device
    memory (their own memory pool or budget, or no implicit synchronisation
    allowed): operand copies go to a fixed 32 MiB array in the library's
    device image instead of a cudaMalloc'd workspace."""
    return _check(calls.gemm_f16_tn_noalloc(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc,
                                            _stream(stream)))


def gemm_poll_device_status(stream=None) -> int:
    return _check(_lib.gemm_poll_device_status(_stream(stream)))


def gemm_release_workspace() -> None:
    _lib.gemm_release_workspace()


def gemm_tile_coord(tiles_m, tiles_n, group, tile_id):
    tm, tn = ctypes.c_int64(), ctypes.c_int64()
    rc = _lib.gemm_tile_coord(tiles_m, tiles_n, group, tile_id, ctypes.byref(tm), ctypes.byref(tn))
    if rc != 0:
        raise ValueError("gemm_tile_coord: argument out of range")
    return tm.value, tn.value


def gemm_set_wait_limit_ns(limit_ns: int) -> None:
    _lib.gemm_set_wait_limit_ns(int(limit_ns))


def gemm_debug_inject_stall(mode) -> None:
    """0 off; 1 stall the MMA thread; 2 / 3 stall the even / odd CTA's producer."""
    _lib.gemm_debug_inject_stall(int(mode))


def gemm_debug_force_cta_group(group: int) -> None:
    if _lib.gemm_debug_force_cta_group(int(group)) != 0:
        raise ValueError("cta group must be 0 (automatic), 1 or 2")


def gemm_debug_force_wide_tiles(mode: int) -> None:
    """0 automatic; 1 CTA pairs always compute 256 x 512 tiles; -1 never."""
    if _lib.gemm_debug_force_wide_tiles(int(mode)) != 0:
        raise ValueError("mode must be -1, 0 or 1")


def gemm_debug_set_raster_group(rows: int) -> None:
    """Tile rows per raster group of the scheduler (even, 2 .. 64); 0 the default."""
    if _lib.gemm_debug_set_raster_group(int(rows)) != 0:
        raise ValueError("rows must be 0 or an even number up to 64")


def gemm_debug_set_k_order(mode: int) -> None:
    """0 the library's choice; 1 every tile walks K forward; 2 odd waves walk it backwards."""
    if _lib.gemm_debug_set_k_order(int(mode)) != 0:
        raise ValueError("mode must be 0, 1 or 2")


def gemm_debug_set_clock_probe(counters) -> None:
    """A device pointer (int) to 3 zeroed 64-bit words, or None: while set,
    each GEMM launch adds its SM cycles, nanoseconds and 1 to them."""
    _lib.gemm_debug_set_clock_probe(None if counters is None else ctypes.c_void_p(int(counters)))


def gemm_debug_set_long_k_mode(mode: int) -> None:
    """0 the library's choice; 1 split-reduce (HBM partials); 2 reduce inside a cluster of single CTAs."""
    if _lib.gemm_debug_set_long_k_mode(int(mode)) != 0:
        raise ValueError("mode must be 0, 1 or 2")


def gemm_debug_set_skinny_mode(mode: int) -> None:
    """N <= 64: 0 the library's choice; 1 never the skinny kernel; 2 always."""
    if _lib.gemm_debug_set_skinny_mode(int(mode)) != 0:
        raise ValueError("mode must be 0, 1 or 2")


def gemm_debug_set_lean_mode(mode: int) -> None:
    """m-part launches: 0 the library's choice; 1 the full configuration; 2 the
    lean one (two CTAs per SM) wherever the units are quarters or halves."""
    if _lib.gemm_debug_set_lean_mode(int(mode)) != 0:
        raise ValueError("mode must be 0, 1 or 2")


# ---------------------------------------------------------------- torch helpers
def _rows(t, dtype, name, shape=None, cuda=True):
    """Checks a 2-D CUDA tensor of `dtype` whose rows are contiguous (the layout
    the C ABI reads with a leading dimension) and returns its row stride."""
    import torch
    if not isinstance(t, torch.Tensor) or t.dim() != 2:
        raise ValueError(f"{name} must be a 2-D torch tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, not {t.dtype}")
    if t.numel() > 0 and t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit stride along its second dimension")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, not {tuple(t.shape)}")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.stride(0) if t.shape[0] > 1 else max(t.shape[1], 1)


def _operands(A, Bt, dtype):
    """(M, N, K, lda, ldb) of A (M, K) and Bt (N, K), both checked by _rows."""
    lda = _rows(A, dtype, "A", cuda=False)
    ldb = _rows(Bt, dtype, "Bt", cuda=False)
    (M, K), N = A.shape, Bt.shape[0]
    if Bt.shape[1] != K:
        raise ValueError(f"A is {tuple(A.shape)} and Bt {tuple(Bt.shape)}: their second dimensions (K) differ")
    for t, name in ((A, "A"), (Bt, "Bt")):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    if A.device != Bt.device:
        raise ValueError("A and Bt must be on the same device")
    return M, N, K, lda, ldb


def _output(C, M, N, dtype, device):
    import torch
    if C is None:
        C = torch.empty((N, M), dtype=dtype, device=device)
    ldc = _rows(C, dtype, "C", (N, M))
    if C.device != device:
        raise ValueError(f"C is on {C.device}, the operands on {device}")
    return C, ldc


def _on(device):
    """The C ABI works on the calling thread's current device: make it the
    operands' device for the call."""
    import torch
    return torch.cuda.device(device)


def f16_tn(A, Bt, C=None, stream=None):
    """C^T (N, M) = Bt (N, K) @ A (M, K)^T, i.e. column-major C = A x B.
    A, Bt (and C) are fp16 CUDA tensors whose rows are contiguous."""
    import torch
    M, N, K, lda, ldb = _operands(A, Bt, torch.float16)
    C, ldc = _output(C, M, N, torch.float16, A.device)
    with _on(A.device):
        gemm_f16_tn(M, N, K, A, lda, Bt, ldb, C, ldc, stream)
    return C


def f16_tn_softmax_stats(Q, Kmat, scale, C=None, stream=None):
    """Q (M, K) and Kmat (N, K) fp16 CUDA tensors -> (S^T as an (N, M) fp16
    tensor, row_max (M,), row_sum (M,)): S = scale * Q Kmat^T."""
    import torch
    M, N, K, lda, ldb = _operands(Q, Kmat, torch.float16)
    C, ldc = _output(C, M, N, torch.float16, Q.device)
    row_max = torch.empty(M, dtype=torch.float32, device=Q.device)
    row_sum = torch.empty(M, dtype=torch.float32, device=Q.device)
    with _on(Q.device):
        gemm_f16_tn_softmax_stats(M, N, K, Q, lda, Kmat, ldb, C, ldc, scale, row_max, row_sum, stream)
    return C, row_max, row_sum


def quantize_e4m3(x, stream=None):
    """x: a 2-D float32 / float16 / bfloat16 CUDA tensor with unit column
    stride.  Returns (codes as a uint8 tensor of x's shape, scale as a
    1-element float32 tensor), both on x's device."""
    import torch
    types = {torch.float32: GEMM_IN_F32, torch.float16: GEMM_IN_F16, torch.bfloat16: GEMM_IN_BF16}
    if x.dtype not in types or x.dim() != 2 or (x.numel() > 0 and x.stride(1) != 1):
        raise ValueError("x must be a 2-D float32/float16/bfloat16 tensor with unit column stride")
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    rows, cols = x.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    scale = torch.empty(1, dtype=torch.float32, device=x.device)
    ld = max(cols, 1)
    with _on(x.device):
        gemm_quantize_e4m3(x, types[x.dtype], rows, cols, x.stride(0) if rows > 1 else ld, q, ld, scale, stream)
    return q, scale


def _scale_tensor(t, name):
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda or t.numel() < 1:
        raise ValueError(f"{name} must be a float32 CUDA tensor with at least one element")


def f8e4m3_tn_dscale(A, Bt, scale_a, scale_b, C=None, stream=None):
    """f8e4m3_tn with the scales as 1-element float32 CUDA tensors.  A, Bt:
    uint8 E4M3 codes (CUDA, rows contiguous); C: bf16 (N, M)."""
    import torch
    M, N, K, lda, ldb = _operands(A, Bt, torch.uint8)
    _scale_tensor(scale_a, "scale_a")
    _scale_tensor(scale_b, "scale_b")
    if scale_a.device != A.device or scale_b.device != A.device:
        raise ValueError("scale_a and scale_b must be on the operands' device")
    C, ldc = _output(C, M, N, torch.bfloat16, A.device)
    with _on(A.device):
        gemm_f8e4m3_tn_dscale(M, N, K, A, lda, Bt, ldb, C, ldc, scale_a, scale_b, stream)
    return C


def f8e4m3_tn(A, Bt, scale_a, scale_b, C=None, stream=None):
    """C^T (N, M) = bf16(scale_a * scale_b * Bt A^T) for uint8 E4M3 codes A
    (M, K) and Bt (N, K); the scales are Python floats."""
    import torch
    M, N, K, lda, ldb = _operands(A, Bt, torch.uint8)
    C, ldc = _output(C, M, N, torch.bfloat16, A.device)
    with _on(A.device):
        gemm_f8e4m3_tn(M, N, K, A, lda, Bt, ldb, C, ldc, float(scale_a), float(scale_b), stream)
    return C
