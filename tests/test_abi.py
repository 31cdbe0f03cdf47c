"""CPU-side checks of the C ABI: the library loads and exports every function
include/tn_gemm.h declares, host-side argument validation, the scheduler's
tile order, and the no-GPU failure mode.  No kernel runs here."""
import os
import re

import pytest

from tests.conftest import GOLDEN, ROOT

g = pytest.importorskip("dense_gemm_tn_gb300", reason="library not built")

HEADER = os.path.join(ROOT, "include", "tn_gemm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert "gemm_f16_tn" in names and "gemm_f8e4m3_tn" in names
    for n in names:
        assert hasattr(g.lib, n), n
    assert sorted(g.EXPORTS) == names


def test_status_strings():
    assert g.status_string(0) == "GEMM_OK"
    assert g.status_string(4) == "GEMM_ERR_TIMEOUT"
    assert g.status_string(99) == "GEMM_ERR_UNKNOWN"
    assert "sm_103a" in g.build_info()


BAD_ARGS = [
    dict(M=-1), dict(N=-1), dict(K=-1),
    dict(lda=3), dict(ldb=3), dict(ldc=7),
    dict(C=0), dict(A=0), dict(B=0), dict(C=0x1001),
]


@pytest.mark.parametrize("bad", BAD_ARGS)
def test_invalid_arguments_rejected_before_any_cuda_call(bad):
    args = dict(M=8, N=8, K=4, A=0x1000, lda=4, B=0x2000, ldb=4, C=0x3000, ldc=8)
    args.update(bad)
    st = g.lib.gemm_f16_tn(args["M"], args["N"], args["K"], args["A"], args["lda"], args["B"],
                           args["ldb"], args["C"], args["ldc"], None)
    assert st == g.GEMM_ERR_INVALID_ARG
    assert g.last_error() != ""
    st8 = g.lib.gemm_f8e4m3_tn(args["M"], args["N"], args["K"], args["A"], args["lda"], args["B"],
                               args["ldb"], args["C"], args["ldc"], 1.0, 1.0, None)
    assert st8 == g.GEMM_ERR_INVALID_ARG


def test_misaligned_f16_operand_rejected():
    assert g.lib.gemm_f16_tn(8, 8, 4, 0x1001, 4, 0x2000, 4, 0x3000, 8, None) == g.GEMM_ERR_INVALID_ARG
    # one-byte alignment is enough for e4m3 operands: this passes validation
    # and then fails only for lack of a device (or runs on a GPU machine; not here)


def test_oversized_dimensions_unsupported():
    assert g.lib.gemm_f16_tn(1 << 31, 8, 4, 0x1000, 4, 0x2000, 4, 0x3000, 1 << 31, None) == \
        g.GEMM_ERR_UNSUPPORTED


def test_empty_output_is_noop_without_device():
    assert g.lib.gemm_f16_tn(0, 8, 4, None, 4, None, 4, None, 1, None) == g.GEMM_OK
    assert g.lib.gemm_f16_tn(8, 0, 4, None, 4, None, 4, None, 8, None) == g.GEMM_OK


def test_no_device_reports_cuda_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = g.lib.gemm_f16_tn(8, 8, 4, 0x1000, 4, 0x2000, 4, 0x3000, 8, None)
    assert st == g.GEMM_ERR_CUDA


# ------------------------------------------------------------------ scheduler
def test_tile_order_matches_hand_mapping():
    """hello-gpu ch.11 section 11.3.4: 4 x 3 output blocks, GROUP_M = 1 and 2."""
    import json
    with open(os.path.join(GOLDEN, "group_m_mapping.json")) as f:
        gold = json.load(f)
    tm, tn = gold["tiles_m"], gold["tiles_n"]
    assert [list(g.gemm_tile_coord(tm, tn, 1, i)) for i in range(4)] == gold["group_1_first"]
    assert [list(g.gemm_tile_coord(tm, tn, 2, i)) for i in range(4)] == gold["group_2_first"]


def rocm_blog_step6(block, tiles_m, tiles_n, group):
    """The grouped block order as the ROCm blog's Step 6 states it (rows of
    tiles are grouped by `group`, the last group short)."""
    index_n = block % tiles_n
    index_m = block // tiles_n
    group_rows = group if index_m < tiles_m - tiles_m % group else tiles_m % group
    grp = index_m // group
    local = index_n + (index_m % group) * tiles_n
    return local % group_rows + grp * group, local // group_rows


@pytest.mark.parametrize("tiles_m,tiles_n,group", [(4, 3, 2), (32, 64, 8), (12, 97, 8), (13, 7, 8),
                                                   (1, 5, 8), (9, 1, 4), (24, 49, 8), (8, 8, 8)])
def test_tile_order_matches_step6_and_covers_grid(tiles_m, tiles_n, group):
    seen = set()
    for i in range(tiles_m * tiles_n):
        t = g.gemm_tile_coord(tiles_m, tiles_n, group, i)
        assert t == rocm_blog_step6(i, tiles_m, tiles_n, group)
        assert 0 <= t[0] < tiles_m and 0 <= t[1] < tiles_n
        seen.add(t)
    assert len(seen) == tiles_m * tiles_n


def test_tile_coord_rejects_out_of_range():
    with pytest.raises(ValueError):
        g.gemm_tile_coord(4, 3, 2, 12)
    with pytest.raises(ValueError):
        g.gemm_tile_coord(0, 3, 2, 0)
    with pytest.raises(ValueError):             # 2^32 tiles: more than the scheduler's 32-bit ids
        g.gemm_tile_coord(2 ** 20, 2 ** 12, 8, 0)


def test_raster_group_hook_rejects_odd_and_large():
    for bad in (-2, 3, 66):
        with pytest.raises(ValueError):
            g.gemm_debug_set_raster_group(bad)
    g.gemm_debug_set_raster_group(0)


def test_cta_group_hook_accepts_one_and_two_only():
    assert g.lib.gemm_debug_force_cta_group(4) == -1
    assert g.lib.gemm_debug_force_cta_group(3) == -1
    for v in (1, 2, 0):
        assert g.lib.gemm_debug_force_cta_group(v) == 0


def test_no_multicast_bulk_loads_in_library_sources():
    """No TMA copy in the library writes to several CTAs (cluster multicast):
    every CTA loads its own operand rows.  The one multicast form left is the
    tcgen05.commit that signals both CTAs of a pair that a stage was read."""
    csrc = os.path.join(ROOT, "dense_gemm_tn_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, name)).read()
        for line in text.splitlines():
            if "multicast::cluster" in line:
                assert "tcgen05.commit" in line, (name, line)
            assert not re.search(r"cp\.async\.bulk.*multicast", line), (name, line)


def test_k_order_hook_values():
    assert g.lib.gemm_debug_set_k_order(3) == -1
    assert g.lib.gemm_debug_set_k_order(-1) == -1
    for v in (1, 2, 0):
        assert g.lib.gemm_debug_set_k_order(v) == 0


def test_long_k_mode_hook_values():
    assert g.lib.gemm_debug_set_long_k_mode(3) == -1
    for v in (1, 2, 0):
        assert g.lib.gemm_debug_set_long_k_mode(v) == 0


def test_skinny_mode_hook_values():
    assert g.lib.gemm_debug_set_skinny_mode(3) == -1
    assert g.lib.gemm_debug_set_skinny_mode(-1) == -1
    for v in (1, 2, 0):
        assert g.lib.gemm_debug_set_skinny_mode(v) == 0


def test_lean_mode_hook_values():
    assert g.lib.gemm_debug_set_lean_mode(3) == -1
    assert g.lib.gemm_debug_set_lean_mode(-1) == -1
    for v in (1, 2, 0):
        assert g.lib.gemm_debug_set_lean_mode(v) == 0




# ---------------------------------------------------------------- the CPython-API binding
FAST = pytest.mark.skipif(g.fast is None, reason="the CPython-API binding was not built (no Python.h)")
FAST_CALLS = ("gemm_f16_tn", "gemm_f16_tn_noalloc", "gemm_f8e4m3_tn", "gemm_f8e4m3_tn_dscale",
              "gemm_f16_tn_softmax_stats", "gemm_quantize_e4m3")


def test_fast_binding_built_where_python_headers_exist():
    import sysconfig
    inc = sysconfig.get_paths().get("include", "")
    if os.path.exists(os.path.join(inc, "Python.h")):
        assert g.fast is not None and g.calls is g.fast
    else:
        assert g.calls is g.lib


@FAST
def test_fast_binding_exports_the_compute_calls():
    for name in FAST_CALLS:
        assert callable(getattr(g.fast, name)), name
        assert name in g.EXPORTS, name


@FAST
@pytest.mark.parametrize("bad", BAD_ARGS)
def test_fast_binding_returns_the_c_abi_status(bad):
    args = dict(M=8, N=8, K=4, A=0x1000, lda=4, B=0x2000, ldb=4, C=0x3000, ldc=8)
    args.update(bad)
    v = [args[k] for k in ("M", "N", "K", "A", "lda", "B", "ldb", "C", "ldc")]
    assert g.fast.gemm_f16_tn(*v, None) == g.lib.gemm_f16_tn(*v, None) == g.GEMM_ERR_INVALID_ARG
    assert g.fast.gemm_f16_tn_noalloc(*v, None) == g.lib.gemm_f16_tn_noalloc(*v, None)
    assert g.fast.gemm_f8e4m3_tn(*v, 1.0, 1.0, None) == g.lib.gemm_f8e4m3_tn(*v, 1.0, 1.0, None)
    assert g.fast.gemm_f8e4m3_tn_dscale(*v, 0x4000, 0x4004, None) == \
        g.lib.gemm_f8e4m3_tn_dscale(*v, 0x4000, 0x4004, None) == g.GEMM_ERR_INVALID_ARG
    assert g.fast.gemm_f16_tn_softmax_stats(*v, 0.5, 0x5000, 0x6000, None) == \
        g.lib.gemm_f16_tn_softmax_stats(*v, 0.5, 0x5000, 0x6000, None) == g.GEMM_ERR_INVALID_ARG


@FAST
def test_fast_binding_quantiser_argument_checks():
    # an unknown element type and a negative size fail validation in both bindings
    for args in ((0x1000, 7, 4, 4, 4, 0x2000, 4, 0x3000, None), (0x1000, 0, -1, 4, 4, 0x2000, 4, 0x3000, None)):
        assert g.fast.gemm_quantize_e4m3(*args) == g.lib.gemm_quantize_e4m3(*args) == g.GEMM_ERR_INVALID_ARG


@FAST
def test_fast_binding_empty_output_is_noop():
    assert g.fast.gemm_f16_tn(0, 8, 4, None, 4, None, 4, None, 1, None) == g.GEMM_OK


@FAST
def test_fast_binding_rejects_malformed_arguments():
    with pytest.raises(TypeError):
        g.fast.gemm_f16_tn(8, 8, 4)
    with pytest.raises(TypeError):
        g.fast.gemm_f16_tn(8, 8, 4, "A", 4, 0x2000, 4, 0x3000, 8, None)
    with pytest.raises(TypeError):
        g.fast.gemm_f8e4m3_tn(8, 8, 4, 0x1000, 4, 0x2000, 4, 0x3000, 8, "s", 1.0, None)
    with pytest.raises(OverflowError):
        g.fast.gemm_f16_tn(1 << 70, 8, 4, 0x1000, 4, 0x2000, 4, 0x3000, 8, None)
    with pytest.raises(OverflowError):
        g.fast.gemm_quantize_e4m3(0x1000, 1 << 40, 4, 4, 4, 0x2000, 4, 0x3000, None)


@FAST
def test_fast_binding_shares_the_one_library_copy():
    # the binding links libdense_gemm_tn.so by run path; the loader maps the file
    # ctypes opened once, so both see one device state
    with open("/proc/self/maps") as f:
        paths = {line.split()[-1] for line in f if "libdense_gemm_tn" in line}
    assert paths == {os.path.realpath(g.LIB_PATH)}
