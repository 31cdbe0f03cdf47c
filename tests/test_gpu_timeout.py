"""Bounded waits on the GPU: a kernel whose wait runs out records
GEMM_ERR_TIMEOUT, drains its copies in flight, frees its tensor memory and
returns; the context stays usable.  The wait is made to run out with a
barrier that nothing arrives on (no fault, no hang), in the MMA thread or in
one CTA's TMA producer -- the latter leaves the two CTAs of a pair with
different numbers of loads in flight, which the drain must settle."""
import pytest
import torch

import synth
from tests.gpu_helpers import GuardedC, check_f16_full, to_dev_u16

pytestmark = pytest.mark.gpu

# (CTAs per cluster, 256 x 512 pair tiles, stalled thread)
CASES = [(1, 0, 1), (1, 0, 2), (2, 0, 1), (2, 0, 2), (2, 0, 3), (2, 1, 1), (2, 1, 2), (2, 1, 3)]


@pytest.mark.parametrize("group", [1, 2])
@pytest.mark.parametrize("mode", [1, 2, 3])
def test_stalled_wait_in_a_reducing_cluster(mode, group):
    """The k ranges of each tile in a cluster of single CTAs or CTA pairs: a
    stalled MMA thread or producer (of cluster CTA 0 or 1) times out; the
    other CTAs, waiting for their peers' partials, leave through the abort
    flag."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    M, N, K = 1024, 1024, 8192
    A = synth.gauss_fp16(M * K, 3)
    B = synth.gauss_fp16(N * K, 4)
    dA, dB = to_dev_u16(A), to_dev_u16(B)
    C = GuardedC(M, N, M)
    g.gemm_debug_force_cta_group(group)
    g.gemm_debug_set_long_k_mode(2)
    g.gemm_set_wait_limit_ns(50_000_000)
    g.gemm_debug_inject_stall(mode)
    try:
        g.gemm_f16_tn(M, N, K, dA, K, dB, K, C.ptr, M)
        assert "tail_mode=4" in g.last_launch(), g.last_launch()
        with pytest.raises(g.GemmError) as err:
            g.gemm_poll_device_status()
        assert err.value.status == g.GEMM_ERR_TIMEOUT
    finally:
        g.gemm_debug_inject_stall(0)
        g.gemm_set_wait_limit_ns(0)
    C.host()
    g.gemm_poll_device_status()
    try:
        check_f16_full(M, N, K, A, B, what=f"after timeout in a reducing cluster, mode {mode}")
    finally:
        g.gemm_debug_force_cta_group(0)
        g.gemm_debug_set_long_k_mode(0)


@pytest.mark.parametrize("cta_group,wide,mode", CASES)
def test_stalled_wait_reports_timeout_and_context_survives(cta_group, wide, mode):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    M, N, K = 512, 512, 1024       # several tiles and more k-blocks than stages
    A = synth.gauss_fp16(M * K, 1)
    B = synth.gauss_fp16(N * K, 2)
    dA, dB = to_dev_u16(A), to_dev_u16(B)
    C = GuardedC(M, N, M)
    g.gemm_debug_force_cta_group(cta_group)
    g.gemm_debug_force_wide_tiles(wide if wide else -1)
    g.gemm_set_wait_limit_ns(50_000_000)      # 50 ms
    g.gemm_debug_inject_stall(mode)
    try:
        g.gemm_f16_tn(M, N, K, dA, K, dB, K, C.ptr, M)
        with pytest.raises(g.GemmError) as err:
            g.gemm_poll_device_status()
        assert err.value.status == g.GEMM_ERR_TIMEOUT
    finally:
        g.gemm_debug_inject_stall(0)
        g.gemm_set_wait_limit_ns(0)
    C.host()                                   # canaries intact
    # the status word was cleared and the next call (same tile shape) is right
    g.gemm_poll_device_status()
    try:
        check_f16_full(M, N, K, A, B, what=f"after timeout, group {cta_group} wide {wide} mode {mode}")
    finally:
        g.gemm_debug_force_cta_group(0)
        g.gemm_debug_force_wide_tiles(0)

