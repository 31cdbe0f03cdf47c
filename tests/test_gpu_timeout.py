"""Bounded waits on the GPU: a kernel whose wait runs out records
GEMM_ERR_TIMEOUT, drains its copies, frees its tensor memory and returns;
the context stays usable.  The wait is made to run out with a barrier that
nothing arrives on (no fault, no hang)."""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_helpers import check_f16_full, to_dev_u16, GuardedC

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cta_group", [1, 2])
def test_stalled_wait_reports_timeout_and_context_survives(cta_group):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    g.gemm_debug_force_cta_group(cta_group)
    M, N, K = 256, 256, 256
    A = synth.gauss_fp16(M * K, 1)
    B = synth.gauss_fp16(N * K, 2)
    dA, dB = to_dev_u16(A), to_dev_u16(B)
    C = GuardedC(M, N, M)
    g.gemm_set_wait_limit_ns(50_000_000)      # 50 ms
    g.gemm_debug_inject_stall(True)
    try:
        g.gemm_f16_tn(M, N, K, dA, K, dB, K, C.ptr, M)
        with pytest.raises(g.GemmError) as err:
            g.gemm_poll_device_status()
        assert err.value.status == g.GEMM_ERR_TIMEOUT
    finally:
        g.gemm_debug_inject_stall(False)
        g.gemm_set_wait_limit_ns(0)
        g.gemm_debug_force_cta_group(0)
    C.host()                                   # canaries intact
    # the status word was cleared and the next call computes correctly
    g.gemm_poll_device_status()
    check_f16_full(M, N, K, A, B, what="after timeout")
