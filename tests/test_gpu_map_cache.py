"""The host's tensor-map cache under many distinct buffers.

Each call encodes (or finds) maps for A, B and C keyed by address, shape,
stride and box.  3000 calls on distinct slices of large buffers need about
9000 maps: more than the cache holds, so it evicts while the calls run, and
every call must still compute on its own operands.  +-1 inputs: bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import to_dev_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    return g


def test_many_distinct_buffers_each_call_reads_its_own():
    import dense_gemm_tn_gb300 as g
    M, N, K = 64, 48, 64
    calls = 3000
    step = 64                                  # elements between consecutive operand slices (128 bytes)
    A = synth.sign_fp16(calls * step + M * K, 601)
    B = synth.sign_fp16(calls * step + N * K, 602)
    dA, dB = to_dev_u16(A), to_dev_u16(B)
    C = torch.full((calls, N * M), 0x7E00, dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    for i in range(calls):
        j = (7 * i) % calls                    # B slices in another order than A's
        g.gemm_f16_tn(M, N, K, dA.data_ptr() + 2 * step * i, K, dB.data_ptr() + 2 * step * j, K, C[i].data_ptr(), M, s)
    g.gemm_poll_device_status(s)
    got = C.cpu().numpy().view(np.uint16)
    for i in range(calls):
        j = (7 * i) % calls
        ref, _, _ = oracle.gemm_f16_tn(M, N, K, A[step * i: step * i + M * K], K, B[step * j: step * j + N * K], K)
        assert np.array_equal(got[i], ref[: N * M]), f"call {i}"
