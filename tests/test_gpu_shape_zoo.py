"""Parity on shapes beyond the benchmark workloads: large and tall problems,
long K, decode-like skinny N, and the feed-forward variants, each of which
takes another tile shape, tail mode or k-range cut.  +-1 inputs make every
FP32 sum an exact integer, so C must equal the oracle's one rounding of it
bit for bit on every sampled output (tile edges included); a second call must
return the same bits."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import run_f16, sample_positions

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    return g


SHAPES = [
    (12288, 12288, 12288),   # 256 x 512 pair tiles: 15 waves and a short one (cut into m halves)
    (32768, 1024, 1024),     # tall: 64 x 2 wide tiles
    (2048, 2048, 2048),      # medium: about one wave
    (8192, 4096, 14336),     # long K on a full grid
    (4096, 14336, 4096),     # the feed-forward variant with N = 14336
    (8192, 64, 8192),        # skinny N: k ranges reduced in clusters, 64 of 128 rows n valid
    (16384, 128, 4096),      # one tile row n, 64 tiles m
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_shape_pm1_sampled_exact_and_repeatable(M, N, K):
    A = synth.sign_fp16(M * K, 9500 + M % 97)
    B = synth.sign_fp16(N * K, 9600 + N % 97)
    got = run_f16(M, N, K, A, K, B, K)
    mi, ni = sample_positions(M, N, 20000, seed=M + N + K)
    want, _, _ = oracle.gemm_f16_tn_at(M, N, K, A, K, B, K, mi, ni)
    assert np.array_equal(got[ni, mi], want), f"{np.sum(got[ni, mi] != want)} sampled outputs differ"
    again = run_f16(M, N, K, A, K, B, K)
    assert np.array_equal(got, again)
