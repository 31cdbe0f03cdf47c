"""Calls from several host threads at once, each on its own stream.

The library keeps per-device state (tile-shape caches, the tensor-map cache)
and per-(device, stream) buffers (split-K and split-reduce partials), guarded
internally.  Four threads drive every launch mode concurrently -- split
reduce, split-K tail, m-part units, 256 x 512 tiles, plain tiles -- each on
its own stream and buffers (ctypes releases the GIL during each call).  +-1
inputs: every sampled output is the oracle's bits.  A thread that has made
no CUDA call before its first GEMM gets the device's context from the
library.  Operands the TMA cannot address in place are copied into each
stream's own workspace, so those calls run at once too.
"""
import threading

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import sample_positions, to_dev_u16

pytestmark = pytest.mark.gpu

SHAPES = [
    (1024, 1024, 8192),     # split-reduce: 32 one-CTA tiles, four k ranges each
    (2000, 3000, 520),      # 96 pair tiles: a split-K last wave
    (1024, 1024, 128),      # m-part units
    (4096, 4096, 1024),     # 256 x 512 pair tiles
    (3000, 2000, 136),      # plain pair tiles
    (1000, 700, 1001),      # K * 2 bytes not a 16-byte multiple: operands copied into the stream's workspace
]
THREADS = 4
ROUNDS = 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import dense_gemm_tn_gb300 as g
    return g


@pytest.mark.parametrize("per_thread_default", [False, True])
def test_concurrent_threads_each_on_its_own_stream(per_thread_default):
    """per_thread_default: every thread passes cudaStreamPerThread (one handle
    value, a different stream on each thread) instead of a stream of its own."""
    import dense_gemm_tn_gb300 as g
    host = {}
    dev = {}
    for t in range(THREADS):
        for i, (M, N, K) in enumerate(SHAPES):
            A = synth.sign_fp16(M * K, 1000 * t + 2 * i + 1)
            B = synth.sign_fp16(N * K, 1000 * t + 2 * i + 2)
            host[t, i] = (A, B)
            dev[t, i] = (to_dev_u16(A), to_dev_u16(B),
                         torch.full((N, M), 0x7E00, dtype=torch.int16, device="cuda"))
    torch.cuda.synchronize()
    errors, records = [], {}
    streams = [torch.cuda.Stream() for _ in range(THREADS)]   # made here: the workers make no torch call

    def worker(t):
        try:
            handle = 0x2 if per_thread_default else streams[t].cuda_stream
            for r in range(ROUNDS):
                for i, (M, N, K) in enumerate(SHAPES):
                    dA, dB, C = dev[t, i]
                    rc = g.lib.gemm_f16_tn(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, C.data_ptr(), M, handle)
                    if rc != 0:
                        errors.append(f"thread {t} shape {i}: status {rc}: {g.last_error()}")
                        return
                    records[t, i] = g.last_launch()
        except Exception as e:          # reported below, on the main thread
            errors.append(f"thread {t}: {e!r}")

    workers = [threading.Thread(target=worker, args=(t,)) for t in range(THREADS)]
    for w in workers:
        w.start()
    for w in workers:
        w.join()
    torch.cuda.synchronize()          # (the per-thread default streams synchronise with the device too)
    g.gemm_poll_device_status()
    assert not errors, errors
    for t in range(THREADS):
        for i, (M, N, K) in enumerate(SHAPES):
            # the launch record is per host thread: set by this thread's own call of this shape
            assert records[t, i].startswith("gemm_f16_tn:"), (t, i, records[t, i])
            A, B = host[t, i]
            got = dev[t, i][2].cpu().numpy().view(np.uint16)
            mi, ni = sample_positions(M, N, 4000, seed=7 * t + i)
            c, _, _ = oracle.gemm_f16_tn_at(M, N, K, A, K, B, K, mi, ni)
            bad = np.flatnonzero(got[ni, mi] != c)
            assert bad.size == 0, f"thread {t} shape {(M, N, K)}: {bad.size} sampled outputs differ"


GROWING = [(500, 300, 1001), (1000, 700, 1001), (1024, 1024, 8192), (2000, 1500, 2049), (2048, 1024, 8192),
           (3000, 2000, 4097)]


def test_threads_share_the_default_stream_while_buffers_grow():
    """Every thread issues its calls on the legacy default stream, so all of
    them share that stream's buffers.  The shapes grow the row-copy workspace
    (K * 2 bytes not a 16-byte multiple) and the split-reduce partials (a long
    K on a small grid) while other threads may be between looking a buffer up
    and launching into it; one more thread releases the workspaces now and
    then.  +-1 inputs: every sampled output is the oracle's bits."""
    import dense_gemm_tn_gb300 as g
    host, dev = {}, {}
    for t in range(THREADS):
        for i, (M, N, K) in enumerate(GROWING):
            A = synth.sign_fp16(M * K, 5000 + 100 * t + 2 * i)
            B = synth.sign_fp16(N * K, 5001 + 100 * t + 2 * i)
            host[t, i] = (A, B)
            dev[t, i] = (to_dev_u16(A), to_dev_u16(B),
                         torch.full((N, M), 0x7E00, dtype=torch.int16, device="cuda"))
    torch.cuda.synchronize()
    g.gemm_release_workspace()
    errors = []
    stop = threading.Event()

    def worker(t):
        try:
            for r in range(3):
                order = GROWING if (t + r) % 2 == 0 else GROWING[::-1]
                for (M, N, K) in order:
                    i = GROWING.index((M, N, K))
                    dA, dB, C = dev[t, i]
                    rc = g.lib.gemm_f16_tn(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, C.data_ptr(), M, None)
                    if rc != 0:
                        errors.append(f"thread {t} shape {i}: status {rc}: {g.last_error()}")
                        return
        except Exception as e:          # reported below, on the main thread
            errors.append(f"thread {t}: {e!r}")

    def releaser():
        while not stop.wait(0.02):
            g.gemm_release_workspace()

    workers = [threading.Thread(target=worker, args=(t,)) for t in range(THREADS)]
    rel = threading.Thread(target=releaser)
    rel.start()
    for w in workers:
        w.start()
    for w in workers:
        w.join()
    stop.set()
    rel.join()
    torch.cuda.synchronize()
    g.gemm_poll_device_status()
    assert not errors, errors
    for t in range(THREADS):
        for i, (M, N, K) in enumerate(GROWING):
            A, B = host[t, i]
            got = dev[t, i][2].cpu().numpy().view(np.uint16)
            mi, ni = sample_positions(M, N, 3000, seed=11 * t + i)
            c, _, _ = oracle.gemm_f16_tn_at(M, N, K, A, K, B, K, mi, ni)
            bad = np.flatnonzero(got[ni, mi] != c)
            assert bad.size == 0, f"thread {t} shape {(M, N, K)}: {bad.size} sampled outputs differ"
