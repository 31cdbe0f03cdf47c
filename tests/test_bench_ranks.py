"""The multi-process side of bench.py, on CPU with the gloo backend.

With N GPUs every rank runs its own replica of the GEMM (the path does not
shard), the ranks' times are max-reduced and the whole-job throughput counts
every rank's FLOPs over the slowest rank's time.  These tests run two ranks as
spawned processes with gloo on 127.0.0.1; no GPU is involved.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        total_ms, e2e_ms = bench.max_over_ranks(times[rank], dist, "cpu")
        flop = 2.0 * 64 * 32 * 16
        value = bench.replica_tflops(world, flop, 10, total_ms)
        out_q.put((rank, total_ms, e2e_ms, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo_2():
    world = 2
    times = [[3.0, 9.5], [4.5, 7.0]]          # (timed ms, e2e ms) per rank
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    flop = 2.0 * 64 * 32 * 16
    for rank, total_ms, e2e_ms, value in got:
        # every rank sees the slowest rank's times
        assert total_ms == 4.5 and e2e_ms == 9.5
        assert value == pytest.approx(world * flop * 10 / 4.5e-3 / 1e12, rel=1e-12)


def test_single_process_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.25, 2.5]) == [1.25, 2.5]
    assert bench.replica_tflops(1, 1e12, 1, 1000.0) == pytest.approx(1.0)


def test_reference_arm_other_ranks_exit_without_output():
    """Under torchrun only rank 0 runs the reference arm; rank 1 prints
    nothing and exits 0."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "pm1_512", "--steps", "1", "--warmup", "3", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_json_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "pm1_512", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_kernel_hash_ignores_comments_only():
    """A traffic record stays valid across comment edits, not across code edits."""
    import bench
    src = 'int a = 1; // one\n/* block\n comment */ const char *s = "x // not a comment";\n'
    assert bench.code_of(src) == 'int a = 1; const char *s = "x // not a comment";'
    assert bench.code_of(src.replace("// one", "// uno")) == bench.code_of(src)
    assert bench.code_of(src.replace("a = 1", "a = 2")) != bench.code_of(src)
    assert bench.code_of("char c = '\\\\'; // x") == "char c = '\\\\';"


def test_roofline_bound_peak_and_kernel_name():
    """The roofline object: HBM-bound below the ridge point (algorithmic bytes
    over the launch time against the copy bandwidth), tensor-bound above it
    against the burst peak for a region under a second and the sustained one
    beyond; the kernel named is the one the library ran."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    peaks = {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "src": "test"}
    sq = synth.WORKLOADS["sq_8192"]
    rf = bench.roofline_of(sq, 0.6, 12.0, peaks, {"sm_mhz": 1700.0}, 152, False)
    assert rf["bound"] == "tensor" and rf["peak_kind"] == "burst" and rf["peak"] == 1900.0
    assert abs(rf["achieved"] - 2.0 * 8192 ** 3 / 0.6e-3 / 1e12) < 1e-6
    assert rf["kernel"] == "tn_gemm_kernel<KindF16>"
    rf = bench.roofline_of(sq, 0.6, 2000.0, peaks, None, 152, False)
    assert rf["peak_kind"] == "sustained" and rf["peak"] == 1700.0
    e4 = synth.WORKLOADS["e4m3_8192"]
    rf = bench.roofline_of(e4, 0.3, 12.0, peaks, None, 152, False)
    assert rf["peak"] == 3800.0 and rf["kernel"] == "tn_gemm_kernel<KindE4M3>"
    sk = synth.WORKLOADS["skinny_8192x16x2048"]
    rf = bench.roofline_of(sk, 0.01, 20.0, peaks, None, 152, False, True)
    alg = (8192 * 2048 + 16 * 2048) * 2 + 2 * 8192 * 16
    assert rf["bound"] == "hbm" and rf["algorithmic_bytes"] == alg
    assert abs(rf["achieved"] - alg / 0.01e-3 / 1e9) < 1e-6 and rf["peak"] == 6800.0
    assert rf["kernel"] == "tn_skinny_kernel<KindF16>"
