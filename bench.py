#!/usr/bin/env python3
"""Throughput of the sm_103a TN GEMM: TFLOP/s = 2MNK / t on one GB300.

One step = one call of the C ABI on one rotating input set of the workload
(default sq_8192: FP16, M = N = K = 8192, N(0,1) inputs, 4 rotating sets of
256 MiB each, larger than L2, so no L2 flush is needed between steps).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

Prints ONE JSON line on rank 0.  Under torchrun (N > 1) every rank runs its
own replica on its own GPU (the GEMM does not shard across GPUs here), times
are max-reduced, and `value` sums all ranks' FLOPs ("scaling": "weak").
--impl reference times the CPU oracle (fp64 triple loop) on a bounded sample
of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "TFLOP/s (2MNK/t) FP16 TN GEMM 8192³ on 1 GB300; % of dense tensor peak"
NOMINAL_PEAK = {"f16": 2250.0, "e4m3": 4500.0}          # dense TFLOP/s per GPU
KERNEL_NAME = {"f16": "tn_gemm_kernel<KindF16>", "e4m3": "tn_gemm_kernel<KindE4M3>"}
KERNEL_SOURCES = ["dense_gemm_tn_gb300/csrc/tn_gemm_kernel.cuh", "dense_gemm_tn_gb300/csrc/sm103_ptx.cuh"]
PROFILES_DIR = os.path.join(ROOT, "profiles")


def metric_for(w: synth.Workload) -> str:
    if w.name == "sq_8192":
        return METRIC
    what = "FP8 e4m3" if w.dtype == "e4m3" else "FP16"
    if w.values == "bf16":
        what = "bf16 -> e4m3 quantise + FP8"
    if w.op == "softmax_stats":
        what = "FP16 scaled scores + softmax row statistics,"
    return f"TFLOP/s (2MNK/t) {what} TN GEMM {w.M}x{w.N}x{w.K} on 1 GB300; % of dense tensor peak"


def code_of(src: str) -> str:
    """C++ source without its comments and with whitespace runs collapsed, so
    that editing a comment does not count as changing the kernel."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"' or c == "'":                       # string or character literal
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_sha() -> str:
    """Hash of the kernel sources' code: a traffic record taken on other code is stale."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(code_of(fh.read()).encode())
    return h.hexdigest()[:16]


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"bf16_burst": d.get("bf16_tflops"), "bf16_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d.get("hbm_gbs"), "src": "measured"}
    return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "src": "fallback"}


def measured_traffic(workload: str):
    """dram read+write bytes per launch, from the `traffic-record:` line of a
    committed ncu summary under profiles/, if it was taken on the current
    kernel source (else None)."""
    import glob
    import re
    pat = re.compile(r"^traffic-record: workload=(\S+) kernel_sha=(\S+) dram_bytes_per_launch=(\d+)")
    sha = kernel_sha()
    for path in sorted(glob.glob(os.path.join(PROFILES_DIR, "*.md"))):
        with open(path) as f:
            for line in f:
                m = pat.match(line.strip())
                if m and m.group(1) == workload and m.group(2) == sha:
                    return int(m.group(3))
    return None


# ---------------------------------------------------------------- ranks
def max_over_ranks(values, dist=None, device="cpu") -> list[float]:
    """Element-wise maximum of `values` over all ranks of the default process
    group (identity when `dist` is None, i.e. one process)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def replica_tflops(world: int, flop_per_step: float, steps: int, slowest_ms: float) -> float:
    """Whole-job throughput of `world` replicas that each ran `steps` steps of
    `flop_per_step`, the slowest taking `slowest_ms` milliseconds."""
    return world * flop_per_step * steps / (slowest_ms * 1e-3) / 1e12


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, pw = [], [], []
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        loaded = [s for s, p in zip(sm, pw) if p > 300.0] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw)}


# ---------------------------------------------------------------- CPU oracle timing
def oracle_sample(w: synth.Workload, A, B, sa, sb, target_s: float):
    """Times the oracle on a random sample of the workload's outputs (full K
    each); the sample grows until one run takes about `target_s` seconds.
    Returns (TFLOP/s, cores, description)."""
    import oracle
    rng = np.random.default_rng(12345)
    count = 256
    while True:
        mi = rng.integers(0, w.M, count)
        ni = rng.integers(0, w.N, count)
        t0 = time.perf_counter()
        if w.dtype == "e4m3":
            oracle.gemm_f8e4m3_tn_at(w.M, w.N, w.K, A, w.K, B, w.K, sa, sb, mi, ni)
        else:
            oracle.gemm_f16_tn_at(w.M, w.N, w.K, A, w.K, B, w.K, mi, ni)
        dt = time.perf_counter() - t0
        if dt >= target_s or count >= w.M * w.N:
            break
        count = int(min(w.M * w.N, count * max(2.0, 1.2 * target_s / max(dt, 1e-4))))
    tflops = 2.0 * count * w.K / dt / 1e12
    desc = f"{count} random outputs of {w.name} (full K={w.K} each), {dt:.1f} s"
    return tflops, oracle.num_threads(), desc


L2_BYTES = 129 * 10**6          # GB300's L2


def l2_note(sets: int, set_bytes: int) -> str:
    total = sets * set_bytes
    where = "larger than L2, no flush needed" if total > L2_BYTES else "they fit in L2"
    return f"{sets} rotating input set(s) of {set_bytes / 2**20:.2f} MiB, {total / 2**20:.0f} MiB in all: {where}"


def host_inputs(w: synth.Workload, sets: int):
    out = []
    for i in range(sets):
        A, B, sa, sb = synth.make_inputs(w, i)
        out.append((A, B, sa, sb))
    return out


# ---------------------------------------------------------------- reference arm
def run_reference(args, w: synth.Workload, rank: int) -> None:
    if rank != 0:
        return
    import oracle
    A, B, sa, sb = synth.make_inputs(w, 0)
    note = ""
    if w.op == "softmax_stats":
        # one step = the whole (small) problem, scores and statistics
        t_steps = []
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            oracle.gemm_f16_tn_softmax_stats(w.M, w.N, w.K, A, w.K, B, w.K, 1.0 / float(np.sqrt(w.K)))
            if i >= args.warmup:
                t_steps.append(time.perf_counter() - t0)
        dt = sum(t_steps) / len(t_steps)
        value = 2.0 * w.M * w.N * w.K / dt / 1e12
        print(json.dumps({
            "impl": "reference", "metric": metric_for(w), "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{w.name}: M={w.M} N={w.N} K={w.K}, the whole problem per step",
                       "M": w.M, "N": w.N, "K": w.K},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": "the whole problem per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return
    if w.values == "bf16":
        # the oracle's quantisation runs once, outside the timed steps
        A, sa = oracle.quantize_e4m3(A, "bf16", w.M, w.K)
        B, sb = oracle.quantize_e4m3(B, "bf16", w.N, w.K)
        note = "; operands quantised by the oracle once, untimed"
    cores = oracle.num_threads()
    # one step = a sample of outputs sized to about 0.5 s of host work
    rng = np.random.default_rng(7)
    count = 256
    while True:
        mi, ni = rng.integers(0, w.M, count), rng.integers(0, w.N, count)
        t0 = time.perf_counter()
        (oracle.gemm_f8e4m3_tn_at if w.dtype == "e4m3" else oracle.gemm_f16_tn_at)(
            *((w.M, w.N, w.K, A, w.K, B, w.K) + ((sa, sb) if w.dtype == "e4m3" else ()) + (mi, ni)))
        dt = time.perf_counter() - t0
        if dt > 0.5 or count >= w.M * w.N:
            break
        count *= 2
    fn = oracle.gemm_f8e4m3_tn_at if w.dtype == "e4m3" else oracle.gemm_f16_tn_at
    extra = (sa, sb) if w.dtype == "e4m3" else ()
    samples = [(rng.integers(0, w.M, count), rng.integers(0, w.N, count)) for _ in range(4)]
    for i in range(args.warmup):
        mi, ni = samples[i % 4]
        fn(*((w.M, w.N, w.K, A, w.K, B, w.K) + extra + (mi, ni)))
    t0 = time.perf_counter()
    for i in range(args.steps):
        mi, ni = samples[i % 4]
        fn(*((w.M, w.N, w.K, A, w.K, B, w.K) + extra + (mi, ni)))
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = 2.0 * count * w.K / dt / 1e12
    line = {
        "impl": "reference", "metric": metric_for(w), "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: M={w.M} N={w.N} K={w.K}, {count} sampled outputs per step",
                   "M": w.M, "N": w.N, "K": w.K},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{count} random outputs per step, full K{note}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm
def run_ours(args, w: synth.Workload, rank: int, world: int, local_rank: int) -> None:
    import torch

    import dense_gemm_tn_gb300 as g

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    sets = w.rotating if args.sets is None else max(1, args.sets)
    host = host_inputs(w, sets)
    is_f8 = w.dtype == "e4m3"
    pipeline = w.values == "bf16"          # bf16 operands quantised to E4M3 on the device every step
    esz = 2 if (pipeline or not is_f8) else 1   # bytes per input element
    dA, dB, scales = [], [], []
    for A, B, sa, sb in host:
        if esz == 1:
            dA.append(torch.from_numpy(A).to(dev))
            dB.append(torch.from_numpy(B).to(dev))
        else:
            dA.append(torch.from_numpy(A.view(np.int16)).to(dev))
            dB.append(torch.from_numpy(B.view(np.int16)).to(dev))
        scales.append((sa, sb))
    C = torch.empty((w.N, w.M), dtype=torch.bfloat16 if is_f8 else torch.float16, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = int(stream.cuda_stream)
    M, N, K = w.M, w.N, w.K
    if pipeline:
        qA = torch.empty((M, K), dtype=torch.uint8, device=dev)
        qB = torch.empty((N, K), dtype=torch.uint8, device=dev)
        dscale = torch.empty(2, dtype=torch.float32, device=dev)
        qa_p, qb_p, sa_p, sb_p = qA.data_ptr(), qB.data_ptr(), dscale.data_ptr(), dscale.data_ptr() + 4
    # our kernels per step: the GEMM; one repack of the operands when a row of K
    # elements is not a whole number of 16-byte units; two per quantisation
    launches_per_step = (5 if pipeline else 1) + (1 if (K * (1 if is_f8 and not pipeline else 2)) % 16 else 0)
    stats = w.op == "softmax_stats"
    if stats:
        sm_scale = 1.0 / float(np.sqrt(K))
        row_max = torch.empty(M, dtype=torch.float32, device=dev)
        row_sum = torch.empty(M, dtype=torch.float32, device=dev)
        rmax_p, rsum_p = row_max.data_ptr(), row_sum.data_ptr()

    # the C ABI's entry points, bound once
    f_quant, f_f8_dscale = g.lib.gemm_quantize_e4m3, g.lib.gemm_f8e4m3_tn_dscale
    f_f8, f_stats, f_f16 = g.lib.gemm_f8e4m3_tn, g.lib.gemm_f16_tn_softmax_stats, g.lib.gemm_f16_tn

    def issue(j, a, b, c, mid=None):
        """One step's work on the stream: returns the status codes of its calls."""
        if pipeline:
            r = [f_quant(a, g.GEMM_IN_BF16, M, K, K, qa_p, K, sa_p, sh),
                 f_quant(b, g.GEMM_IN_BF16, N, K, K, qb_p, K, sb_p, sh)]
            if mid is not None:
                mid.record(stream)
            r.append(f_f8_dscale(M, N, K, qa_p, K, qb_p, K, c, M, sa_p, sb_p, sh))
            return r
        if is_f8:
            return [f_f8(M, N, K, a, K, b, K, c, M, scales[j][0], scales[j][1], sh)]
        if stats:
            return [f_stats(M, N, K, a, K, b, K, c, M, sm_scale, rmax_p, rsum_p, sh)]
        return [f_f16(M, N, K, a, K, b, K, c, M, sh)]

    # device addresses looked up once: a torch call per operand and step would
    # add host time to every launch of a microsecond-scale problem
    ptr_a = [t.data_ptr() for t in dA]
    ptr_b = [t.data_ptr() for t in dB]
    ptr_c = C.data_ptr()

    def step(i, mid=None):
        j = i % sets
        return issue(j, ptr_a[j], ptr_b[j], ptr_c, mid)

    def one_call():
        """A callable of the input set j that issues that step's single GEMM call."""
        if is_f8:
            sa = [sc[0] for sc in scales]
            sb = [sc[1] for sc in scales]
            return lambda j: f_f8(M, N, K, ptr_a[j], K, ptr_b[j], K, ptr_c, M, sa[j], sb[j], sh)
        if stats:
            return lambda j: f_stats(M, N, K, ptr_a[j], K, ptr_b[j], K, ptr_c, M, sm_scale, rmax_p, rsum_p, sh)
        return lambda j: f_f16(M, N, K, ptr_a[j], K, ptr_b[j], K, ptr_c, M, sh)

    # validate once before timing (sampled against the oracle happens in the tests)
    rcs = step(0)
    if any(rc != 0 for rc in rcs):
        raise RuntimeError(f"GEMM call failed: {rcs}: {g.last_error()}")
    g.gemm_poll_device_status(sh)

    clocks = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    clocks.start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    # Only the pipeline records events inside the timed region (to time its
    # quantisations apart from its GEMMs): an event between two launches ends
    # the overlap of a kernel's setup with the previous kernel's tail, which
    # back-to-back calls of a small problem otherwise get.
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1 if pipeline else 2)]
    mid = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)] if pipeline else None
    ev[0].record(stream)
    if pipeline:
        for i in range(args.steps):
            step(i, mid[i])
            ev[i + 1].record(stream)
    else:
        # one C ABI call per step, its arguments bound beforehand: the loop's own
        # Python work per step stays well under a microsecond-scale GEMM's time
        call = one_call()
        failed = 0
        for i in range(args.steps):
            failed |= call(i % sets)
        ev[-1].record(stream)
        if failed:
            raise RuntimeError(f"a GEMM call in the timed loop failed: {g.last_error()}")
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    g.gemm_poll_device_status(sh)
    total_ms = ev[0].elapsed_time(ev[-1])
    if pipeline:
        # the GEMM is the dominant kernel; the two quantisations are timed beside it
        kernel_ms = statistics.mean(mid[i].elapsed_time(ev[i + 1]) for i in range(args.steps))
        quant_ms = statistics.mean(ev[i].elapsed_time(mid[i]) for i in range(args.steps))
    else:
        kernel_ms = total_ms / args.steps      # one GEMM per step (after a repack where one is needed)

    # ---- end to end: pinned host inputs -> device -> GEMM -> pinned host output.
    # Every step copies its own A and B in and its C out; the copies of the
    # neighbouring steps overlap the GEMM (three streams, two buffer slots).
    e2e_steps = max(4, min(args.steps, 50))
    hsets = min(sets, 2)
    hA = [torch.from_numpy(host[j][0].view(np.int16) if esz == 2 else host[j][0]).pin_memory()
          for j in range(hsets)]
    hB = [torch.from_numpy(host[j][1].view(np.int16) if esz == 2 else host[j][1]).pin_memory()
          for j in range(hsets)]
    hC = [torch.empty(C.shape, dtype=C.dtype, pin_memory=True) for _ in range(2)]
    eA = [torch.empty_like(dA[0]) for _ in range(2)]
    eB = [torch.empty_like(dB[0]) for _ in range(2)]
    eC = [torch.empty_like(C) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_done = [torch.cuda.Event() for _ in range(2)]
    gemm_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    for e in gemm_done + out_done:
        e.record(stream)

    def e2e_step(i):
        j, b = i % hsets, i % 2
        s_in.wait_event(gemm_done[b])            # slot b's inputs were read by step i-2
        with torch.cuda.stream(s_in):
            eA[b].copy_(hA[j], non_blocking=True)
            eB[b].copy_(hB[j], non_blocking=True)
        in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        stream.wait_event(out_done[b])           # slot b's C was read back by step i-2
        issue(j, eA[b].data_ptr(), eB[b].data_ptr(), eC[b].data_ptr())
        gemm_done[b].record(stream)
        s_out.wait_event(gemm_done[b])
        with torch.cuda.stream(s_out):
            hC[b].copy_(eC[b], non_blocking=True)
        out_done[b].record(s_out)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_event(out_done[(e2e_steps - 1) % 2])
    stream.wait_event(out_done[e2e_steps % 2])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    g.gemm_poll_device_status(sh)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    h2d = (M * K + N * K) * esz
    d2h = M * N * 2 + (8 * M if stats else 0)
    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], dist, dev)
    ms_per_step = total_ms / args.steps
    flop = 2.0 * M * N * K
    value = replica_tflops(world, flop, args.steps, total_ms)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    peaks = load_peaks()
    ratio = 2.0 if is_f8 else 1.0      # nominal fp8 / bf16 dense ratio (4.5 / 2.25 PF)
    peak = peaks["bf16_sustained"] * ratio
    achieved = flop / (kernel_ms * 1e-3) / 1e12
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        if pipeline:
            import oracle
            t0 = time.perf_counter()
            qa_ref, sa_ref = oracle.quantize_e4m3(host[0][0], "bf16", M, K)
            qb_ref, sb_ref = oracle.quantize_e4m3(host[0][1], "bf16", N, K)
            t_q = time.perf_counter() - t0
            tf, cores, desc = oracle_sample(w, qa_ref, qb_ref, sa_ref, sb_ref, target_s=args.cpu_seconds)
            desc += f"; the oracle's quantisation of both operands took a further {t_q:.1f} s"
        elif stats:
            import oracle
            t0 = time.perf_counter()
            oracle.gemm_f16_tn_softmax_stats(M, N, K, host[0][0], K, host[0][1], K, 1.0 / float(np.sqrt(K)))
            dt = time.perf_counter() - t0
            tf, cores = 2.0 * M * N * K / dt / 1e12, oracle.num_threads()
            desc = f"the whole {w.name} problem (scores and statistics), {dt:.2f} s"
        else:
            tf, cores, desc = oracle_sample(w, *host[0], target_s=args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}
    # The dominant kernel's roofline: below the ridge point (peak FLOP/s over HBM
    # bytes/s) the bound is HBM, and the achieved figure is the algorithmic bytes
    # (operands read once, C and the row statistics written once) per launch
    # over the launch's time; above it, FLOP/s against the tensor peak.
    alg_bytes = (M * K + N * K) * (1 if is_f8 or pipeline else 2) + 2 * M * N + (8 * M if stats else 0)
    ridge = peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    intensity = flop / alg_bytes
    roofline = {"intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
                "kernel": KERNEL_NAME[w.dtype], "kernel_ms": kernel_ms, "traffic": measured_traffic(w.name),
                "algorithmic_bytes": alg_bytes}
    if intensity < ridge:
        gbs = alg_bytes / (kernel_ms * 1e-3) / 1e9
        roofline.update({"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "peak_src": f"{peaks['src']} copy bandwidth",
                         "tensor_frac": achieved / peak})
    else:
        roofline.update({"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak,
                         "peak_src": f"{peaks['src']} bf16 sustained" + (" x2 (nominal fp8/bf16)" if is_f8 else
                                                                          " (fp16 = bf16 rate)")})
    line = {
        "metric": metric_for(w), "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.dtype} TN GEMM M={M} N={N} K={K}, {w.values} inputs, "
                               f"{sets} rotating input set(s)"
                               + (", both operands quantised to e4m3 on the device each step" if pipeline else ""),
                   "M": M, "N": N, "K": K, "accumulate": "f32",
                   "l2": l2_note(sets, (M + N) * K * esz),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_of_dense_peak": 100.0 * value / world / NOMINAL_PEAK[w.dtype],
        "e2e": {"value": replica_tflops(world, flop, 1, e2e_ms), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "overlap": "the copies of steps i-1 and i+1 run beside the GEMM of step i "
                           "(copy-in, GEMM and copy-out streams, two buffer slots)"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "clocks": clk,
        "gpu_launches": args.steps * launches_per_step,
    }
    if pipeline:
        # algorithmic bytes: each bf16 input read once, each e4m3 code and scale written once
        qbytes = 2 * (M * K + N * K) + (M * K + N * K) + 8
        line["quantize"] = {"bound": "hbm", "achieved": qbytes / (quant_ms * 1e-3) / 1e9,
                            "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": qbytes / (quant_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                            "ms": quant_ms, "algorithmic_bytes": qbytes,
                            "kernels": "quant_amax_kernel + quant_store_kernel, one pair per operand"}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="sq_8192", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--sets", type=int, default=None,
                    help="input sets to rotate (default: the workload's; 1 for small profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w, rank)
    else:
        run_ours(args, w, rank, world, local_rank)


if __name__ == "__main__":
    main()
