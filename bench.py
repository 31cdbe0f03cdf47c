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
import math
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
SKINNY_KERNEL_NAME = {"f16": "tn_skinny_kernel<KindF16>", "e4m3": "tn_skinny_kernel<KindE4M3>"}
KERNEL_SOURCES = ["dense_gemm_tn_gb300/csrc/tn_gemm_kernel.cuh", "dense_gemm_tn_gb300/csrc/sm103_ptx.cuh",
                  "dense_gemm_tn_gb300/csrc/skinny_kernel.cuh"]
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


class NvmlSampler:
    """SM clock, board power and clock-event reasons of one GPU, read with
    NVML's read-only queries from a thread about once a millisecond and
    stamped with the host clock, so that the samples taken inside a timed
    region can be picked out (the 200 ms nvidia-smi loop misses a region of a
    few milliseconds).  NVML is the driver's library (libnvidia-ml.so.1),
    loaded with ctypes; nothing is set."""
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    NVML_CLOCK_SM = 1

    def __init__(self, torch_device, period_s: float = 0.001):
        import ctypes
        self.ct = ctypes
        self.period = period_s
        self.samples: list[tuple[float, float, float, int]] = []   # (host time, SM MHz, W, reason bits)
        self.max_mhz = None
        self.handle = None
        self._stop = threading.Event()
        self.thread = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
        except OSError:
            return
        self.lib = lib
        h = ctypes.c_void_p()
        found = False
        try:
            import torch
            props = torch.cuda.get_device_properties(torch_device)
            uuid = str(getattr(props, "uuid", "") or "")
            if uuid:
                key = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
                found = lib.nvmlDeviceGetHandleByUUID(key.encode(), ctypes.byref(h)) == 0
            if not found and hasattr(props, "pci_bus_id"):
                bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
                found = lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
        except Exception:
            found = False
        if not found:
            return
        self.handle = h
        v = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(v)) == 0:
            self.max_mhz = float(v.value)
        self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)

    @property
    def ok(self) -> bool:
        return self.handle is not None

    def _query(self):
        ct, lib, h = self.ct, self.lib, self.handle
        clk, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if lib.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, ct.byref(clk)) != 0:
            return None
        power = float(pw.value) / 1000.0 if lib.nvmlDeviceGetPowerUsage(h, ct.byref(pw)) == 0 else float("nan")
        bits = int(rs.value) if self._reasons_fn and self._reasons_fn(h, ct.byref(rs)) == 0 else 0
        return float(clk.value), power, bits

    def _run(self):
        while not self._stop.is_set():
            t = time.perf_counter()
            q = self._query()
            if q is not None:
                self.samples.append((t, *q))
            time.sleep(self.period)

    def start(self):
        if self.ok and self.thread is None:
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()

    def stop(self):
        if self.thread is not None:
            self._stop.set()
            self.thread.join(timeout=2)
            self.thread = None

    def window(self, t0: float, t1: float) -> dict | None:
        """Clock record of the samples taken between host times t0 and t1."""
        inside = [s for s in list(self.samples) if t0 <= s[0] <= t1]
        if not inside:
            return None
        sm = [s[1] for s in inside]
        pw = [s[2] for s in inside if s[2] == s[2]]
        reasons = sorted({name for s in inside for bit, name in self.REASON_BITS.items() if s[3] & bit})
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": self.max_mhz or max(sm),
                "reasons": reasons, "samples": len(inside), "power_w_max": max(pw) if pw else None,
                "source": "NVML read-only queries every ~1 ms inside the timed region"}


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
BURST_REGION_MS = 1000.0     # a timed region shorter than this runs before the power cap settles
PROBE_MIN_MS = 0.05          # launches at least this long measure their own SM clock


class KernelClock:
    """The SM clock the timed launches ran at, measured by the GEMM kernel
    itself: with the library's clock probe set, the first thread of each
    launch's first CTA adds its SM cycles (%clock64) and nanoseconds
    (%globaltimer) from start to end to a device counter (three atomic adds
    per launch).  NVML's readings lag load changes of a few milliseconds; a
    kernel spinning beside the GEMM to time the clock slowed the GEMM down."""

    def __init__(self, torch, dev, g):
        self.g = g
        self.buf = torch.zeros(3, dtype=torch.int64, device=dev)

    def start(self):
        self.buf.zero_()
        self.g.lib.gemm_debug_set_clock_probe(self.buf.data_ptr())

    def stop(self):
        self.g.lib.gemm_debug_set_clock_probe(None)

    def mhz(self) -> float | None:
        cycles, ns, launches = (int(x) for x in self.buf.tolist())
        return (cycles / ns * 1e3, launches) if ns > 0 else None


def timed_loop(torch, dev, stream, call, sets: int, steps: int, warmup: int, sampler, dist=None, probe=None):
    """W untimed calls, then exactly `steps` calls bracketed by a barrier and a
    device synchronisation on both sides, timed with CUDA events on the
    launching stream.  Events are recorded only before and after the loop: an
    event between two launches would end the overlap of a kernel's setup
    with the previous kernel's tail, which back-to-back calls otherwise get.
    With `probe` (KernelClock), the timed launches measure their own SM clock
    when a launch lasts at least PROBE_MIN_MS (judged from the warm-up): its
    atomic adds at the end of a launch of a few microseconds would delay the
    next dependent launch.
    Returns (device ms, clock record of the timed region, any call failed)."""
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for i in range(warmup):
        call(i % sets)
    w1.record(stream)
    torch.cuda.synchronize(dev)
    if probe is not None and warmup > 0 and w0.elapsed_time(w1) / warmup < PROBE_MIN_MS:
        probe = None
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if probe is not None:
        probe.start()
    t0 = time.perf_counter()
    e0.record(stream)
    failed = 0
    for i in range(steps):
        failed |= call(i % sets)
    e1.record(stream)
    if probe is not None:
        probe.stop()
    torch.cuda.synchronize(dev)
    t1 = time.perf_counter()
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clk = sampler.window(t0, t1)
    measured = probe.mhz() if probe is not None else None
    if measured is not None:
        clk = dict(clk or {})
        clk["sm_mhz_nvml"] = clk.get("sm_mhz")
        clk["sm_mhz"] = measured[0]
        clk["sm_mhz_source"] = (f"measured by the timed GEMM launches themselves ({measured[1]} launches: SM cycles "
                                "over globaltimer ns of each launch's first CTA)")
    return e0.elapsed_time(e1), clk, failed


def roofline_of(w: synth.Workload, kernel_ms: float, region_ms: float, peaks: dict, clk: dict | None,
                sms: int, stats: bool, skinny: bool = False) -> dict:
    """The dominant kernel's roofline.  Below the ridge point (tensor peak over
    HBM bytes/s) the bound is HBM and `achieved` is the algorithmic bytes per
    launch (operands read once, C and any row statistics written once) over
    the launch's time; above it, 2MNK per launch over that time against the
    tensor peak.  The tensor peak is the measured cuBLAS bf16 rate (x2 for
    E4M3, the nominal fp8 / bf16 ratio): its burst figure for a timed region
    under a second (the GPU has not reached its power cap yet), its sustained
    figure for a longer one; both fractions are given."""
    M, N, K = w.M, w.N, w.K
    is_f8 = w.dtype == "e4m3" or w.values == "bf16"
    flop = 2.0 * M * N * K
    ratio = 2.0 if is_f8 else 1.0
    burst, sustained = peaks["bf16_burst"] * ratio, peaks["bf16_sustained"] * ratio
    kind = "burst" if region_ms < BURST_REGION_MS else "sustained"
    peak = burst if kind == "burst" else sustained
    achieved = flop / (kernel_ms * 1e-3) / 1e12
    alg_bytes = (M * K + N * K) * (1 if is_f8 else 2) + 2 * M * N + (8 * M if stats else 0)
    ridge = peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    intensity = flop / alg_bytes
    rf = {"intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
          "kernel": (SKINNY_KERNEL_NAME if skinny else KERNEL_NAME)["e4m3" if is_f8 else "f16"], "kernel_ms": kernel_ms,
          "traffic": measured_traffic(w.name), "algorithmic_bytes": alg_bytes}
    dtype_note = " x2 (nominal fp8/bf16)" if is_f8 else " (fp16 = bf16 rate)"
    if intensity < ridge:
        gbs = alg_bytes / (kernel_ms * 1e-3) / 1e9
        rf.update({"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                   "frac": gbs / peaks["hbm_gbs"], "peak_src": f"{peaks['src']} copy bandwidth",
                   "tensor_frac": achieved / peak})
    else:
        rf.update({"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                   "frac": achieved / peak, "peak_kind": kind,
                   "peak_src": f"{peaks['src']} bf16 {kind}{dtype_note}; {kind} because the timed region "
                               f"lasted {region_ms:.0f} ms ({'<' if kind == 'burst' else '>='} "
                               f"{BURST_REGION_MS:.0f} ms)",
                   "frac_burst": achieved / burst, "frac_sustained": achieved / sustained,
                   "peak_burst": burst, "peak_sustained": sustained})
    # per-clock view: cycles of the launch at the sampled SM clock against the
    # cycles its MMAs take at the tensor peak (8192 dense FP16 FLOP per clock
    # per SM, twice that for E4M3)
    mma_cycles = flop / ((16384.0 if is_f8 else 8192.0) * sms)
    rf["tensor_cycles_per_launch"] = mma_cycles
    if clk and clk.get("sm_mhz"):
        cyc = kernel_ms * 1e-3 * clk["sm_mhz"] * 1e6
        rf["cycles_per_launch"] = cyc
        rf["tensor_frac_per_clock"] = mma_cycles / cyc
        rf["sm_mhz_in_region"] = clk["sm_mhz"]
    return rf


def clocks_record(nvml_clk: dict | None, smi: dict | None) -> dict | None:
    """The timed region's clocks: the NVML samples taken inside it; without
    NVML, the nvidia-smi loop (which may have no sample inside a short region)."""
    if nvml_clk:
        out = dict(nvml_clk)
        if smi:
            out["nvidia_smi"] = smi
        return out
    return smi


def cpu_line(w: synth.Workload, host0, seconds: float, stats: bool) -> dict:
    if w.values == "bf16":
        import oracle
        t0 = time.perf_counter()
        qa_ref, sa_ref = oracle.quantize_e4m3(host0[0], "bf16", w.M, w.K)
        qb_ref, sb_ref = oracle.quantize_e4m3(host0[1], "bf16", w.N, w.K)
        t_q = time.perf_counter() - t0
        tf, cores, desc = oracle_sample(w, qa_ref, qb_ref, sa_ref, sb_ref, target_s=seconds)
        desc += f"; the oracle's quantisation of both operands took a further {t_q:.1f} s"
    elif stats:
        import oracle
        t0 = time.perf_counter()
        oracle.gemm_f16_tn_softmax_stats(w.M, w.N, w.K, host0[0], w.K, host0[1], w.K, 1.0 / float(np.sqrt(w.K)))
        dt = time.perf_counter() - t0
        tf, cores = 2.0 * w.M * w.N * w.K / dt / 1e12, oracle.num_threads()
        desc = f"the whole {w.name} problem (scores and statistics), {dt:.2f} s"
    else:
        tf, cores, desc = oracle_sample(w, *host0, target_s=seconds)
    return {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}


def device_operands(torch, dev, host, esz: int):
    dA, dB = [], []
    for A, B, _, _ in host:
        if esz == 1:
            dA.append(torch.from_numpy(A).to(dev))
            dB.append(torch.from_numpy(B).to(dev))
        else:
            dA.append(torch.from_numpy(A.view(np.int16)).to(dev))
            dB.append(torch.from_numpy(B.view(np.int16)).to(dev))
    return dA, dB


def run_secondary(args, torch, g, dev, stream, sampler, peaks, sms) -> dict:
    """The FP8 headline shape (e4m3_8192: E4M3 operands with per-tensor
    scales, bf16 C, 4 rotating sets) with the same steps and warm-up as the
    main line, and its own clocks, roofline and CPU baseline."""
    w = synth.WORKLOADS["e4m3_8192"]
    sets = w.rotating
    host = host_inputs(w, sets)
    dA, dB = device_operands(torch, dev, host, 1)
    C = torch.empty((w.N, w.M), dtype=torch.bfloat16, device=dev)
    sh = int(stream.cuda_stream)
    M, N, K = w.M, w.N, w.K
    pa, pb, pc = [t.data_ptr() for t in dA], [t.data_ptr() for t in dB], C.data_ptr()
    sa, sb = [h[2] for h in host], [h[3] for h in host]
    f_f8 = g.calls.gemm_f8e4m3_tn

    def call(j):
        return f_f8(M, N, K, pa[j], K, pb[j], K, pc, M, sa[j], sb[j], sh)

    if call(0) != 0:
        raise RuntimeError(f"FP8 GEMM call failed: {g.last_error()}")
    g.gemm_poll_device_status(sh)
    total_ms, clk, failed = timed_loop(torch, dev, stream, call, sets, args.steps, args.warmup, sampler,
                                       probe=KernelClock(torch, dev, g))
    if failed:
        raise RuntimeError(f"an FP8 GEMM call in the timed loop failed: {g.last_error()}")
    g.gemm_poll_device_status(sh)
    kernel_ms = total_ms / args.steps
    value = 2.0 * M * N * K / (kernel_ms * 1e-3) / 1e12
    out = {"metric": metric_for(w), "value": value, "unit": "TFLOP/s", "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": kernel_ms, "dtype": "e4m3",
           "config": {"workload": f"{w.name}: e4m3 TN GEMM M={M} N={N} K={K}, per-tensor scales, bf16 C, "
                                  f"{sets} rotating input sets",
                      "l2": l2_note(sets, (M + N) * K)},
           "pct_of_dense_peak": 100.0 * value / NOMINAL_PEAK["e4m3"],
           "roofline": roofline_of(w, kernel_ms, total_ms, peaks, clk, sms, False, "skinny=1" in g.last_launch()),
           "clocks": clk, "gpu_launches": args.steps}
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_line(w, host[0], args.cpu_seconds / 2, False)
    del dA, dB, C
    torch.cuda.empty_cache()
    return out


def run_ours(args, w: synth.Workload, rank: int, world: int, local_rank: int) -> None:
    import torch

    import dense_gemm_tn_gb300 as g

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    sets = w.rotating if args.sets is None else max(1, args.sets)
    host = host_inputs(w, sets)
    is_f8 = w.dtype == "e4m3"
    pipeline = w.values == "bf16"          # bf16 operands quantised to E4M3 on the device every step
    esz = 2 if (pipeline or not is_f8) else 1   # bytes per input element
    dA, dB = device_operands(torch, dev, host, esz)
    scales = [(h[2], h[3]) for h in host]
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

    # the C ABI's entry points, bound once (through the CPython-API binding where
    # it was built: a ctypes call costs about 1.5 us of host time per step)
    f_quant, f_f8_dscale = g.calls.gemm_quantize_e4m3, g.calls.gemm_f8e4m3_tn_dscale
    f_f8, f_stats, f_f16 = g.calls.gemm_f8e4m3_tn, g.calls.gemm_f16_tn_softmax_stats, g.calls.gemm_f16_tn

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

    smi = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    smi.start()
    sampler = NvmlSampler(dev)
    sampler.start()
    if pipeline:
        # The pipeline also records one event between its quantisations and its
        # GEMM per step, to time them apart.
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        mid = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        t0 = time.perf_counter()
        ev[0].record(stream)
        for i in range(args.steps):
            step(i, mid[i])
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        t1 = time.perf_counter()
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        nvml_clk = sampler.window(t0, t1)
        total_ms = ev[0].elapsed_time(ev[-1])
        # the GEMM is the dominant kernel; the two quantisations are timed beside it
        kernel_ms = statistics.mean(mid[i].elapsed_time(ev[i + 1]) for i in range(args.steps))
        quant_ms = statistics.mean(ev[i].elapsed_time(mid[i]) for i in range(args.steps))
    else:
        # one C ABI call per step, its arguments bound beforehand: the loop's own
        # Python work per step stays well under a microsecond-scale GEMM's time
        total_ms, nvml_clk, failed = timed_loop(torch, dev, stream, one_call(), sets, args.steps, args.warmup,
                                                sampler, dist, probe=KernelClock(torch, dev, g))
        if failed:
            raise RuntimeError(f"a GEMM call in the timed loop failed: {g.last_error()}")
        kernel_ms = total_ms / args.steps      # one GEMM per step (after a repack where one is needed)
    smi_clk = smi.stop()
    clk = clocks_record(nvml_clk, smi_clk)
    g.gemm_poll_device_status(sh)

    peaks = load_peaks()
    flop = 2.0 * M * N * K
    # (which GEMM kernel the library ran: the last launch's record says)
    skinny = "skinny=1" in g.last_launch()
    roofline = roofline_of(w, kernel_ms, total_ms, peaks, clk, sms, stats, skinny)

    # ---- sustained: the same calls back to back for about `sustained_s`
    # seconds, long enough for the GPU to settle at its power cap
    sustained = None
    if args.sustained_s > 0 and roofline["bound"] == "tensor" and not pipeline:
        s_steps = max(args.steps, int(math.ceil(args.sustained_s * 1e3 / max(kernel_ms, 1e-3))))
        s_ms, s_clk, failed = timed_loop(torch, dev, stream, one_call(), sets, s_steps, 0, sampler, dist,
                                         probe=KernelClock(torch, dev, g))
        if failed:
            raise RuntimeError(f"a GEMM call in the sustained loop failed: {g.last_error()}")
        g.gemm_poll_device_status(sh)
        s_ms = max_over_ranks([s_ms], dist, dev)[0]
        s_kernel = s_ms / s_steps
        s_rf = roofline_of(w, s_kernel, s_ms, peaks, s_clk, sms, stats, skinny)
        sustained = {"steps": s_steps, "seconds": s_ms * 1e-3, "ms_per_step": s_kernel,
                     "value": replica_tflops(world, flop, s_steps, s_ms), "unit": "TFLOP/s",
                     "frac": s_rf["frac"], "peak": s_rf["peak"], "peak_kind": s_rf["peak_kind"],
                     "cycles_per_launch": s_rf.get("cycles_per_launch"),
                     "tensor_frac_per_clock": s_rf.get("tensor_frac_per_clock"), "clocks": s_clk}

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
    del hA, hB, hC, eA, eB, eC
    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], dist, dev)
    ms_per_step = total_ms / args.steps
    value = replica_tflops(world, flop, args.steps, total_ms)

    # ---- the FP8 headline shape beside the FP16 one (one GPU only)
    secondary = None
    if world == 1 and w.name == "sq_8192" and not args.no_secondary:
        secondary = run_secondary(args, torch, g, dev, stream, sampler, peaks, sms)
    sampler.stop()

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_line(w, host[0], args.cpu_seconds, stats)
    line = {
        "metric": metric_for(w), "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.dtype} TN GEMM M={M} N={N} K={K}, {w.values} inputs, "
                               f"{sets} rotating input set(s)"
                               + (", both operands quantised to e4m3 on the device each step" if pipeline else ""),
                   "M": M, "N": N, "K": K, "accumulate": "f32",
                   "l2": l2_note(sets, (M + N) * K * esz),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "binding": "cpython" if g.fast is not None else "ctypes"},
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
    if sustained is not None:
        line["sustained"] = sustained
    if secondary is not None:
        line["secondary"] = secondary
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
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the FP8 8192^3 measurement that follows the default FP16 one")
    ap.add_argument("--sustained-s", type=float, default=2.0,
                    help="seconds of back-to-back calls for the sustained figure (0: skip)")
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
