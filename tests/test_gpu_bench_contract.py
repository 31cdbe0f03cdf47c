"""bench.py's one-line JSON contract, on a small workload: every key the
driver reads is present, typed, and consistent with the others."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


def run_bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", ["qk_1024", "qk_stats_1024", "pm1_512"])
def test_json_line(workload):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    d = run_bench("--workload", workload, "--steps", "20", "--warmup", "3", "--cpu-seconds", "0.5")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "e2e", "roofline", "cpu_baseline",
                "clocks", "gpu_launches"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["gpu_launches"] == 20
    assert "workload" in d["config"]
    rf = d["roofline"]
    # these small shapes lie below the ridge point: HBM-bound by the roofline
    assert rf["intensity_flop_per_byte"] < rf["ridge_flop_per_byte"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"])
    assert rf["achieved"] == pytest.approx(rf["algorithmic_bytes"] / (rf["kernel_ms"] * 1e-3) / 1e9)
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] > 0 and cpu["cores"] >= 1 and cpu["sample"]


def test_headline_line_carries_fp8_sustained_and_clocks():
    """The default workload's line: a burst peak for a timed region of a few
    milliseconds, clocks sampled inside it, the FP8 8192^3 secondary with its
    own roofline, clocks and CPU baseline, and a sustained sub-measurement
    against the sustained peak."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    d = run_bench("--steps", "20", "--warmup", "3", "--cpu-seconds", "1", "--sustained-s", "1.5")
    assert d["config"]["workload"].startswith("sq_8192") and d["gpu_launches"] == 20
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["peak_kind"] == "burst"
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"])
    assert rf["frac_burst"] == pytest.approx(rf["frac"]) and rf["frac_sustained"] > rf["frac_burst"]
    clk = d["clocks"]
    assert clk["samples"] >= 1 and clk["sm_mhz"] > 0
    assert rf["cycles_per_launch"] > rf["tensor_cycles_per_launch"] * 0.9
    sec = d["secondary"]
    assert sec["config"]["workload"].startswith("e4m3_8192") and sec["dtype"] == "e4m3"
    assert sec["value"] > 0 and sec["roofline"]["bound"] == "tensor"
    assert sec["roofline"]["peak"] == pytest.approx(2 * rf["peak"])
    assert sec["cpu_baseline"]["kind"] == "oracle" and sec["clocks"]["samples"] >= 1
    sus = d["sustained"]
    assert sus["seconds"] >= 1.4 and sus["peak_kind"] == "sustained"
    assert sus["clocks"]["samples"] >= 100


def test_reference_arm_line():
    d = run_bench("--impl", "reference", "--workload", "qk_1024", "--steps", "1", "--warmup", "3")
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
