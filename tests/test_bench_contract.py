"""bench.py's JSON line: the keys and types every run must print.

The reference arm (the float64 oracle on the host cores) runs here on the CPU;
the GPU arm is run on a small step count under the gpu marker."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"}


def run_bench(*args, timeout=900):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_arm_line():
    line = run_bench("--impl", "reference", "--workload", "bs4_kv1024", "--steps", "2",
                     "--warmup", "1", "--ref-budget", "2")
    assert BASE_KEYS <= set(line)
    assert line["impl"] == "reference" and line["unit"] == "us/call"
    assert line["higher_is_better"] is False and line["value"] > 0
    assert line["config"]["workload"] == "bs4_kv1024"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"]
    assert cb["cores"] == len(os.sched_getaffinity(0))  # every host core this process may use
    assert line["e2e"] == {"value": line["value"], "unit": "us/call", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


@pytest.mark.gpu
@pytest.mark.parametrize("workload,cache,kernels", [
    ("bs64_kv8192", "e4m3", 2), ("bs64_kv8192", "mxfp4", 2),
    ("bs4_kv1024", "e4m3", 1),    # the cluster split: stage 1 alone
    ("bs4_kv1024", "mxfp4", 2)])  # an MXFP4 cache runs the persistent split
def test_gpu_arm_line(workload, cache, kernels):
    line = run_bench("--workload", workload, "--steps", "20", "--warmup", "3",
                     "--no-per-config", "--no-cpu-baseline", "--e2e-steps", "2", "--cache", cache)
    assert BASE_KEYS <= set(line) and line["n_gpus"] == 1 and line["steps"] == 20
    assert line["config"]["workload"] == workload
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and 0 < rf["frac"] < 1.2
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    e2e = line["e2e"]
    assert e2e["value"] > line["value"] and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert line["gpu_launches"] == kernels * 20
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(line["clocks"])


def test_cpu_baseline_leg_uses_every_host_core():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-sample",
                        "bs4_kv1024", "--budget", "1"], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    cb = json.loads(r.stdout.strip().splitlines()[-1])
    assert cb["kind"] == "oracle" and cb["cores"] == len(os.sched_getaffinity(0))
    assert cb["value"] > 0 and cb["single_core_value"] > 0
