"""Benchmark of the MLA forward_absorb decode step on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one decode call (split-attention stage 1 + combine stage 2) over the
whole batch of the headline workload, bs=256 rows x kv_len=8192 cached tokens
of an FP8 e4m3 latent cache (1.21 GB, larger than L2, so consecutive steps
stream it from HBM).  ``value`` is device time per call with the inputs resident
in HBM; ``e2e`` is the same call through the Python binding with the step's
inputs copied from pinned host memory and the output read back inside the
timed region.  ``--impl reference`` times the float64 CPU oracle instead, on a
bounded sample of rows per step.

Under torchrun each rank runs its own replica of the workload (the decode of
independent batches shards with no exchange); rank 0 prints the line.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mla_decode_attention_08_gb300.inputs import HEADLINE, WORKLOADS, make_inputs  # noqa: E402

METRIC = "µs/call and effective HBM TB/s (fraction of GB300 peak) per (bs, kv_len)"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def algorithmic_bytes(inp) -> int:
    """Bytes one call must move: every cached token's 576-byte row (+4 for its
    page-table entry), the bf16 query and output rows, and both indptr arrays."""
    tokens = int(inp.kv_indptr[-1])
    per_token = 576 + (4 if inp.kv_indices is not None else 0)
    return tokens * per_token + inp.batch * 16 * (576 + 512) * 2 + 2 * (inp.batch + 1) * 4


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        inside = [p for t, p in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        use = inside or [p for _, p in self.samples]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in use for n, v in zip(names, p[5:9]) if v.strip() == "Active"})
        sm = [num(p[1]) for p in use if num(p[1]) is not None]
        mx = [num(p[2]) for p in use if num(p[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": len(inside)}


def source_hash() -> str:
    """Hash of the stage-1 kernel source (ties recorded ncu traffic to a kernel version)."""
    h = hashlib.sha256()
    for f in ("stage1.cu", "ptx.cuh", "kernels.h", "schedule.h"):
        with open(os.path.join(ROOT, "mla_decode_attention_08_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """Per-launch DRAM bytes of stage 1 from the committed ncu summary, if it
    was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"stage1_{workload}_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_hash") != source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- device arm
class DeviceWorkload:
    """One workload resident on the GPU: query, quantised cache, indptr, output, workspace."""

    def __init__(self, name: str, torch, binding, sms: int):
        self.name = name
        self.inp = inp = make_inputs(name)
        dev = "cuda"

        def bf16(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

        self.q = bf16(inp.q_bits)
        kv = bf16(inp.kv_bits)
        self.kv = torch.empty((kv.shape[0], 576), dtype=torch.uint8, device=dev)
        self.kv_scale = torch.empty(1, dtype=torch.float32, device=dev)
        binding.mla_fp8_quantize_per_tensor(kv, self.kv, self.kv_scale,
                                            torch.empty(16, dtype=torch.uint8, device=dev))
        del kv
        self.qo_indptr = torch.from_numpy(inp.qo_indptr).to(dev)
        self.kv_indptr = torch.from_numpy(inp.kv_indptr).to(dev)
        self.kv_indices = None if inp.kv_indices is None else torch.from_numpy(inp.kv_indices).to(dev)
        self.out = torch.empty((inp.batch, 16, 512), dtype=torch.bfloat16, device=dev)
        self.plan = binding.mla_decode_plan(inp.batch, inp.max_kv_len, sms)
        self.ws = binding.new_workspace(self.plan)
        self.bytes = algorithmic_bytes(inp)
        self.binding = binding
        torch.cuda.synchronize()
        self.inp.kv_bits = None  # release the host copy of the cache source

    def call(self, stream=None):
        self.binding.mla_decode_fwd(self.q, self.kv, self.kv_scale, self.qo_indptr, self.kv_indptr,
                                    self.out, stream, plan=self.plan, workspace=self.ws,
                                    kv_indices=self.kv_indices)

    def stage1(self, stream=None):
        self.binding.mla_decode_stage1(self.q, self.kv, self.kv_scale, self.qo_indptr,
                                       self.kv_indptr, self.out, stream, plan=self.plan,
                                       workspace=self.ws, kv_indices=self.kv_indices)


def time_loop(torch, fn, steps: int, stream) -> float:
    """Milliseconds for `steps` back-to-back calls, CUDA events on `stream`."""
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn(stream)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def per_call_cold(torch, w: DeviceWorkload, reps: int, stream, flush) -> list:
    """Per-call device times (µs) with L2 flushed before each call."""
    times = []
    for _ in range(reps):
        flush.add_(1)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        w.call(stream)
        e.record(stream)
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e) * 1e3)
    return times


def e2e_timing(torch, w: DeviceWorkload, steps: int, stream) -> dict:
    """Host-buffer round trip per call: pinned H2D of the step's inputs, the
    decode call, D2H of the output, all inside the timed region."""
    host = {k: getattr(w, k).cpu().pin_memory() for k in ("q", "kv", "kv_scale", "qo_indptr", "kv_indptr")}
    if w.kv_indices is not None:
        host["kv_indices"] = w.kv_indices.cpu().pin_memory()
    out_host = torch.empty(w.out.shape, dtype=w.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()
    dev = {k: torch.empty_like(v, device="cuda") for k, v in host.items()}

    def step():
        for k, v in host.items():
            dev[k].copy_(v, non_blocking=True)
        w.binding.mla_decode_fwd(dev["q"], dev["kv"], dev["kv_scale"], dev["qo_indptr"],
                                 dev["kv_indptr"], w.out, stream, plan=w.plan, workspace=w.ws,
                                 kv_indices=dev.get("kv_indices"))
        out_host.copy_(w.out, non_blocking=True)

    with torch.cuda.stream(stream):
        step()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
    us = start.elapsed_time(end) * 1e3 / steps
    return {"value": round(us, 2), "unit": "us/call", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps}
