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

import os as _os
import sys as _sys

# The CPU oracle legs run one batch row per host thread, on every core this
# process may use; BLAS stays single-threaded inside each so that the reported
# core count is exactly the threads used.  BLAS reads these before numpy is
# first imported.
if "--impl=reference" in _sys.argv or "--oracle-sample" in _sys.argv or \
        any(a == "reference" and _sys.argv[i - 1] == "--impl" for i, a in enumerate(_sys.argv)):
    for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        _os.environ[_v] = "1"

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


CACHE_ROW_BYTES = {"e4m3": 576, "bf16": 1152, "mxfp4": 288 + 18}


def algorithmic_bytes(inp, cache: str = "e4m3") -> int:
    """Bytes one call must move: every cached token's row (576 bytes of e4m3
    codes, 1152 of bf16, or 288 of E2M1 elements plus 18 scale bytes; +4 for its
    page-table entry), the bf16 query and output rows, and both indptr arrays."""
    tokens = int(inp.kv_indptr[-1])
    per_token = CACHE_ROW_BYTES[cache] + (4 if inp.kv_indices is not None else 0)
    queries = inp.batch * getattr(inp, "qo_len", 1)
    return tokens * per_token + queries * 16 * (576 + 512) * 2 + 2 * (inp.batch + 1) * 4


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


def recorded_traffic(workload: str, cache: str = "e4m3"):
    """Per-launch DRAM bytes of stage 1 from the committed ncu summary, if it
    was taken on the current kernel source; else None."""
    tag = "" if cache == "e4m3" else f"{cache}_"
    path = os.path.join(ROOT, "profiles", f"stage1_{tag}{workload}_traffic.json")
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
        self.kv_bf16 = kv  # the bf16 cache the e4m3 codes came from (the bf16-cache step's input)
        # The MXFP4 cache of the same source (mla_decode_fwd_mxfp4: contiguous rows,
        # one query token).
        self.mx = inp.kv_indices is None and inp.qo_len == 1
        if self.mx:
            self.kv_fp4 = torch.empty((kv.shape[0], 288), dtype=torch.uint8, device=dev)
            self.kv_mxs = torch.empty((kv.shape[0], 18), dtype=torch.uint8, device=dev)
            binding.mla_mxfp4_quantize(kv, self.kv_fp4, self.kv_mxs)
        self.qo_indptr = torch.from_numpy(inp.qo_indptr).to(dev)
        self.kv_indptr = torch.from_numpy(inp.kv_indptr).to(dev)
        self.kv_indices = None if inp.kv_indices is None else torch.from_numpy(inp.kv_indices).to(dev)
        self.out = torch.empty((inp.batch * inp.qo_len, 16, 512), dtype=torch.bfloat16, device=dev)
        self.plan = binding.mla_decode_plan(inp.batch, inp.max_kv_len, sms, qo_len=inp.qo_len)
        self.ws = binding.new_workspace(self.plan)
        self.bytes = algorithmic_bytes(inp)
        self.bytes_bf16 = algorithmic_bytes(inp, "bf16")
        self.bytes_mx = algorithmic_bytes(inp, "mxfp4")
        self.binding = binding
        torch.cuda.synchronize()
        self.inp.kv_bits = None  # release the host copy of the cache source

    def call(self, stream=None):
        self.binding.mla_decode_fwd(self.q, self.kv, self.kv_scale, self.qo_indptr, self.kv_indptr,
                                    self.out, stream, plan=self.plan, workspace=self.ws,
                                    kv_indices=self.kv_indices)

    def call_bf16kv(self, stream=None):
        self.binding.mla_decode_fwd_bf16kv(self.q, self.kv_bf16, self.qo_indptr, self.kv_indptr,
                                           self.out, stream, plan=self.plan, workspace=self.ws,
                                           kv_indices=self.kv_indices)

    def call_mxfp4(self, stream=None):
        self.binding.mla_decode_fwd_mxfp4(self.q, self.kv_fp4, self.kv_mxs, self.qo_indptr,
                                          self.kv_indptr, self.out, stream, plan=self.plan,
                                          workspace=self.ws)

    def stage1_mxfp4(self, stream=None):
        self.binding.mla_decode_stage1_mxfp4(self.q, self.kv_fp4, self.kv_mxs, self.qo_indptr,
                                             self.kv_indptr, self.out, stream, plan=self.plan,
                                             workspace=self.ws)

    def stage1(self, stream=None):
        self.binding.mla_decode_stage1(self.q, self.kv, self.kv_scale, self.qo_indptr,
                                       self.kv_indptr, self.out, stream, plan=self.plan,
                                       workspace=self.ws, kv_indices=self.kv_indices)

    def stage1_bf16kv(self, stream=None):
        self.binding.mla_decode_stage1_bf16kv(self.q, self.kv_bf16, self.qo_indptr,
                                              self.kv_indptr, self.out, stream, plan=self.plan,
                                              workspace=self.ws, kv_indices=self.kv_indices)

    def timed(self, cache: str):
        """(whole step, stage 1 alone, algorithmic bytes) for the selected cache format."""
        if cache == "bf16":
            return self.call_bf16kv, self.stage1_bf16kv, self.bytes_bf16
        if cache == "mxfp4":
            return self.call_mxfp4, self.stage1_mxfp4, self.bytes_mx
        return self.call, self.stage1, self.bytes


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


def per_call_cold(torch, call, reps: int, stream, flush, clean=None) -> tuple:
    """Per-call device times (µs) of ``call(stream)`` with L2 flushed before each
    call, and how many of the calls the host enqueued too late.

    The flush writes a buffer of twice the L2 size; ``clean`` (as large) is then
    read, so that the flush's dirty lines are written back before the timed
    call rather than while it reads its inputs (both outside the events).  A
    device-side wait of ~0.5 ms then holds the stream while the host records
    the start event and enqueues the call, so that the host's launch path stays
    outside the timed region; a call whose start event had already completed
    when the host finished enqueueing it counts as late (its time holds host
    latency)."""
    times, late = [], 0
    for _ in range(reps):
        flush.add_(1)
        if clean is not None:
            clean.max()
        # The flush kernels end before the start event (the call, a programmatic
        # dependent launch, must not overlap them).
        torch.cuda.synchronize()
        torch.cuda._sleep(1_000_000)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        call(stream)
        late += int(s.query())
        e.record(stream)
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e) * 1e3)
    return times, late


def graph_back_to_back(torch, call, n: int, reps: int = 5) -> float:
    """Device µs per call of ``n`` calls back to back, captured once in a CUDA
    graph and replayed (median of ``reps`` replays): the host's launch path,
    longer than a small call, stays out of it.  A call that cannot be captured
    is timed eagerly instead (a negative return marks that)."""
    try:
        return _graph_back_to_back(torch, call, n, reps)
    except RuntimeError:
        torch.cuda.synchronize()
        return -time_loop(torch, call, n, torch.cuda.current_stream()) / n * 1e3


def _graph_back_to_back(torch, call, n: int, reps: int) -> float:
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            call(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for _ in range(n):
            call(side)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(side)
        with torch.cuda.stream(side):
            g.replay()
        e.record(side)
        torch.cuda.synchronize()
        out.append(s.elapsed_time(e) * 1e3 / n)
    del g
    return statistics.median(out)


def e2e_timing(torch, w: DeviceWorkload, steps: int, stream) -> dict:
    """Host-buffer round trip per call: pinned H2D of the step's inputs, the
    decode call, D2H of the output, all inside the timed region."""
    cache = getattr(w, "cache", "e4m3")
    keys = {"e4m3": ("q", "kv", "kv_scale"), "bf16": ("q", "kv_bf16"),
            "mxfp4": ("q", "kv_fp4", "kv_mxs")}[cache] + ("qo_indptr", "kv_indptr")
    host = {k: getattr(w, k).cpu().pin_memory() for k in keys}
    if w.kv_indices is not None:
        host["kv_indices"] = w.kv_indices.cpu().pin_memory()
    out_host = torch.empty(w.out.shape, dtype=w.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()
    dev = {k: torch.empty_like(v, device="cuda") for k, v in host.items()}

    def step():
        for k, v in host.items():
            dev[k].copy_(v, non_blocking=True)
        if cache == "mxfp4":
            w.binding.mla_decode_fwd_mxfp4(dev["q"], dev["kv_fp4"], dev["kv_mxs"], dev["qo_indptr"],
                                           dev["kv_indptr"], w.out, stream, plan=w.plan,
                                           workspace=w.ws)
        elif cache == "bf16":
            w.binding.mla_decode_fwd_bf16kv(dev["q"], dev["kv_bf16"], dev["qo_indptr"],
                                            dev["kv_indptr"], w.out, stream, plan=w.plan,
                                            workspace=w.ws, kv_indices=dev.get("kv_indices"))
        else:
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


# ---------------------------------------------------------------- CPU oracle legs
class OracleSample:
    """The float64 oracle on single batch rows of a workload (quantisation is
    input preparation and stays outside the timed calls)."""

    def __init__(self, name: str, cache: str = "e4m3"):
        from mla_decode_attention_08_gb300.inputs import bf16_bits_to_f32
        from oracle.attention import bf16_bits_to_f64
        from oracle.quant import per_tensor_scale
        self.cache = cache
        self.inp = make_inputs(name)
        self.kv_f32 = bf16_bits_to_f32(self.inp.kv_bits)
        self.inp.kv_bits = None
        self.scale = per_tensor_scale(self.kv_f32)
        self.q = bf16_bits_to_f64(self.inp.q_bits)

    def prepare(self, b: int):
        """The row's cache in the selected format (a tuple of arrays) and its length."""
        from mla_decode_attention_08_gb300.inputs import f32_to_bf16_bits
        from oracle.mxfp4 import quantize_rows
        from oracle.quant import encode_with_scale
        inp = self.inp
        j0, j1 = int(inp.kv_indptr[b]), int(inp.kv_indptr[b + 1])
        slots = np.arange(j0, j1) if inp.kv_indices is None else inp.kv_indices[j0:j1].astype(np.int64)
        rows = self.kv_f32[slots]
        if self.cache == "mxfp4":
            return quantize_rows(rows.astype(np.float64)), j1 - j0
        if self.cache == "bf16":
            return (f32_to_bf16_bits(rows),), j1 - j0
        return (encode_with_scale(rows, self.scale),), j1 - j0

    def run_row(self, b: int, prepared) -> float:
        """Seconds of one oracle call restricted to row b."""
        from oracle.attention import mla_decode_ref, mla_decode_ref_bf16kv
        from oracle.mxfp4 import mla_decode_ref_mxfp4
        data, length = prepared
        n = self.inp.qo_len
        t0 = int(self.inp.qo_indptr[b])
        q, qo, kv = self.q[t0:t0 + n], np.array([0, n]), np.array([0, length])
        t = time.perf_counter()
        if self.cache == "mxfp4":
            mla_decode_ref_mxfp4(q, data[0], data[1], qo, kv)
        elif self.cache == "bf16":
            mla_decode_ref_bf16kv(q, data[0], qo, kv)
        else:
            mla_decode_ref(q, data[0], self.scale, qo, kv)
        return time.perf_counter() - t


def host_cores() -> int:
    """Host cores this process may run on (its CPU affinity)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def run_rows_parallel(o: "OracleSample", jobs, cores: int) -> float:
    """Wall seconds of the oracle over prepared rows, ``cores`` rows at a time
    (one host thread per row; numpy's kernels and BLAS release the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(cores) as ex:
        t = time.perf_counter()
        list(ex.map(lambda job: o.run_row(*job), jobs))
        return time.perf_counter() - t


def oracle_sample_main(name: str, budget_s: float, cache: str = "e4m3") -> None:
    """Worker: time the oracle on as many rows as fit the budget, on every host
    core (one row per thread), plus one row alone on one core; print JSON."""
    o = OracleSample(name, cache)
    batch = o.inp.batch
    cores = host_cores()
    first = o.run_row(0, o.prepare(0))
    n = int(max(1, min(batch, budget_s * cores / max(first, 1e-6))))
    rows = [int(b) for b in np.linspace(0, batch - 1, n).astype(int)]
    jobs = [(b, o.prepare(b)) for b in rows]   # quantisation: input preparation, untimed
    wall = run_rows_parallel(o, jobs, cores)
    # extrapolate by cached tokens, which is what the oracle's work scales with
    tok = np.diff(o.inp.kv_indptr.astype(np.int64))
    sampled = int(tok[rows].sum())
    call_us = wall / max(1, sampled) * int(tok.sum()) * 1e6
    single_us = first / max(1, int(tok[0])) * int(tok.sum()) * 1e6
    print(json.dumps({"value": round(call_us, 1), "unit": "us/call", "cores": cores,
                      "kind": "oracle",
                      "sample": f"{n} of {batch} rows ({sampled} cached tokens) on {cores} threads, "
                                f"{wall:.1f} s wall, extrapolated by cached tokens",
                      "single_core_value": round(single_us, 1),
                      "single_core_sample": f"row 0 alone ({int(tok[0])} cached tokens) on one "
                                            f"thread, {first:.2f} s"}))


def cpu_baseline(name: str, budget_s: float = 15.0, cache: str = "e4m3"):
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", name, "--budget", str(budget_s),
           "--cache", cache]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        tail = r.stderr.strip().splitlines()[-1][:200] if r.stderr.strip() else "no output"
        return {"value": None, "unit": "us/call", "cores": host_cores(), "kind": "oracle",
                "sample": "failed: " + tail}
    return json.loads(r.stdout.strip().splitlines()[-1])


def reference_main(args) -> None:
    """The reference arm: the float64 oracle on the host cores, same workload and metric.

    Each step runs the oracle on ``cores`` batch rows at once (one host thread
    per row), each restricted to its first n cached tokens, n sized from a
    calibration call so that warm-up plus timed steps take about
    ``--ref-budget`` seconds; the wall time per token is extrapolated to the
    whole call."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if int(os.environ.get("RANK", "0")) != 0:
        return
    o = OracleSample(args.workload, args.cache)
    batch = o.inp.batch
    cores = host_cores()
    tok = np.diff(o.inp.kv_indptr.astype(np.int64))
    calib_row = int(np.argmax(tok))
    data_c, len_c = o.prepare(calib_row)
    per_tok = o.run_row(calib_row, (data_c, len_c)) / max(1, len_c)
    n_steps = args.warmup + args.steps
    cap = int(args.ref_budget / max(n_steps * per_tok, 1e-12))
    step_rows = [[(cores * i + k) * 37 % batch for k in range(cores)] for i in range(n_steps)]
    prepared = {}
    for b in {b for rows in step_rows for b in rows}:
        data, length = o.prepare(b)
        n = max(1, min(length, cap))
        prepared[b] = (tuple(a[:n] for a in data), n)
    for rows in step_rows[:args.warmup]:
        run_rows_parallel(o, [(b, prepared[b]) for b in rows], cores)
    timed = step_rows[args.warmup:]
    total = 0.0
    for rows in timed:
        total += run_rows_parallel(o, [(b, prepared[b]) for b in rows], cores)
    done = sum(prepared[b][1] for rows in timed for b in rows)
    call_us = total / max(1, done) * int(tok.sum()) * 1e6
    sample = (f"{len(timed)} steps of {cores} single-row oracle calls in parallel ({cores} threads) "
              f"over {done} cached tokens (at most {cap} per row), extrapolated by cached tokens "
              f"to the {batch}-row call")
    line = {"impl": "reference", "metric": METRIC, "value": round(call_us, 1), "unit": "us/call",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total * 1e3 / max(1, len(timed)), 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload, world, args.cache),
            "cpu_baseline": {"value": round(call_us, 1), "unit": "us/call", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(call_us, 1), "unit": "us/call", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


CACHE_DESC = {"e4m3": "e4m3fn, per-tensor scale", "bf16": "bf16",
              "mxfp4": "MXFP4 (E2M1 elements, E8M0 scale per 32)"}
DTYPE_DESC = {"e4m3": "e4m3 x e4m3 -> f32 (tcgen05 kind::f8f6f4), bf16 out",
              "bf16": "bf16 x bf16 -> f32 (tcgen05 kind::f16), bf16 out",
              "mxfp4": "MXFP4 converted to e4m3 in shared memory; e4m3 x e4m3 -> f32 "
                       "(tcgen05 kind::f8f6f4), bf16 out"}


def workload_config(name: str, world: int, cache: str = "e4m3") -> dict:
    w = WORKLOADS[name]
    return {"workload": name, "batch": w.batch, "kv_len": w.kv_len,
            "kv_len_dist": "uniform 1..kv_len" if w.ragged else "fixed",
            "page_table": "random permutation, page size 1" if w.paged else "identity",
            "heads": 16, "qk_head_dim": 576, "v_head_dim": 512,
            "kv_cache": CACHE_DESC[cache], "qseqlen": w.qo_len,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "cache larger than L2, no flush between steps"}


# ---------------------------------------------------------------- main
def max_over_ranks(value: float, dist=None, device: str = "cpu") -> float:
    """The slowest rank's value (a step ends when every replica has finished)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_bytes(name: str, cache: str = "e4m3") -> int:
    """Algorithmic bytes of a workload from its shapes only."""
    from mla_decode_attention_08_gb300.inputs import workload_lengths
    wl = WORKLOADS[name]
    lengths = workload_lengths(wl)

    class _Shape:
        batch = wl.batch
        qo_len = wl.qo_len
        kv_indptr = np.concatenate([[0], np.cumsum(lengths)])
        kv_indices = np.zeros(1) if wl.paged else None
    return algorithmic_bytes(_Shape, cache)


def ours_main(args) -> None:
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from mla_decode_attention_08_gb300 import binding
    from mla_decode_attention_08_gb300.build import build
    binding.load_library(build())
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    w = DeviceWorkload(args.workload, torch, binding, sms)
    # kernels a call launches: stage 1 and stage 2, or stage 1 alone under the
    # cluster split (which combines inside stage 1; not for a page table or an
    # MXFP4 cache, which run the persistent split from the same plan)
    kernels_per_call = 1 if (w.plan.cluster and w.kv_indices is None and args.cache != "mxfp4") else 2
    if args.cache != "e4m3" and (w.kv_indices is not None or (args.cache == "mxfp4" and not w.mx)):
        raise SystemExit(f"--cache {args.cache} takes contiguous workloads"
                         + (" with one query token per row" if args.cache == "mxfp4" else ""))
    w.cache = args.cache
    step_fn, stage1_fn, step_bytes = w.timed(args.cache)
    for _ in range(args.warmup):
        step_fn(stream)
    barrier()
    sampler = ClockSampler(local).start()
    time.sleep(0.3)  # let the sampler attach before the timed region
    barrier()
    t0 = time.time()
    ms = time_loop(torch, step_fn, args.steps, stream)
    t1 = time.time()
    barrier()
    clocks = sampler.stop(t0, t1)
    ms_step = max_over_ranks(ms / args.steps, dist, "cuda")
    if binding.mla_decode_read_error(w.ws) != 0:
        raise SystemExit("device error word set during the benchmark")

    # stage 1 alone, the dominant kernel, for the roofline
    for _ in range(3):
        stage1_fn(stream)
    ms1 = time_loop(torch, stage1_fn, args.steps, stream) / args.steps
    peak, peak_src = measured_peak()
    achieved = step_bytes / (ms1 * 1e-3) / 1e9
    us_call = ms_step * 1e3
    eff_tbps = step_bytes / (us_call * 1e-6) / 1e12

    per_config = []
    if not args.no_per_config and rank == 0:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
        clean = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
        def cold(call, nbytes):
            for _ in range(5):
                call(stream)
            times, late = per_call_cold(torch, call, args.cold_reps, stream, flush, clean)
            med = statistics.median(times)
            return {"us_median": round(med, 2),
                    "us_p10": round(float(np.percentile(times, 10)), 2),
                    "us_p90": round(float(np.percentile(times, 90)), 2),
                    "effective_tbps": round(nbytes / (med * 1e-6) / 1e12, 3),
                    "frac_of_peak": round(nbytes / (med * 1e-6) / 1e9 / peak, 3),
                    "algorithmic_bytes": nbytes, "host_late_calls": late}

        for name in WORKLOADS:
            ww = w if name == args.workload else DeviceWorkload(name, torch, binding, sms)
            entry = {"workload": name, **cold(ww.call, ww.bytes), "grid": int(ww.plan.grid),
                     "cluster": int(ww.plan.cluster),
                     "l2": "flushed before each call (2x L2 written, then 2x L2 of other data read)"}
            # the same step back to back (L2 warm for the small workloads), for
            # reference: 50 calls replayed from a CUDA graph
            entry["us_back_to_back"] = round(graph_back_to_back(torch, ww.call, 50), 2)
            # the same step over the bf16 cache (mla_decode_fwd_bf16kv; contiguous caches only)
            if ww.kv_indices is None:
                bf = cold(ww.call_bf16kv, ww.bytes_bf16)
                bf["us_back_to_back"] = round(graph_back_to_back(torch, ww.call_bf16kv, 50), 2)
                entry["bf16_cache"] = bf
            else:
                entry["bf16_cache"] = {"unsupported": "page table (bf16 caches are read contiguously)"}
            # and over the MXFP4 cache (mla_decode_fwd_mxfp4), with its stage 1 timed
            # alone back to back (the MXFP4 kernel's roofline)
            if ww.mx:
                mx = cold(ww.call_mxfp4, ww.bytes_mx)
                us_mx = graph_back_to_back(torch, ww.call_mxfp4, 50)
                us_mx1 = graph_back_to_back(torch, ww.stage1_mxfp4, 50)
                mx["us_back_to_back"] = round(us_mx, 2)
                mx["stage1_us_back_to_back"] = round(us_mx1, 2)
                mx["stage1_frac_of_peak"] = round(ww.bytes_mx / (us_mx1 * 1e-6) / 1e9 / peak, 3)
                if binding.mla_decode_read_error(ww.ws) != 0:
                    raise SystemExit("device error word set during the MXFP4 timing")
                entry["mxfp4_cache"] = mx
            else:
                entry["mxfp4_cache"] = {"unsupported": "page table or several query tokens per row"}
            per_config.append(entry)
            if ww is not w:
                del ww
                torch.cuda.empty_cache()
        del flush, clean

    if args.cache != "bf16":
        w.kv_bf16 = None
    if args.cache != "mxfp4":
        w.kv_fp4 = w.kv_mxs = None
    torch.cuda.empty_cache()
    e2e = e2e_timing(torch, w, args.e2e_steps, stream)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        del w
        torch.cuda.empty_cache()
        cpu = cpu_baseline(args.workload, args.cpu_budget, args.cache)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": round(us_call, 2), "unit": "us/call", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE_DESC[args.cache], "data": "synthetic",
        "config": workload_config(args.workload, world, args.cache),
        "effective_tbps": round(eff_tbps, 3),
        "aggregate_effective_tbps": round(eff_tbps * world, 3),
        "frac_of_peak": round(eff_tbps * 1e3 / peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": recorded_traffic(args.workload, args.cache),
                     "kernel": "mla_decode_stage1_kernel", "peak_source": f"{peak_src} hbm_gbs",
                     "stage1_us_per_launch": round(ms1 * 1e3, 2),
                     "algorithmic_bytes_per_launch": workload_bytes(args.workload, args.cache)},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": kernels_per_call * args.steps, "clocks": clocks,
        "per_config": per_config,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=list(WORKLOADS))
    ap.add_argument("--cache", default="e4m3", choices=["e4m3", "bf16", "mxfp4"],
                    help="cache format of the timed step (the e4m3 cache is the headline)")
    ap.add_argument("--cold-reps", type=int, default=30)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=60.0)
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-sample", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--budget", type=float, default=15.0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_sample:
        oracle_sample_main(args.oracle_sample, args.budget, args.cache)
    elif args.impl == "reference":
        reference_main(args)
    else:
        if args.warmup < 3:
            raise SystemExit("--warmup must be at least 3")
        ours_main(args)


if __name__ == "__main__":
    main()
