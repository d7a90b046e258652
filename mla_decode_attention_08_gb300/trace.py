"""Start-up breakdown of one decode call, from the trace build's clock stamps.

    python -m mla_decode_attention_08_gb300.trace --workload bs4_kv1024 [--calls 20] [--cold]

Builds ``libmla_decode_trace.so`` (``-DMLA_TRACE``), runs the workload's decode
step ``--calls`` times back to back (or once after an idle GPU with
``--cold``), and prints, for the last call, where each stage-1 CTA's time went
on its way to its first output (SM cycles from the CTA's entry, median and
maximum over CTAs) and the two kernels' spans on the global timer.  The stamps
cost a few stores per CTA; the numbers describe the release kernels to within
that.
"""
from __future__ import annotations

import argparse
import sys

import numpy as np

EVENTS = [
    (2, "before the wait for the previous kernel"),
    (3, "after that wait"),
    (4, "schedule prologue done"),
    (5, "producer: first cache copy issued"),
    (6, "softmax: first Q operand published"),
    (7, "QK issuer: first rope panel landed"),
    (8, "QK issuer: first tile's QK issued"),
    (9, "softmax: first scores read"),
    (10, "softmax: first P published"),
    (11, "PV issuer: first PV issued"),
    (12, "softmax: first epilogue starts"),
    (13, "softmax: first output stores issued"),
    (14, "exit barrier passed"),
    (16, "prologue: thread 0's kv_indptr loads returned"),
    (33, "prologue: the batch's totals known"),
    (34, "prologue: first row found, its L2 prefetches issued"),
    (35, "producer: loop starts"),
    (38, "producer: first panel's barrier about to be armed"),
    (36, "softmax: loop starts"),
    (37, "softmax: first query loads issued"),
    (17, "prologue: first block barrier passed"),
    (18, "softmax: first query loads returned"),
    (19, "observer: first rope panel arrived"),
    (20, "observer: first tile's last latent panel arrived"),
    (21, "cluster split: cluster barrier passed"),
    (32, "cluster split: the partials landed"),
    (31, "cluster split: thread 0's combine weight formed"),
    (22, "cluster split: combine written"),
    (24, "softmax: first segment's last P published"),
    (25, "softmax: second segment's Q operand published"),
    (26, "softmax: second segment's first scores read"),
    (27, "softmax: second segment's first P published"),
    (28, "PV issuer: second segment's first PV issued"),
]


def summarise(s1: np.ndarray, s2: np.ndarray, workload: str, mode: str) -> str:
    live = s1[:, 1] > 0
    t = s1[live].astype(np.int64)
    clk = t[:, 1:] - t[:, [1]]                         # cycles since entry
    span_ns = (t[:, 15] - t[:, 0]).astype(np.float64)
    mhz = np.median((t[:, 14] - t[:, 1]) / np.maximum(span_ns, 1.0)) * 1e3
    e0 = int(t[:, 0].min())
    lines = [f"# Start-up trace: {workload} ({mode})", "",
             f"{int(live.sum())} stage-1 CTAs; SM clock from the stamps ~{mhz:.0f} MHz.", "",
             "| stage-1 milestone | cycles from CTA entry, median | max | us, median |",
             "|---|---|---|---|"]
    for ev, name in EVENTS:
        col = clk[:, ev - 1]
        ok = t[:, ev] > 0
        if not ok.any():
            continue
        med, mx = float(np.median(col[ok])), float(np.max(col[ok]))
        lines.append(f"| {name} | {med:.0f} | {mx:.0f} | {med / mhz:.2f} |")
    shape = t[:, 23]
    if shape.any():
        segs, tiles = shape >> 16, shape & 0xFFFF
        exit_ns = t[:, 15] - e0
        lines += ["", "| CTAs by (segments, tiles) | count | exit ns, median | exit ns, max |",
                  "|---|---|---|---|"]
        for key in sorted(set(zip(segs.tolist(), tiles.tolist()))):
            sel = (segs == key[0]) & (tiles == key[1])
            lines.append(f"| {key[0]} segments, {key[1]} tiles | {int(sel.sum())} | "
                         f"{int(np.median(exit_ns[sel]))} | {int(exit_ns[sel].max())} |")
    two = (shape >> 16) >= 2 if shape.any() else np.zeros(len(t), bool)
    if two.any():
        base = t[two, 24]
        lines += ["", "| segment boundary (CTAs with two or more segments) | cycles after the first "
                  "segment's last P, median | max |", "|---|---|---|"]
        for ev, name in ((29, "second segment's Q preparation starts"),
                         (30, "second segment's query loads returned"),
                         (25, "second segment's Q operand published"),
                         (12, "first segment's epilogue starts (its last PV done)"),
                         (13, "first segment's output stores issued"),
                         (26, "second segment's first scores read"),
                         (27, "second segment's first P published"),
                         (28, "second segment's first PV issued")):
            d = t[two, ev] - base
            lines.append(f"| {name} | {int(np.median(d))} | {int(d.max())} |")
    live2 = s2[:, 0] > 0
    u = s2[live2].astype(np.int64)
    lines += ["", "| global timer (ns from the first stage-1 CTA's entry) | first | last |",
              "|---|---|---|",
              f"| stage-1 CTA entry | 0 | {int(t[:, 0].max()) - e0} |",
              f"| stage-1 CTA exit | {int(t[:, 15].min()) - e0} | {int(t[:, 15].max()) - e0} |"]
    if live2.any():
        lines += [f"| stage-2 block entry | {int(u[:, 0].min()) - e0} | {int(u[:, 0].max()) - e0} |",
                  f"| stage-2 block after its wait for stage 1 | {int(u[:, 1].min()) - e0} | "
                  f"{int(u[:, 1].max()) - e0} |",
                  f"| stage-2 block exit | {int(u[:, 2].min()) - e0} | {int(u[:, 2].max()) - e0} |"]
    return "\n".join(lines) + "\n"


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--workload", default="bs4_kv1024")
    ap.add_argument("--calls", type=int, default=20)
    ap.add_argument("--cold", action="store_true", help="one call on an idle GPU")
    ap.add_argument("--flush", action="store_true",
                    help="with --cold: write then read two L2-sized buffers before the call, "
                         "as the benchmark's flushed timing does")
    ap.add_argument("--lib", default=None, help="a trace-built library to load instead of building one")
    args = ap.parse_args(argv)

    import torch

    from . import binding
    from .build import build
    from .inputs import make_inputs

    binding.load_library(args.lib or build(trace=True))
    inp = make_inputs(args.workload)

    def dev16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()

    q = dev16(inp.q_bits)
    kv = dev16(inp.kv_bits)
    codes = torch.empty((kv.shape[0], 576), dtype=torch.uint8, device="cuda")
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    binding.mla_fp8_quantize_per_tensor(kv, codes, scale, torch.empty(16, dtype=torch.uint8, device="cuda"))
    del kv
    qo = torch.from_numpy(inp.qo_indptr).cuda()
    kvi = torch.from_numpy(inp.kv_indptr).cuda()
    idx = None if inp.kv_indices is None else torch.from_numpy(inp.kv_indices).cuda()
    out = torch.empty((inp.batch * inp.qo_len, 16, 512), dtype=torch.bfloat16, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = binding.mla_decode_plan(inp.batch, inp.max_kv_len, sms, qo_len=inp.qo_len)
    ws = binding.new_workspace(plan)

    def call():
        binding.mla_decode_fwd(q, codes, scale, qo, kvi, out, plan=plan, workspace=ws, kv_indices=idx)

    for _ in range(5):
        call()
    torch.cuda.synchronize()
    binding.mla_decode_trace_read(clear=True)
    if args.cold and args.flush:
        l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 129 << 20)
        flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device="cuda")
        clean = torch.zeros_like(flush)
        flush.add_(1)
        clean.max()
        torch.cuda.synchronize()
        torch.cuda._sleep(1_000_000)  # the call is enqueued before the stream reaches it
    for _ in range(1 if args.cold else args.calls):
        call()
    torch.cuda.synchronize()
    if binding.mla_decode_read_error(ws) != 0:
        raise SystemExit("device error word set")
    s1, s2 = binding.mla_decode_trace_read(clear=True)
    mode = ("one call on an idle GPU" + (", L2 flushed before it" if args.flush else "")
            if args.cold else f"last of {args.calls} calls back to back")
    sys.stdout.write(summarise(s1, s2, args.workload, mode))


if __name__ == "__main__":
    main()
