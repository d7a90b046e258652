"""The start-up breakdown printed from a trace build's stamps
(`mla_decode_attention_08_gb300.trace.summarise`), on synthetic stamps whose
medians, maxima and tables are known: the stamp layout (entry and exit on the
global timer and the SM clock, event columns, the CTA-shape word) is the one
the kernels write, so a mislabelled column or a wrong unit shows here."""
import numpy as np

from mla_decode_attention_08_gb300 import binding, trace


def _stamps():
    s1 = np.zeros((binding.TRACE_CTAS, binding.TRACE_EVENTS), dtype=np.uint64)
    s2 = np.zeros((binding.TRACE2_BLOCKS, 3), dtype=np.uint64)
    # three CTAs; SM clock 2,000 MHz: 2 cycles per ns
    for c, (entry_ns, clk0, extra, segs, tiles) in enumerate(
            [(1000, 50_000, 0, 1, 3), (1100, 60_000, 100, 1, 3), (1200, 70_000, 400, 2, 2)]):
        s1[c, 0] = entry_ns                  # global timer at entry
        s1[c, 1] = clk0                      # SM clock at entry
        s1[c, 4] = clk0 + 2000 + extra       # schedule prologue done
        s1[c, 11] = clk0 + 9000 + extra      # first PV issued
        s1[c, 14] = clk0 + 20_000 + 2 * extra  # exit barrier passed
        s1[c, 15] = entry_ns + 10_000 + extra  # global timer at exit: 20,000 cycles = 10,000 ns
        s1[c, 23] = segs * 65536 + tiles     # CTA shape
    s2[0] = (10_500, 11_500, 12_000)
    s2[1] = (10_700, 11_600, 12_400)
    return s1, s2


def test_summary_tables():
    s1, s2 = _stamps()
    text = trace.summarise(s1, s2, "bs_test", "synthetic")
    lines = text.splitlines()
    assert lines[0] == "# Start-up trace: bs_test (synthetic)"
    assert "3 stage-1 CTAs; SM clock from the stamps ~2000 MHz." in text
    row = {l.split(" | ")[0].lstrip("| "): l for l in lines if l.startswith("| ")}
    # medians and maxima in cycles from each CTA's entry, and the median in us at 2 GHz
    assert row["schedule prologue done"] == "| schedule prologue done | 2100 | 2400 | 1.05 |"
    assert row["PV issuer: first PV issued"] == "| PV issuer: first PV issued | 9100 | 9400 | 4.55 |"
    # events never stamped are left out
    assert "QK issuer: first tile's QK issued" not in row
    # CTA shapes with their exit times on the global timer, from the first entry
    assert row["1 segments, 3 tiles"] == "| 1 segments, 3 tiles | 2 | 10100 | 10200 |"
    assert row["2 segments, 2 tiles"] == "| 2 segments, 2 tiles | 1 | 10600 | 10600 |"
    assert row["stage-1 CTA entry"] == "| stage-1 CTA entry | 0 | 200 |"
    assert row["stage-1 CTA exit"] == "| stage-1 CTA exit | 10000 | 10600 |"
    assert row["stage-2 block entry"] == "| stage-2 block entry | 9500 | 9700 |"
    assert row["stage-2 block after its wait for stage 1"] == "| stage-2 block after its wait for stage 1 | 10500 | 10600 |"
    assert row["stage-2 block exit"] == "| stage-2 block exit | 11000 | 11400 |"


def test_cta_rows_without_stamps_are_ignored():
    s1, s2 = _stamps()
    s1[5, 0] = 999   # a global-timer entry stamp alone (no clock stamps): not a live CTA
    text = trace.summarise(s1, s2, "bs_test", "synthetic")
    assert "3 stage-1 CTAs" in text
