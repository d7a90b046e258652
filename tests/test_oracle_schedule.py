"""Pins of the oracle's split schedule: a hand-derived case and partition invariants."""
import numpy as np
import pytest

from oracle.schedule import TILE_TOKENS, plan_grid, schedule, token_segments, worker_table

from .golden_util import load_table


def test_hand_derived_case():
    sch = schedule([0, 300, 300, 1000, 1128], 4)
    got = [[s["worker"], s["row"], s["tile_begin"], s["tile_end"], int(s["split"]), s["slot"]]
           for s in sch["segments"]]
    want = [[int(v) for v in row] for row in load_table("schedule_small.txt")]
    assert got == want
    assert sch["prefix"] == [0, 3, 3, 9, 10]
    assert worker_table([0, 300, 300, 1000, 1128], 4).tolist() == [
        [0, 2, 0, 0], [2, 5, 0, 2], [5, 7, 2, 2], [7, 10, 2, 3]]


@pytest.mark.parametrize("batch,max_len,sms,want", [
    (4, 1024, 152, 32), (32, 1024, 152, 128), (64, 8192, 152, 152), (256, 8192, 152, 152),
    (64, 8192, 76, 76), (1, 0, 152, 1), (3, 1, 152, 3), (0, 100, 152, 1), (200, 128, 152, 100)])
def test_plan_grid(batch, max_len, sms, want):
    assert plan_grid(batch, max_len, sms) == want


def random_indptr(rng, batch, max_len, zero_frac=0.1):
    lengths = rng.integers(1, max_len + 1, size=batch)
    lengths[rng.random(batch) < zero_frac] = 0
    return np.concatenate([[0], np.cumsum(lengths)])


@pytest.mark.parametrize("seed", range(8))
def test_partition_invariants(seed):
    rng = np.random.default_rng(seed)
    batch = int(rng.integers(1, 40))
    indptr = random_indptr(rng, batch, int(rng.integers(1, 3000)))
    grid = int(rng.integers(1, 160))
    sch = schedule(indptr, grid)
    total = sch["total_tiles"]
    sizes = [w["t1"] - w["t0"] for w in sch["workers"]]
    assert sum(sizes) == total and max(sizes) - min(sizes) <= 1
    # segments tile every row exactly once, in order
    segs = token_segments(indptr, grid)
    for b in range(batch):
        length = int(indptr[b + 1] - indptr[b])
        ranges = segs.get(b, [])
        if length == 0:
            assert ranges == []
            continue
        assert ranges[0][0] == 0 and ranges[-1][1] == length
        assert all(r0 < r1 for r0, r1 in ranges)
        assert all(a[1] == b_[0] for a, b_ in zip(ranges, ranges[1:]))
        assert all(r0 % TILE_TOKENS == 0 for r0, _ in ranges)
    # slots: unique, two per worker at most, only for split rows
    slots = [s["slot"] for s in sch["segments"] if s["split"]]
    assert len(slots) == len(set(slots))
    assert all(0 <= s < 2 * grid for s in slots)
    assert all(s["slot"] == -1 for s in sch["segments"] if not s["split"])
    # closed forms the CUDA side uses: worker of tile t, and first/last rows
    for t in range(total):
        c = ((t + 1) * grid - 1) // total
        w = sch["workers"][c]
        assert w["t0"] <= t < w["t1"]
    # a row is covered by every non-empty worker between its first and last one
    nonempty = [c for c, w in enumerate(sch["workers"]) if w["t1"] > w["t0"]]
    for b, ws in sch["covers"].items():
        if ws:
            assert ws == [c for c in nonempty if ws[0] <= c <= ws[-1]]
