"""Pins of the oracle's split schedule: a hand-derived case and partition invariants."""
import numpy as np
import pytest

from oracle.schedule import (TILE_TOKENS, cluster_shares, plan_cluster, plan_grid, row_start_units,
                             schedule, token_segments, worker_table)

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


@pytest.mark.parametrize("tiles,grid,want", [
    (30, 3, 3),    # ranges of 10 tiles >= 8: three start units per row
    (20, 3, 0),    # ceil(20 / 3) = 7 < 8
    (8, 1, 3), (7, 1, 0), (0, 5, 0), (4096, 152, 3), (256, 128, 0), (16384, 152, 3)])
def test_row_start_units_by_hand(tiles, grid, want):
    assert row_start_units(tiles, grid) == want


def test_hand_derived_case_with_row_start_units():
    """Rows of 20 and 10 tiles over 3 workers: 30 tiles, ranges of 10 >= 8, so
    each row is preceded by 3 start units.  Units: row 0 start [0, 3), tiles
    [3, 23); row 1 start [23, 26), tiles [26, 36); 36 units, workers [0, 12),
    [12, 24), [24, 36).  Worker 0 holds row 0's tiles 0-8, worker 1 its tiles
    9-19 (and one start unit of row 1, no tile of it), worker 2 row 1 whole.
    Row 0 is split: worker 0's range begins before the row's first tile (slot
    2c + 1 = 1), worker 1's after it (slot 2c = 2)."""
    indptr = [0, 2560, 3840]
    sch = schedule(indptr, 3)
    assert sch["row_start"] == 3
    assert sch["prefix"] == [0, 23, 36]
    assert worker_table(indptr, 3).tolist() == [[0, 12, 0, 0], [12, 24, 0, 0], [24, 36, 1, 1]]
    got = [[s["worker"], s["row"], s["tile_begin"], s["tile_end"], int(s["split"]), s["slot"]]
           for s in sch["segments"]]
    assert got == [[0, 0, 0, 9, 1, 1], [1, 0, 9, 20, 1, 2], [2, 1, 0, 10, 0, -1]]
    # an empty row in between takes no units: [0, 13, 13, 26] for 10, 0, 10 tiles
    assert schedule([0, 1280, 1280, 2560], 2)["prefix"] == [0, 13, 13, 26]


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
    grid = int(rng.integers(1, 160)) if seed % 2 else int(rng.integers(1, 8))
    sch = schedule(indptr, grid)
    total = sch["total_tiles"]  # units: tiles and start units
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


# The cluster split's size, worked out by hand from its rule (largest of 8, 4, 2
# not above the longest row's tiles whose clusters fit at once: num_sms // 10 of
# 8, 7 num_sms // 32 of 4, num_sms // 2 of 2; taken when ceil(tiles / size) <=
# the persistent longest range + 2).
@pytest.mark.parametrize("batch,max_len,sms,qo_len,want", [
    (4, 1024, 152, 1, 8),      # 8 tiles; 4 <= 15 clusters of 8; share 1 <= 1 + 2
    (32, 1024, 152, 1, 4),     # 32 > 15 of 8; 32 <= 33 of 4; share 2 <= ceil(256/152) + 2
    (34, 1024, 152, 1, 2),     # 34 > 33 of 4; 34 <= 76 of 2; share 4 <= 2 + 2
    (64, 8192, 152, 1, 0),     # of 2 only; share 32 > ceil(4096/152) + 2 = 29
    (256, 8192, 152, 1, 0),    # no size fits
    (4, 8192, 152, 1, 0),      # share 8 > ceil(256/152) + 2 = 4
    (4, 1024, 152, 2, 0),      # two query tokens per row
    (1, 128, 152, 1, 0),       # one tile
    (3, 300, 152, 1, 2),       # 3 tiles: 8 and 4 exceed them; share 2 <= 1 + 2
    (8, 2048, 148, 1, 8),      # 148 // 10 = 14 clusters of 8; share 2 <= 1 + 2
    (16, 2048, 152, 1, 4),     # 16 > 15 of 8; share 4 <= ceil(256/152) + 2 = 4
    (5, 1024, 40, 1, 4),       # 40 // 10 = 4 < 5 of 8; 7*40 // 32 = 8 of 4; share 2 <= 1 + 2
])
def test_plan_cluster_by_hand(batch, max_len, sms, qo_len, want):
    assert plan_cluster(batch, qo_len, max_len, sms) == want


def test_cluster_shares_partition_each_row():
    indptr = [0, 1000, 1000, 1001, 3000, 3129]
    for size in (2, 4, 8):
        sh = cluster_shares(indptr, size)
        for b, n in enumerate([8, 0, 1, 16, 2]):
            ranges = [sh[(b, r)] for r in range(size)]
            assert ranges[0][0] == 0 and ranges[-1][1] == n
            assert all(r0 <= r1 for r0, r1 in ranges)
            assert all(ranges[i][1] == ranges[i + 1][0] for i in range(size - 1))
            k = -(-n // size)
            assert max(r1 - r0 for r0, r1 in ranges) == k
