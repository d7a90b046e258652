"""Token-balanced split-KV schedule, restated with plain loops.

The pages split each row's cache into ``num_kv_splits`` contiguous ranges and
combine the partials afterwards (submission 722089, ``_mla_multihead_stage1``:
``tokens_per_split = ceil(kv_len / NUM_SPLITS)``, split s covers
``[s * tps, min((s + 1) * tps, kv_len))``; submission 663509 and 738050 build
"work" and "reduce" maps for a persistent kernel with ``get_mla_metadata_v1``
from ``qo_indptr`` / ``kv_indptr`` at a token granularity ``kv_granularity``).

The schedule here is the persistent, token-balanced form of that split, fixed
as follows (the pages print no formula for their persistent work map):

* every row is cut into tiles of ``TILE_TOKENS`` tokens, ``ceil(L_b / 128)``
  tiles, the last one partial;
* the grid has the fewest workers ``G`` whose longest equal split of the
  batch's upper bound ``U = B * ceil(max_kv_len / 128)`` tiles is no longer
  than with ``min(num_sms, U)`` workers (1 for an empty batch);
* the rows, row after row, form one global sequence of units: each row with
  tiles contributes ``S`` start units followed by its tiles, where
  ``S = ROW_START_UNITS`` (3) when the batch's ``N`` tiles give ranges of at
  least ``ROW_START_MIN_RANGE`` (8) tiles, ``ceil(N / G) >= 8``, else 0 (a
  worker whose range takes on a row start pays for that row's query
  preparation and the previous segment's epilogue, and gets ``S`` fewer tiles
  for it; this is a property of the library's kernel, not of the pages);
  worker c takes the contiguous unit range ``[floor(c T / G), floor((c+1) T / G))``
  of the ``T`` units;
* the part of a row inside one worker's range is a segment; a row covered by a
  single worker is "whole", otherwise "split" and each of its segments writes a
  partial (normalised output and base-2 log-sum-exp) to a workspace slot:
  slot ``2c`` when worker c's range begins at or after the row's first tile,
  else ``2c + 1``.

Small batches of one query token per row take the cluster split instead
(``plan_cluster``): each row is shared by ``size`` CTAs of one thread-block
cluster, rank r taking the row's tiles ``[r k, min((r + 1) k, n))`` with
``k = ceil(n / size)``, and their partials are combined inside the cluster;
the size follows the rule stated in ``plan_cluster``.

This module is the restatement the CUDA path's schedule must match bit for bit.
"""
from __future__ import annotations

import numpy as np

TILE_TOKENS = 128


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def plan_grid(batch: int, max_kv_len: int, num_sms: int) -> int:
    """Number of persistent workers for a batch of ``batch`` rows: the fewest
    that give no worker more tiles than spreading the batch's upper bound
    ``U = batch * ceil(max_kv_len / 128)`` over ``min(num_sms, U)`` workers."""
    upper = batch * ceil_div(max(0, max_kv_len), TILE_TOKENS)
    g0 = min(num_sms, upper)
    if g0 < 1:
        return 1
    most = ceil_div(upper, g0)          # tiles of the longest range
    for g in range(1, g0 + 1):          # the fewest workers with ranges no longer
        if ceil_div(upper, g) <= most:
            return g
    return g0


def cluster_capacity(size: int, num_sms: int) -> int:
    """Clusters of ``size`` CTAs the GPU runs at once (the library's estimate):
    num_sms // 10 of 8, 7 num_sms // 32 of 4, num_sms // 2 of 2."""
    return {8: num_sms // 10, 4: (7 * num_sms) // 32, 2: num_sms // 2}[size]


def plan_cluster(batch: int, qo_len: int, max_kv_len: int, num_sms: int) -> int:
    """CTAs per row of the cluster split, or 0 for the persistent split.

    Rows of one query token only.  The candidate sizes 8, 4, 2 are tried from
    the largest: a size must not exceed the tiles of the longest row and its
    clusters for the whole batch must fit the GPU at once.  The first that does
    is taken when the longest share it gives, ceil(tiles / size), is at most two
    tiles longer than the persistent split's longest range; otherwise 0.
    """
    tiles = ceil_div(max(0, max_kv_len), TILE_TOKENS)
    if qo_len != 1 or batch < 1 or num_sms < 1 or tiles < 2:
        return 0
    chosen = 0
    for size in (8, 4, 2):
        if size <= tiles and batch <= cluster_capacity(size, num_sms):
            chosen = size
            break
    if chosen == 0:
        return 0
    upper = batch * tiles
    longest = ceil_div(upper, min(num_sms, upper))
    return chosen if ceil_div(tiles, chosen) <= longest + 2 else 0


def cluster_shares(kv_indptr, size: int) -> dict:
    """(row, rank) -> (first tile, end tile) of each CTA's share under the cluster split."""
    out = {}
    for b, n in enumerate(row_tiles(kv_indptr)):
        k = ceil_div(n, size)
        for r in range(size):
            j0 = min(r * k, n)
            out[(b, r)] = (j0, min(j0 + k, n))
    return out


def row_tiles(kv_indptr) -> list[int]:
    """Tiles per row; a decreasing indptr counts as an empty row."""
    out = []
    for b in range(len(kv_indptr) - 1):
        length = int(kv_indptr[b + 1]) - int(kv_indptr[b])
        out.append(ceil_div(length, TILE_TOKENS) if length > 0 else 0)
    return out


ROW_START_UNITS = 3
ROW_START_MIN_RANGE = 8


def row_start_units(total_tiles: int, grid: int) -> int:
    """Start units before each row with tiles: ROW_START_UNITS when the ranges
    hold at least ROW_START_MIN_RANGE tiles (``ceil(N / G) >= 8``), else 0."""
    if grid < 1 or total_tiles < 1:
        return 0
    return ROW_START_UNITS if ceil_div(total_tiles, grid) >= ROW_START_MIN_RANGE else 0


def schedule(kv_indptr, grid: int) -> dict:
    """Per-worker ranges, per-row covers and segment list, by enumeration of
    the unit sequence (each unit labelled with its row and tile, or -1 for a
    start unit)."""
    tiles = row_tiles(kv_indptr)
    start = row_start_units(sum(tiles), grid)
    units = []                       # (row, tile) per unit; tile -1: a start unit
    prefix = []                      # units before each row
    first_tile = []                  # unit index of each row's first tile
    for b, n in enumerate(tiles):
        prefix.append(len(units))
        if n > 0:
            units.extend([(b, -1)] * start)
        first_tile.append(len(units))
        units.extend((b, j) for j in range(n))
    prefix.append(len(units))
    total = len(units)

    workers = []
    for c in range(grid):
        t0 = (c * total) // grid
        t1 = ((c + 1) * total) // grid
        workers.append({"t0": t0, "t1": t1, "first_row": -1, "last_row": -1})

    # Which workers touch which row: enumerate every unit.
    owner = []                       # owner[u] = worker holding unit u
    for c, w in enumerate(workers):
        owner.extend([c] * (w["t1"] - w["t0"]))
    assert len(owner) == total

    covers = {b: [] for b in range(len(tiles))}  # row -> ordered workers holding its tiles
    for u, (b, j) in enumerate(units):
        if j >= 0 and (not covers[b] or covers[b][-1] != owner[u]):
            covers[b].append(owner[u])
    segments = []
    for c, w in enumerate(workers):
        rows = [b for b in range(len(tiles)) if c in covers[b]]
        if rows:
            w["first_row"], w["last_row"] = rows[0], rows[-1]
        for b in rows:
            f, n = first_tile[b], tiles[b]
            j0 = max(w["t0"], f) - f
            j1 = min(w["t1"], f + n) - f
            split = len(covers[b]) > 1
            slot = -1
            if split:
                slot = 2 * c if w["t0"] >= f else 2 * c + 1
            segments.append({"worker": c, "row": b, "tile_begin": j0, "tile_end": j1,
                             "split": split, "slot": slot})
    return {"grid": grid, "total_tiles": total, "row_start": start, "prefix": prefix,
            "workers": workers, "covers": covers, "segments": segments}


def token_segments(kv_indptr, grid: int) -> dict:
    """Row -> list of row-local token ranges, in the form ``mla_decode_split_ref`` takes."""
    sch = schedule(kv_indptr, grid)
    out = {}
    for s in sch["segments"]:
        b = s["row"]
        length = int(kv_indptr[b + 1]) - int(kv_indptr[b])
        out.setdefault(b, []).append((s["tile_begin"] * TILE_TOKENS,
                                      min(length, s["tile_end"] * TILE_TOKENS)))
    return out


def worker_table(kv_indptr, grid: int) -> np.ndarray:
    """int64 ``[grid, 4]``: (t0, t1, first_row, last_row) per worker."""
    sch = schedule(kv_indptr, grid)
    return np.array([[w["t0"], w["t1"], w["first_row"], w["last_row"]] for w in sch["workers"]],
                    dtype=np.int64).reshape(grid, 4)
