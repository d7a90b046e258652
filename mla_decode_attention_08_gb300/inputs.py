"""Seeded synthetic inputs for the MLA forward_absorb decode step.

This module is shared by the float64 oracle (under ``oracle/``), the CUDA
path's tests and ``bench.py``.  It holds no attention, quantisation or
scheduling arithmetic: it only draws random numbers and rounds them to bf16,
which is how the pages' harness hands ``q`` and the bf16 latent cache to a
submission (kernelbot-amd-mixed-mla submission 738050, ``custom_kernel``
docstring: ``q`` is ``(total_q, 16, 576)`` bf16 and ``kv_data["bf16"]`` is
``(total_kv, 1, 576)`` bf16, with the fp8 copy derived from it).

Recipe (every stream is NumPy ``PCG64`` seeded from a ``SeedSequence``):

* ``q``: ``standard_normal`` float32 of shape ``[B, 16, 576]`` from
  ``SeedSequence([seed, 0])``, rounded to bf16 (round to nearest even).
* ragged lengths (ragged workloads only): ``integers(1, max_len, endpoint=True)``
  for each of the ``B`` rows, from ``SeedSequence([seed, 2])``.
* latent cache source ``kv_src``: ``standard_normal`` float32 of shape
  ``[N, 576]``, drawn in chunks of ``KV_CHUNK_ROWS`` rows; chunk ``k`` comes
  from ``SeedSequence([seed, 1, k])`` so that the values do not depend on how
  many threads fill them.  Rounded to bf16.
* page table (paged workloads only): ``permutation(N)`` from
  ``SeedSequence([seed, 3])``; token ``j`` of the flattened batch lives in cache
  slot ``kv_indices[j]`` (page size 1).

``qo_indptr = arange(B + 1)`` (one query token per row) and
``kv_indptr = [0, cumsum(lengths)]``, both int32, as in the pages' benchmark
(submission 663509, ``_precompute_metadata``: the indptr tensors are
``arange(0, bs + 1) * seqlen``).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

NUM_HEADS = 16
QK_HEAD_DIM = 576
V_HEAD_DIM = 512
BASE_SEED = 20261202
KV_CHUNK_ROWS = 16384


@dataclass(frozen=True)
class Workload:
    """One benchmark shape: ``batch`` rows of ``qo_len`` query tokens each."""

    name: str
    batch: int
    kv_len: int                # uniform length, or the maximum when ``ragged``
    ragged: bool = False       # lengths ~ U{1..kv_len}
    paged: bool = False        # cache rows addressed through a permuted page table
    seed: int = BASE_SEED
    qo_len: int = 1            # query tokens per row (2: two-token decode)

    @property
    def max_kv_len(self) -> int:
        return self.kv_len


WORKLOADS = {
    w.name: w
    for w in (
        Workload("bs4_kv1024", 4, 1024, seed=BASE_SEED + 0),
        Workload("bs32_kv1024", 32, 1024, seed=BASE_SEED + 1),
        Workload("bs64_kv8192", 64, 8192, seed=BASE_SEED + 2),
        Workload("bs256_kv8192", 256, 8192, seed=BASE_SEED + 3),
        Workload("ragged_bs128_kv8192_paged", 128, 8192, ragged=True, paged=True,
                 seed=BASE_SEED + 4),
        # Two and four query tokens per row (speculative / multi-token-prediction decode).
        Workload("bs64_q2_kv8192", 64, 8192, seed=BASE_SEED + 5, qo_len=2),
        Workload("bs64_q4_kv8192", 64, 8192, seed=BASE_SEED + 6, qo_len=4),
    )
}

# The workload the headline number is quoted on (largest single-GPU shape).
HEADLINE = "bs256_kv8192"


@dataclass
class Inputs:
    """Host arrays for one decode call; bf16 values are kept as raw uint16 bits."""

    q_bits: np.ndarray              # uint16 [B * qo_len, 16, 576]
    kv_bits: np.ndarray             # uint16 [N, 576]   (bf16 source of the latent cache)
    qo_indptr: np.ndarray           # int32 [B + 1]
    kv_indptr: np.ndarray           # int32 [B + 1]
    kv_indices: Optional[np.ndarray]  # int32 [kv_indptr[-1]] or None (identity)
    max_kv_len: int
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.qo_indptr.shape[0] - 1)

    @property
    def qo_len(self) -> int:
        return int(self.meta.get("qo_len", 1))

    @property
    def lengths(self) -> np.ndarray:
        return np.diff(self.kv_indptr.astype(np.int64))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def normal_bf16_rows(seed: int, rows: int, cols: int = QK_HEAD_DIM,
                     row_start: int = 0, row_stop: Optional[int] = None) -> np.ndarray:
    """Rows ``[row_start, row_stop)`` of the chunked N(0,1) bf16 cache source.

    Only the chunks that intersect the requested rows are drawn, so a caller can
    regenerate a few cache rows of a multi-GB workload cheaply.
    """
    if row_stop is None:
        row_stop = rows
    out = np.empty((row_stop - row_start, cols), dtype=np.uint16)
    if row_stop <= row_start:
        return out
    first, last = row_start // KV_CHUNK_ROWS, (row_stop - 1) // KV_CHUNK_ROWS

    def fill(k: int) -> None:
        c0 = k * KV_CHUNK_ROWS
        c1 = min(rows, c0 + KV_CHUNK_ROWS)
        vals = np.empty((c1 - c0, cols), dtype=np.float32)
        _rng(seed, 1, k).standard_normal(out=vals, dtype=np.float32)
        lo, hi = max(c0, row_start), min(c1, row_stop)
        out[lo - row_start:hi - row_start] = f32_to_bf16_bits(vals[lo - c0:hi - c0])

    chunks = range(first, last + 1)
    if len(chunks) == 1:
        fill(first)
    else:
        with ThreadPoolExecutor(min(_threads(), len(chunks))) as ex:
            list(ex.map(fill, chunks))
    return out


def make_from_lengths(lengths, seed: int, *, paged: bool = False,
                      max_kv_len: Optional[int] = None, qo_len: int = 1) -> Inputs:
    """Inputs for arbitrary per-row cache lengths (zero allowed) and
    ``qo_len`` query tokens per row (``qo_indptr = qo_len * arange``)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    batch = int(lengths.shape[0])
    q = np.empty((batch * qo_len, NUM_HEADS, QK_HEAD_DIM), dtype=np.float32)
    _rng(seed, 0).standard_normal(out=q, dtype=np.float32)
    kv_indptr = np.zeros(batch + 1, dtype=np.int64)
    np.cumsum(lengths, out=kv_indptr[1:])
    total = int(kv_indptr[-1])
    if total >= 2**31:
        raise ValueError("total cache tokens must fit in int32")
    kv_bits = normal_bf16_rows(seed, total)
    kv_indices = None
    if paged:
        kv_indices = _rng(seed, 3).permutation(total).astype(np.int32)
    return Inputs(
        q_bits=f32_to_bf16_bits(q),
        kv_bits=kv_bits,
        qo_indptr=(qo_len * np.arange(batch + 1)).astype(np.int32),
        kv_indptr=kv_indptr.astype(np.int32),
        kv_indices=kv_indices,
        max_kv_len=int(max_kv_len if max_kv_len is not None else max(1, int(lengths.max(initial=0)))),
        meta={"seed": seed, "paged": paged, "qo_len": qo_len},
    )


def workload_lengths(w: Workload) -> np.ndarray:
    if w.ragged:
        return _rng(w.seed, 2).integers(1, w.kv_len, size=w.batch, endpoint=True).astype(np.int64)
    return np.full(w.batch, w.kv_len, dtype=np.int64)


def workload_query_bits(w) -> np.ndarray:
    """The query of a named workload alone (the same draw as ``make_inputs``,
    without generating its cache): uint16 bf16 bits ``[B * qo_len, 16, 576]``."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    q = np.empty((w.batch * w.qo_len, NUM_HEADS, QK_HEAD_DIM), dtype=np.float32)
    _rng(w.seed, 0).standard_normal(out=q, dtype=np.float32)
    return f32_to_bf16_bits(q)


def make_inputs(w) -> Inputs:
    """Inputs of a named workload (see ``WORKLOADS``)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    inp = make_from_lengths(workload_lengths(w), w.seed, paged=w.paged, max_kv_len=w.max_kv_len,
                            qo_len=w.qo_len)
    inp.meta["workload"] = w.name
    return inp
