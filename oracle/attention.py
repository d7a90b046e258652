"""Exact softmax attention for the MLA forward_absorb decode step, in float64.

What the step computes (submission 738050, the comment block above the
``mla_decode_fwd`` call in ``_run_a8w8``; constants block of submission 663509):

    O_i = softmax(Q_i K^T / sqrt(576)) V

per batch row i with one query token of 16 heads x 576 dims ("absorbed" Q);
K is all 576 dims of each cached latent row (512 kv_lora_rank + 64 rope) and
V is the first 512 dims of the same row.  There is one KV head shared by the 16
query heads, page size 1, and no logit soft-capping (``logit_cap=0.0``).

Cache rows hold e4m3fn codes with one float32 per-tensor scale; a row's value
is ``code * scale`` (submission 738050, ``_quantize_fp8`` docstring).  The query
is the exact bf16 value handed in.  The harness also hands over the bf16 copy
of the same cache (submission 738050, ``custom_kernel`` docstring), which
submission 722089 reads, with the unquantised bf16 query, whenever the batch
holds at most 131072 cached tokens (its AITER PATH section, ``_aiter_path``):
``mla_decode_ref_bf16kv`` is that variant, the cache rows' values being the
exact bf16 values.

Readings taken where the pages are silent:
  * a row with no cached tokens (``kv_len == 0``) yields all-zero output;
  * a row may hold n >= 1 query tokens (``qo_indptr[b+1] - qo_indptr[b] = n``;
    the pages pass ``max_seqlen_qo`` / ``uni_seqlen_qo`` but only ever run
    n = 1).  Multi-token decode (speculative / multi-token prediction) appends
    the n query tokens' own entries as the row's last n cached tokens, so query
    token i (0-based) attends to the first ``L - n + 1 + i`` cached tokens
    (causal, aligned to the end of the row); a token that sees no cached token
    yields zeros.  For n = 1 this is the plain decode step.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

from .fp8 import e4m3fn_decode

NUM_HEADS = 16
QK_HEAD_DIM = 576
V_HEAD_DIM = 512
SM_SCALE = 1.0 / math.sqrt(QK_HEAD_DIM)   # submission 663509 constants: 1 / sqrt(576)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def _row_tokens(b: int, kv_indptr, kv_indices) -> np.ndarray:
    j0, j1 = int(kv_indptr[b]), int(kv_indptr[b + 1])
    if j1 < j0:
        raise ValueError(f"kv_indptr decreases at row {b}")
    if kv_indices is None:
        return np.arange(j0, j1, dtype=np.int64)
    return np.asarray(kv_indices[j0:j1], dtype=np.int64)


def _query_rows(b: int, qo_indptr) -> tuple[int, int]:
    """(first query token, query token count n >= 1) of row b."""
    t0, t1 = int(qo_indptr[b]), int(qo_indptr[b + 1])
    if t1 - t0 < 1:
        raise ValueError(f"row {b} has {t1 - t0} query tokens")
    return t0, t1 - t0


def _query_row(b: int, qo_indptr) -> int:
    t0, n = _query_rows(b, qo_indptr)
    if n != 1:
        raise ValueError(f"row {b} has {n} query tokens; this function takes one")
    return t0


def visible_tokens(length: int, n: int, i: int) -> int:
    """Cached tokens query token i of an n-token row sees (causal, end-aligned)."""
    return max(0, length - n + 1 + i)


def dequant_rows(kv_codes: np.ndarray, kv_scale, slots: np.ndarray) -> np.ndarray:
    """float64 ``code * scale`` of the selected cache rows, shape ``[L, 576]``."""
    codes = np.asarray(kv_codes).reshape(-1, QK_HEAD_DIM)
    return e4m3fn_decode(codes[slots]) * float(np.float32(kv_scale))


def bf16_rows(kv_bits: np.ndarray, slots: np.ndarray) -> np.ndarray:
    """float64 values of the selected rows of a bf16 cache given as raw bits, ``[L, 576]``."""
    bits = np.asarray(kv_bits, dtype=np.uint16).reshape(-1, QK_HEAD_DIM)
    return bf16_bits_to_f64(bits[slots])


def row_attention(q_row: np.ndarray, k_rows: np.ndarray):
    """Softmax weights ``[16, L]`` and output ``[16, 512]`` for one row, float64."""
    z = (q_row @ k_rows.T) * SM_SCALE
    z = z - z.max(axis=1, keepdims=True)
    w = np.exp(z)
    w /= w.sum(axis=1, keepdims=True)
    return w, w @ k_rows[:, :V_HEAD_DIM]


def mla_decode_ref(q, kv_codes, kv_scale, qo_indptr, kv_indptr,
                   kv_indices: Optional[np.ndarray] = None, rows=None) -> np.ndarray:
    """float64 output ``[T, 16, 512]`` of the decode step.

    ``q`` is float64-convertible ``[T, 16, 576]`` (exact bf16 values);
    ``kv_codes`` uint8 ``[N, 576]`` (or ``[N, 1, 576]``); ``kv_scale`` the float32
    per-tensor scale; ``kv_indices`` maps flattened token j to cache slot
    ``kv_indices[j]`` (identity when None).  Query token ``qo_indptr[b] + i`` of
    an n-token row sees the row's first ``visible_tokens(L, n, i)`` cached tokens.
    ``rows`` restricts the work to a subset of batch rows; the other output rows
    are left as NaN.
    """
    return _decode(q, qo_indptr, kv_indptr, kv_indices, rows,
                   lambda slots: dequant_rows(kv_codes, kv_scale, slots))


def mla_decode_ref_bf16kv(q, kv_bits, qo_indptr, kv_indptr,
                          kv_indices: Optional[np.ndarray] = None, rows=None) -> np.ndarray:
    """float64 output ``[T, 16, 512]`` of the decode step over a bf16 cache.

    As ``mla_decode_ref`` with ``kv_bits`` the uint16 bit patterns ``[N, 576]``
    (or ``[N, 1, 576]``) of the bf16 cache; K and V are their exact values.
    """
    return _decode(q, qo_indptr, kv_indptr, kv_indices, rows,
                   lambda slots: bf16_rows(kv_bits, slots))


def _decode(q, qo_indptr, kv_indptr, kv_indices, rows, row_values) -> np.ndarray:
    """The decode step given ``row_values(slots)``: float64 ``[L, 576]`` cache rows."""
    q = np.asarray(q, dtype=np.float64)
    batch = len(qo_indptr) - 1
    out = np.full((q.shape[0], NUM_HEADS, V_HEAD_DIM), np.nan)
    for b in (range(batch) if rows is None else rows):
        t0, n = _query_rows(b, qo_indptr)
        slots = _row_tokens(b, kv_indptr, kv_indices)
        k_rows = row_values(slots)
        for i in range(n):
            vis = visible_tokens(slots.size, n, i)
            if vis == 0:
                out[t0 + i] = 0.0
                continue
            _, out[t0 + i] = row_attention(q[t0 + i], k_rows[:vis])
    return out


def mla_decode_weights(q, kv_codes, kv_scale, qo_indptr, kv_indptr, b: int,
                       kv_indices: Optional[np.ndarray] = None) -> np.ndarray:
    """Softmax weights ``[16, L_b]`` of row ``b`` (used by the invariant checks)."""
    q = np.asarray(q, dtype=np.float64)
    t = _query_row(b, qo_indptr)
    slots = _row_tokens(b, kv_indptr, kv_indices)
    w, _ = row_attention(q[t], dequant_rows(kv_codes, kv_scale, slots))
    return w


# --------------------------------------------------------------------------
# Split-KV partials and their log-sum-exp combine (flash-decoding).
#
# Submission 722089, ``_mla_multihead_stage1``: each split keeps a running max
# and sum in base 2 (scores pre-multiplied by sm_scale * log2 e), stores its
# normalised partial ``acc / l`` and ``lse = m + log2 l``; an empty split stores
# a zero partial and lse = -inf.  ``_mla_reduce``: M = max_s lse_s,
# w_s = 2^(lse_s - M), out = sum_s w_s * partial_s / sum_s w_s.
# --------------------------------------------------------------------------
LOG2E = 1.0 / math.log(2.0)


def split_partial(q_row: np.ndarray, k_rows: np.ndarray):
    """(normalised partial [16, 512], lse [16] in base 2) over one token range."""
    if k_rows.shape[0] == 0:
        return np.zeros((NUM_HEADS, V_HEAD_DIM)), np.full(NUM_HEADS, -np.inf)
    s = (q_row @ k_rows.T) * (SM_SCALE * LOG2E)
    m = s.max(axis=1)
    p = np.exp2(s - m[:, None])
    l = p.sum(axis=1)
    return (p @ k_rows[:, :V_HEAD_DIM]) / l[:, None], m + np.log2(l)


def combine_partials(partials, lses) -> np.ndarray:
    """Log-sum-exp weighted combine of split partials, float64 ``[16, 512]``."""
    lses = np.asarray(lses, dtype=np.float64)          # [S, 16]
    partials = np.asarray(partials, dtype=np.float64)  # [S, 16, 512]
    top = lses.max(axis=0)
    if np.all(np.isneginf(top)):
        return np.zeros((NUM_HEADS, V_HEAD_DIM))
    w = np.exp2(lses - top[None, :])
    return (w[:, :, None] * partials).sum(axis=0) / w.sum(axis=0)[:, None]


def mla_decode_split_ref(q, kv_codes, kv_scale, qo_indptr, kv_indptr, segments,
                         kv_indices: Optional[np.ndarray] = None) -> np.ndarray:
    """Decode output computed split by split and combined.

    ``segments`` maps batch row b to a list of token ranges ``(j0, j1)`` (row-local
    token offsets) that partition ``[0, L_b)``; any partition gives the same
    result as ``mla_decode_ref`` up to rounding.  With n query tokens per row,
    each split is cut to the tokens the query token sees (an empty cut gives a
    zero partial with lse -inf).
    """
    q = np.asarray(q, dtype=np.float64)
    batch = len(qo_indptr) - 1
    out = np.zeros((q.shape[0], NUM_HEADS, V_HEAD_DIM))
    for b in range(batch):
        t0, n = _query_rows(b, qo_indptr)
        slots = _row_tokens(b, kv_indptr, kv_indices)
        k_rows = dequant_rows(kv_codes, kv_scale, slots)
        for i in range(n):
            vis = visible_tokens(slots.size, n, i)
            parts, lses = [], []
            for (j0, j1) in segments.get(b, [(0, slots.size)]):
                o, lse = split_partial(q[t0 + i], k_rows[j0:min(j1, vis)] if j0 < vis else k_rows[:0])
                parts.append(o)
                lses.append(lse)
            out[t0 + i] = combine_partials(parts, lses) if parts else 0.0
    return out
