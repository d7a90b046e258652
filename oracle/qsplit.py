"""The two-term e4m3 operands of the e4m3-cache step: Q per query token, and P.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages feed the tensor cores FP8 operands: submission 722089's
``_mla_multihead_stage1`` casts each query chunk to ``float8e4nv`` before its
dot with the cache, and rounds the probabilities P to bf16 before the dot with
V; submission 663509 (its "STATIC Q SCALE" note) and submission 738050
(``_run_a8w8``, ``_quantize_fp8``) quantise Q with a per-tensor scale.  None of
them fixes the arithmetic for this GPU.  Reading taken here, for the e4m3 cache
(it is this library's choice, stated so that it can be checked bit for bit):

Query operand, per query token (16 heads x 576 dims of bf16 values v):
  a   = max |v| over the token's 9216 values;
  k2  = the integer k with 224 < a * 2^k <= 448, clamped to [-126, 126]
        (k2 = 0 when a = 0): the token is scaled by a power of two so that its
        largest magnitude lands in the top binade of e4m3 below the maximum;
  x   = float32(v * 2^k2);
  hi  = e4m3fn(x),   lo = e4m3fn(float32(16 * float32(x - hi)))
        (round to nearest even, saturating at 448);
  x ~= hi + lo / 16 with about eight significant bits, i.e. the bf16 query's
  own precision, and the dot products are rescaled by 2^-k2 afterwards.

Probability operand, per probability p (0 <= p <= 256 in the kernel's
exponent units): the pages' P is a bf16 value (eight significant bits); here
  p16 = float16(p),  hi = e4m3fn(p16),
  lo  = e4m3fn(float16(16 * float16(p16 - hi)))
(every step in IEEE half precision, rounded to nearest even), so that
p16 ~= hi + lo / 16 to about eight significant bits.

Both definitions are written as the steps above in NumPy float32 / float16,
whose arithmetic is IEEE round-to-nearest-even, on top of ``oracle.fp8``.
"""
from __future__ import annotations

import numpy as np

from .fp8 import e4m3fn_decode, e4m3fn_encode

SCALED_AMAX_LO = 224.0   # exclusive
SCALED_AMAX_HI = 448.0   # inclusive
K2_LIMIT = 126


def q_scale_exponent(amax: float) -> int:
    """k2 for a token whose largest magnitude is ``amax`` (a finite value >= 0).

    frexp writes amax = f * 2^e with f in [0.5, 1): f * 2^9 lies in [256, 448]
    when f <= 0.875 and f * 2^8 in (224, 256) otherwise.
    """
    a = float(amax)
    if a == 0.0:
        return 0
    f, e = np.frexp(a)
    k2 = 9 - int(e) if f <= 0.875 else 8 - int(e)
    return max(-K2_LIMIT, min(K2_LIMIT, k2))


def bf16_bits_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def q_operand_e4m3(q_token_bits):
    """(hi, lo, k2) of one query token: bf16 bits [16, 576] -> uint8 codes [16, 576] twice."""
    v = bf16_bits_to_f32(q_token_bits)
    a = float(np.max(np.abs(v.astype(np.float64)))) if v.size else 0.0
    k2 = q_scale_exponent(a)
    up = np.float32(2.0 ** k2)
    x = (v * up).astype(np.float32)                        # float32 product, round to nearest even
    hi = e4m3fn_encode(x)
    hv = e4m3fn_decode(hi).astype(np.float32)              # exact
    d = (x - hv).astype(np.float32)
    r = (d * np.float32(16.0)).astype(np.float32)
    lo = e4m3fn_encode(r)
    return hi, lo, k2


def q_operand_tokens(q_bits):
    """Every token of q bits [T, 16, 576]: (hi [T,16,576], lo [T,16,576], k2 [T])."""
    q = np.asarray(q_bits, dtype=np.uint16).reshape(-1, 16, 576)
    hi = np.empty(q.shape, dtype=np.uint8)
    lo = np.empty(q.shape, dtype=np.uint8)
    k2 = np.empty(q.shape[0], dtype=np.int64)
    for t in range(q.shape[0]):
        hi[t], lo[t], k2[t] = q_operand_e4m3(q[t])
    return hi, lo, k2


def p_split_e4m3(p_f32):
    """(hi, lo) e4m3 codes of float32 probabilities through the half-precision steps."""
    p16 = np.asarray(p_f32, dtype=np.float32).astype(np.float16)   # float -> half, nearest even
    hi = e4m3fn_encode(p16.astype(np.float32))
    hb = e4m3fn_decode(hi).astype(np.float16)                       # exact
    d = (p16 - hb).astype(np.float16)
    r = (d * np.float16(16.0)).astype(np.float16)
    lo = e4m3fn_encode(r.astype(np.float32))
    return hi, lo


def two_term_value(hi, lo) -> np.ndarray:
    """hi + lo / 16 in float64 (exact)."""
    return e4m3fn_decode(hi) + e4m3fn_decode(lo) / 16.0
