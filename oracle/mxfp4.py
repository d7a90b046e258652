"""MXFP4 latent cache: E2M1 elements with one E8M0 scale per 32, in plain NumPy.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The harness also hands a submission the cache in MXFP4 (submission 738050,
``custom_kernel`` docstring: ``kv_data["mxfp4"] = (fp4_data, scale)``).
Submission 738050's ``_dequantize_mxfp4_inplace`` docstring fixes the format:
blocks of 32 consecutive elements of a row share one E8M0 scale (an 8-bit
power-of-two exponent, no mantissa); each element is a 4-bit E2M1 float (sign,
2 exponent bits, 1 mantissa bit); two elements are packed per byte, so a row of
576 values is 288 bytes of elements plus 18 scale bytes, and a value is the
element times its block's scale.  Submission 722089 (``_custom_multihead_path``
and ``_mla_multihead_stage1``) reads the same two arrays: elements
``[total_kv, 288]`` uint8 and scales ``[total_kv, >= 18]`` uint8.

Readings taken where the pages are silent (the formats come from the OCP
Microscaling Formats specification v1.0, which the pages' library implements):
  * E2M1: exponent bias 1; e == 0 gives (-1)^s * m * 0.5 (zero and the one
    subnormal 0.5); e > 0 gives (-1)^s * (1 + m / 2) * 2^(e - 1).  No inf/NaN;
    largest magnitude 6.
  * E8M0: value 2^(b - 127); b == 255 is NaN.
  * Packing: element 2i in the low nibble of byte i, element 2i + 1 in the high
    nibble.
  * Quantisation (the pages take the cache as given; this is how the synthetic
    cache is made): per block, shared exponent floor(log2 max|x|) - 2 (2 = the
    largest E2M1 exponent), clamped to [-127, 127] (an all-zero block takes
    -127); each element is x / 2^shared rounded to the nearest E2M1 value,
    ties to the even code, magnitudes above 6 saturating to 6, the sign of zero
    kept.
  * K is the dequantised row (576 values) and V its first 512 values, exactly
    as for the e4m3 cache (submission 738050 dequantises MXFP4 to the bf16
    layout and runs the same attention; submission 722089 reads V from the bf16
    copy of the cache instead, a harness convenience, not a different method).
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from .attention import QK_HEAD_DIM, _decode

BLOCK = 32
SCALES_PER_ROW = QK_HEAD_DIM // BLOCK      # 18
ROW_BYTES = QK_HEAD_DIM // 2               # 288
E2M1_MAX = 6.0
E2M1_EMAX = 2                              # exponent of the largest normal, 4 = 2^2


def e2m1_decode(codes) -> np.ndarray:
    """Exact float64 value of each 4-bit E2M1 code (0..15)."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    s = c >> 3
    e = (c >> 1) & 0x3
    m = c & 0x1
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2((e - 1).astype(np.float64)))
    return np.where(s == 1, -mag, mag)


def e8m0_decode(b) -> np.ndarray:
    """float64 2^(b - 127) for each scale byte (NaN for 0xFF)."""
    v = np.asarray(b, dtype=np.uint8).astype(np.int64)
    return np.where(v == 255, np.nan, np.exp2((v - 127).astype(np.float64)))


# The eight non-negative E2M1 magnitudes, by code.
_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_encode(y) -> np.ndarray:
    """Nearest E2M1 code of each value (ties to the even code, saturating at 6).

    Works from the eight magnitudes: the nearest one wins; of two equally near,
    the one with an even code (mantissa bit 0) wins.  Magnitudes beyond 6 give 6.
    The sign bit follows the input's sign (so -0 keeps it).
    """
    yv = np.asarray(y, dtype=np.float64)
    sign = np.signbit(yv).astype(np.int64)
    a = np.minimum(np.abs(yv), E2M1_MAX)
    d = np.abs(a[..., None] - _GRID)                  # distance to every magnitude
    best = d.min(axis=-1, keepdims=True)
    near = d == best                                  # one or two codes
    even = near & (np.arange(8) % 2 == 0)
    code = np.where(even.any(axis=-1), even.argmax(axis=-1), near.argmax(axis=-1))
    return ((sign << 3) | code).astype(np.uint8)


def shared_exponent(block_amax) -> np.ndarray:
    """floor(log2 amax) - 2 clamped to [-127, 127]; amax == 0 gives -127."""
    a = np.asarray(block_amax, dtype=np.float64)
    safe = np.where(a > 0, a, 1.0)
    _, ex = np.frexp(safe)                             # safe = f * 2^ex, f in [0.5, 1)
    e = np.where(a > 0, (ex - 1) - E2M1_EMAX, -127)
    return np.clip(e, -127, 127).astype(np.int64)


def quantize_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """MXFP4 of rows ``x [N, 576]`` (float64-convertible, finite).

    Returns (elements uint8 ``[N, 288]``, scales uint8 ``[N, 18]``).
    """
    xv = np.asarray(x, dtype=np.float64).reshape(-1, SCALES_PER_ROW, BLOCK)
    amax = np.abs(xv).max(axis=-1)                     # [N, 18]
    e = shared_exponent(amax)
    y = xv / np.exp2(e.astype(np.float64))[..., None]  # exact: a power of two
    codes = e2m1_encode(y).reshape(xv.shape[0], QK_HEAD_DIM)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, (e + 127).astype(np.uint8)


def unpack_codes(packed) -> np.ndarray:
    """E2M1 codes ``[N, 576]`` of packed element bytes ``[N, 288]``."""
    p = np.asarray(packed, dtype=np.uint8).reshape(-1, ROW_BYTES)
    codes = np.empty((p.shape[0], QK_HEAD_DIM), dtype=np.uint8)
    codes[:, 0::2] = p & 0xF
    codes[:, 1::2] = p >> 4
    return codes


def dequant_rows(kv_fp4, kv_scales, slots) -> np.ndarray:
    """float64 values ``[L, 576]`` of the selected MXFP4 cache rows."""
    p = np.asarray(kv_fp4, dtype=np.uint8).reshape(-1, ROW_BYTES)[slots]
    s = np.asarray(kv_scales, dtype=np.uint8).reshape(-1, SCALES_PER_ROW)[slots]
    vals = e2m1_decode(unpack_codes(p)).reshape(-1, SCALES_PER_ROW, BLOCK)
    return (vals * e8m0_decode(s)[..., None]).reshape(-1, QK_HEAD_DIM)


def mla_decode_ref_mxfp4(q, kv_fp4, kv_scales, qo_indptr, kv_indptr,
                         kv_indices: Optional[np.ndarray] = None, rows=None) -> np.ndarray:
    """float64 output ``[T, 16, 512]`` of the decode step over an MXFP4 cache.

    As ``attention.mla_decode_ref`` with the cache given as packed elements
    ``[N, 288]`` and scales ``[N, 18]``; K and V are the rows' exact values.
    """
    return _decode(q, qo_indptr, kv_indptr, kv_indices, rows,
                   lambda slots: dequant_rows(kv_fp4, kv_scales, slots))
