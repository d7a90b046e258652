"""OCP FP8 E4M3 ("fn" flavour) codec in plain NumPy, from the format's definition.

The pages quantise the latent cache and the query to an 8-bit float whose type
is platform-dependent (submission 738050, constant ``FP8_DTYPE`` and its
comment; ``FP8_MAX = torch.finfo(FP8_DTYPE).max``).  On AMD that is e4m3fnuz
with maximum 240 (submission 663509, "STATIC Q SCALE" note).  Reading taken for
this GPU: the fn flavour, whose ``finfo.max`` is 448.

E4M3fn: 1 sign bit s, 4 exponent bits e (bias 7), 3 mantissa bits m.
  e == 0            -> (-1)^s * (m / 8) * 2^-6           (zero and subnormals)
  0 < e, not NaN    -> (-1)^s * (1 + m / 8) * 2^(e - 7)
  e == 15 and m == 7 -> NaN (codes 0x7F and 0xFF); there is no infinity.
Largest finite magnitude: 0x7E = 1.75 * 2^8 = 448.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
MIN_NORMAL = 2.0 ** -6
SUBNORMAL_STEP = 2.0 ** -9


def e4m3fn_decode(codes) -> np.ndarray:
    """Exact float64 value of each e4m3fn code (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = c >> 7
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0,
                   (m / 8.0) * MIN_NORMAL,
                   (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e4m3fn_encode(x) -> np.ndarray:
    """Round float32 values to e4m3fn codes: nearest, ties to even, saturating.

    Magnitudes whose rounded value would exceed 448 become 448 (the pages clamp
    to ``[-finfo.max, finfo.max]`` before the cast: submission 722089,
    ``quantize_fp8``; submission 738050, ``_quantize_fp8``).  The sign of zero
    is kept.  NaN maps to 0x7F with its sign bit.
    """
    xf = np.asarray(x, dtype=np.float32).astype(np.float64)
    sign = np.signbit(xf).astype(np.int64)
    a = np.abs(xf)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    a = np.minimum(a, E4M3_MAX)  # clamp first: every clamped value rounds to 448

    # Grid spacing of the binade holding a: 2^(E-3) for normals, 2^-9 below 2^-6.
    _, ex = np.frexp(np.maximum(a, MIN_NORMAL))  # a = f * 2^ex, f in [0.5, 1)
    step = np.exp2((ex - 1 - 3).astype(np.float64))
    step = np.where(a < MIN_NORMAL, SUBNORMAL_STEP, step)
    v = np.rint(a / step) * step  # a/step is exact (power-of-two step); rint ties to even
    v = np.minimum(v, E4M3_MAX)

    # Encode the grid value v.
    _, vex = np.frexp(np.maximum(v, MIN_NORMAL))
    e_unb = vex - 1                                   # floor(log2 v) for normals
    normal = v >= MIN_NORMAL
    exp_field = np.where(normal, e_unb + 7, 0)
    mant = np.where(normal,
                    np.rint((v / np.exp2(e_unb.astype(np.float64)) - 1.0) * 8.0),
                    np.rint(v / SUBNORMAL_STEP))
    code = (sign << 7) | (exp_field.astype(np.int64) << 3) | mant.astype(np.int64)
    code = np.where(nan, (sign << 7) | 0x7F, code)
    return code.astype(np.uint8)
