"""Per-tensor absmax FP8 quantisation of the bf16 latent cache (input preparation).

The harness hands a submission the cache already quantised, ``kv_data["fp8"] =
(kv_fp8, kv_scale)`` with a float32 ``(1,)`` scale and dequantisation
``x ~= code * scale`` (submission 738050, ``custom_kernel`` docstring and
``_quantize_fp8`` docstring).  The pages' own per-tensor quantiser (submission
722089, ``quantize_fp8``; submission 738050, ``_quantize_fp8``) is:

    amax  = max |x|, clamped below at 1e-12
    scale = amax / finfo(fp8).max
    code  = fp8( clamp(x / scale, -max, max) )

Reading taken where the pages leave the precision open: every step is done in
IEEE float32 (the bf16 inputs widen to float32 exactly; the two divisions are
float32 divisions rounded to nearest even), then e4m3fn rounding to nearest
even.  The pages' torch code divides in the tensor's own dtype; a bf16
intermediate would round twice, which is not a reproducible definition.
"""
from __future__ import annotations

import numpy as np

from .fp8 import E4M3_MAX, e4m3fn_encode

AMAX_FLOOR = np.float32(1e-12)


def per_tensor_scale(x_f32: np.ndarray, chunk_rows: int = 1 << 16) -> np.float32:
    """float32 scale = max(max|x|, 1e-12) / 448, the division rounded in float32."""
    x = np.asarray(x_f32)
    amax = np.float32(0.0)
    flat = x.reshape(x.shape[0], -1) if x.ndim > 1 else x.reshape(-1, 1)
    for r0 in range(0, flat.shape[0], chunk_rows):
        part = np.abs(flat[r0:r0 + chunk_rows].astype(np.float32, copy=False))
        if part.size:
            amax = max(amax, np.float32(part.max()))
    amax = max(np.float32(amax), AMAX_FLOOR)
    return np.float32(np.float32(amax) / np.float32(E4M3_MAX))


def encode_with_scale(x_f32: np.ndarray, scale: np.float32) -> np.ndarray:
    """e4m3fn codes of ``clamp(x / scale, -448, 448)`` with a float32 division."""
    y = np.asarray(x_f32, dtype=np.float32) / np.float32(scale)  # float32 / float32 -> RN float32
    y = np.clip(y, np.float32(-E4M3_MAX), np.float32(E4M3_MAX))
    return e4m3fn_encode(y)


def quantize_per_tensor(x_f32: np.ndarray):
    """(codes uint8, scale float32) for a whole tensor."""
    scale = per_tensor_scale(x_f32)
    return encode_with_scale(x_f32, scale), scale
