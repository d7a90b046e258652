"""Pins of the oracle's per-tensor FP8 quantiser."""
import numpy as np
import torch

from oracle.fp8 import e4m3fn_decode
from oracle.quant import encode_with_scale, per_tensor_scale, quantize_per_tensor
from mla_decode_attention_08_gb300.inputs import bf16_bits_to_f32, normal_bf16_rows


def torch_quantize(x: np.ndarray):
    """The same recipe written with torch float32 ops and torch's fp8 cast."""
    t = torch.from_numpy(x.astype(np.float32))
    amax = t.abs().amax().clamp(min=1e-12)
    scale = amax / 448.0
    codes = (t / scale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.numpy(), np.float32(scale.item())


def test_matches_torch_float32_recipe():
    x = bf16_bits_to_f32(normal_bf16_rows(11, 3000))
    codes, scale = quantize_per_tensor(x)
    tcodes, tscale = torch_quantize(x)
    assert scale == tscale
    assert np.array_equal(codes, tcodes)


def test_absmax_element_maps_to_448_and_error_bound():
    x = bf16_bits_to_f32(normal_bf16_rows(12, 500))
    codes, scale = quantize_per_tensor(x)
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert abs(e4m3fn_decode(codes[i])) == 448.0
    # e4m3 keeps 4 significant bits: relative error <= 2^-4 for normals,
    # absolute error <= 2^-10 * scale in the subnormal range.
    deq = e4m3fn_decode(codes) * float(scale)
    err = np.abs(deq - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * float(scale)) * (1 + 1e-6)
    assert np.all(err <= bound)


def test_power_of_two_amax_is_exact():
    # amax = 448 * 2^-3 -> scale = 2^-3 exactly; values on the e4m3 grid times the
    # scale quantise without error.
    grid = e4m3fn_decode(np.arange(0x7F, dtype=np.uint8))
    x = (np.concatenate([grid, -grid]) * 0.125).astype(np.float32)
    codes, scale = quantize_per_tensor(x)
    assert scale == np.float32(0.125)
    assert np.array_equal(e4m3fn_decode(codes) * 0.125, x.astype(np.float64))


def test_all_zero_uses_floor():
    codes, scale = quantize_per_tensor(np.zeros((4, 576), np.float32))
    assert scale == np.float32(np.float32(1e-12) / np.float32(448.0))
    assert not codes.any()


def test_chunked_amax_equals_global():
    x = bf16_bits_to_f32(normal_bf16_rows(13, 70_000))
    assert per_tensor_scale(x, chunk_rows=4096) == per_tensor_scale(x, chunk_rows=1 << 20)
    s = per_tensor_scale(x)
    assert np.array_equal(encode_with_scale(x[5:9], s), quantize_per_tensor(x)[0][5:9])
