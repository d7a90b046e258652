"""Pins of the oracle's e4m3fn codec against the format definition and torch's cast."""
import numpy as np
import pytest
import torch

from oracle.fp8 import E4M3_MAX, e4m3fn_decode, e4m3fn_encode

from .golden_util import load_table

ALL_CODES = np.arange(256, dtype=np.uint8)


def torch_decode(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_encode(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(x, dtype=np.float32).copy()).clamp(-E4M3_MAX, E4M3_MAX)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_matches_torch_for_all_codes():
    ours, ref = e4m3fn_decode(ALL_CODES), torch_decode(ALL_CODES)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    finite = ~np.isnan(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.signbit(ours[finite]), np.signbit(ref[finite]))


def test_decode_golden_points():
    # Values fixed by the E4M3 definition (bias 7, 3 mantissa bits, 0x7F NaN).
    for code, value in load_table("e4m3fn_points.txt"):
        got = e4m3fn_decode(np.array([int(code, 16)], dtype=np.uint8))[0]
        if value == "nan":
            assert np.isnan(got)
        else:
            assert got == float.fromhex(value), (code, got)


def test_nan_codes_only():
    nan = np.isnan(e4m3fn_decode(ALL_CODES))
    assert sorted(np.nonzero(nan)[0].tolist()) == [0x7F, 0xFF]
    assert np.nanmax(np.abs(e4m3fn_decode(ALL_CODES))) == 448.0


def test_encode_matches_torch_on_every_bf16():
    bits = np.arange(65536, dtype=np.uint32) << np.uint32(16)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    assert np.array_equal(e4m3fn_encode(x), torch_encode(x))


@pytest.mark.parametrize("seed", [0, 1])
def test_encode_matches_torch_on_random_f32(seed):
    rng = np.random.default_rng(seed)
    n = 1_000_000
    mant = rng.uniform(-1, 1, n).astype(np.float32)
    expo = rng.integers(-14, 11, n).astype(np.float32)
    x = (mant * np.exp2(expo)).astype(np.float32)
    # exact ties between adjacent e4m3 values (mid-points) in every binade
    grid = e4m3fn_decode(ALL_CODES[:0x7F]).astype(np.float32)
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids, grid, -grid, np.float32([0.0, -0.0, 448.0, 464.0, 1e9])])
    assert np.array_equal(e4m3fn_encode(x), torch_encode(x))


def test_round_trip_and_monotone():
    finite = ALL_CODES[~np.isnan(e4m3fn_decode(ALL_CODES))]
    assert np.array_equal(e4m3fn_encode(e4m3fn_decode(finite).astype(np.float32)), finite)
    xs = np.sort(np.random.default_rng(3).uniform(-500, 500, 200_000).astype(np.float32))
    vals = e4m3fn_decode(e4m3fn_encode(xs))
    assert np.all(np.diff(vals) >= 0)


def test_saturation_and_signed_zero():
    codes = e4m3fn_encode(np.float32([449.0, 1e30, -1e30, -0.0, 2.0 ** -11]))
    assert codes.tolist() == [0x7E, 0x7E, 0xFE, 0x80, 0x00]
