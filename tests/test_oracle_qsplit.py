"""Pins of the oracle's two-term e4m3 operands (``oracle.qsplit``).

What fixes them, independently of the oracle's own formulas:
  * the exponent rule by brute force: the unique integer k with
    224 < a * 2^k <= 448, searched over every k, for every finite positive bf16
    value a, and the clamp at +-126 where no k in range exists;
  * the codes against torch's own float8_e4m3fn cast (a library routine) on
    every finite bf16 value of a token at a fixed exponent, and on every half
    value in [0, 256] for P;
  * the closed form of the split: with x = v * 2^k2 carrying eight significant
    bits, x - hi is a multiple of 2^(E-7) no larger than 2^(E-4) (2^E <= |x|),
    so 16 (x - hi) is an e4m3 value whenever |x| >= 2^-6 and hi + lo / 16 == x
    exactly there; below, the error stays under 2^-14.
"""
import numpy as np
import pytest
import torch

from oracle.fp8 import e4m3fn_decode
from oracle.qsplit import (bf16_bits_to_f32, p_split_e4m3, q_operand_e4m3, q_operand_tokens,
                           q_scale_exponent, two_term_value)

FINITE_POS_BF16 = np.arange(0x0001, 0x7F80, dtype=np.uint16)  # every finite positive bf16


def torch_e4m3(x_f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_exponent_rule_brute_force_every_bf16():
    a = bf16_bits_to_f32(FINITE_POS_BF16).astype(np.float64)
    for val in a:
        k2 = q_scale_exponent(val)
        hits = [k for k in range(-126, 127) if 224.0 < val * 2.0 ** k <= 448.0]
        if hits:
            assert len(hits) == 1 and k2 == hits[0], (val, k2, hits)
        else:  # outside the range every k in [-126, 126] reaches: clamped
            assert k2 == (126 if val * 2.0 ** 126 <= 224.0 else -126), (val, k2)


@pytest.mark.parametrize("amax,k2,scaled", [
    (1.75, 8, 448.0),             # 0.875 * 2^1: the top of the window is included
    (1.7578125, 7, 225.0),        # the next bf16 above it drops one binade
    (1.0, 8, 256.0),
    (0.875, 9, 448.0),
    (448.0, 0, 448.0),
    (0.0, 0, 0.0),                # all-zero token: no scaling
    (2.0 ** -133, 126, 2.0 ** -7),  # smallest bf16 subnormal: clamped at 126
    (float.fromhex("0x1.fep127"), -120, 255.0),  # largest finite bf16
])
def test_exponent_rule_hand_examples(amax, k2, scaled):
    assert q_scale_exponent(amax) == k2
    assert amax * 2.0 ** k2 == scaled


def _token_with(values_bits: np.ndarray, amax_bits: int) -> np.ndarray:
    tok = np.zeros(16 * 576, dtype=np.uint16)
    tok[: values_bits.size] = values_bits
    tok[-1] = amax_bits
    return tok.reshape(16, 576)


def test_q_codes_match_torch_cast_on_every_bf16_below_amax():
    # amax 1.75 (bf16 0x3FE0) fixes k2 = 8; every finite bf16 of magnitude <= 1.75,
    # both signs, spread over as many tokens as it takes.
    mags = np.arange(0x0000, 0x3FE1, dtype=np.uint16)
    vals = np.concatenate([mags, mags | np.uint16(0x8000)])
    per = 16 * 576 - 1
    for i in range(0, vals.size, per):
        chunk = vals[i:i + per]
        tok = _token_with(chunk, 0x3FE0)
        hi, lo, k2 = q_operand_e4m3(tok)
        assert k2 == 8
        x = (bf16_bits_to_f32(tok) * np.float32(256.0)).astype(np.float32)
        assert np.array_equal(hi, torch_e4m3(x))
        r = ((torch.from_numpy(x) - torch.from_numpy(e4m3fn_decode(hi).astype(np.float32)))
             * 16.0).numpy()
        assert np.array_equal(lo, torch_e4m3(r))


@pytest.mark.parametrize("amax_bits", [0x3FE0, 0x3FE1, 0x0001, 0x7F7F, 0x3C00, 0x4380, 0x0080])
def test_q_split_closed_form(amax_bits):
    rng = np.random.default_rng(amax_bits)
    amax = float(bf16_bits_to_f32(np.uint16(amax_bits)))
    # random bf16 values of magnitude <= amax, both signs, plus the extremes
    mags = rng.integers(0, amax_bits + 1, 16 * 576 - 1).astype(np.uint16)
    signs = rng.integers(0, 2, mags.size).astype(np.uint16) << np.uint16(15)
    tok = _token_with(mags | signs, amax_bits)
    hi, lo, k2 = q_operand_e4m3(tok)
    v = bf16_bits_to_f32(tok).astype(np.float64)
    x = v * 2.0 ** k2
    got = two_term_value(hi, lo)
    big = np.abs(x) >= 2.0 ** -6
    assert np.array_equal(got[big], x[big])
    assert np.all(np.abs(got[~big] - x[~big]) <= 2.0 ** -14)
    if k2 not in (-126, 126):
        assert 224.0 < np.max(np.abs(x)) <= 448.0


def test_q_zero_and_signed_zero_tokens():
    tok = np.zeros((16, 576), dtype=np.uint16)
    tok[3, 7] = 0x8000  # -0
    hi, lo, k2 = q_operand_e4m3(tok)
    assert k2 == 0
    assert hi[3, 7] == 0x80 and lo[3, 7] == 0x00
    hi[3, 7] = 0
    assert not hi.any() and not lo.any()


def test_q_tokens_are_independent():
    rng = np.random.default_rng(5)
    q = (rng.standard_normal((3, 16, 576)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    q[1] = (q[1].astype(np.uint32) & 0x8000) | 0x0001  # a token of tiny values only
    hi, lo, k2 = q_operand_tokens(q)
    for t in range(3):
        h, l, k = q_operand_e4m3(q[t])
        assert np.array_equal(hi[t], h) and np.array_equal(lo[t], l) and k2[t] == k
    assert k2[1] == 126


def test_p_codes_match_torch_cast_on_every_half_in_range():
    bits = np.arange(0x0000, 0x5C01, dtype=np.uint16)  # every half in [0, 256]
    p16 = bits.view(np.float16)
    hi, lo = p_split_e4m3(p16.astype(np.float32))
    t16 = torch.from_numpy(p16.copy())
    assert np.array_equal(hi, t16.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    hb = torch.from_numpy(hi.copy()).view(torch.float8_e4m3fn).to(torch.float16)
    r = (t16 - hb) * 16.0
    assert r.dtype == torch.float16
    assert np.array_equal(lo, r.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    # closed form: eight significant bits kept (hi to four, the remainder to four more)
    got = two_term_value(hi, lo)
    p = p16.astype(np.float64)
    assert np.all(np.abs(got - p) <= 2.0 ** -8 * p + 2.0 ** -14)


def test_p_split_rounds_float_to_half_first():
    rng = np.random.default_rng(9)
    p = rng.uniform(0, 256, 100_000).astype(np.float32)
    p = np.concatenate([p, np.float32([0.0, 1.0, 256.0, 2.0 ** -20, 1.0 + 2.0 ** -12])])
    hi, lo = p_split_e4m3(p)
    hi16, lo16 = p_split_e4m3(p.astype(np.float16).astype(np.float32))
    assert np.array_equal(hi, hi16) and np.array_equal(lo, lo16)
    assert np.all(np.abs(two_term_value(hi, lo) - p) <= 2.0 ** -8 * p + 2.0 ** -11 * p + 2.0 ** -14)
