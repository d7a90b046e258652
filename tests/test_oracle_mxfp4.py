"""Pins of the oracle's MXFP4 codec, quantiser and decode step.

Each check leans on something other than the oracle's own code: the E2M1 value
table of the OCP Microscaling specification, torch's E8M0 type, a second
rounding algorithm, brute force on small blocks, exactly representable data
and the already pinned e4m3 decode step.
"""
import math

import numpy as np
import torch

from oracle.attention import mla_decode_ref, SM_SCALE
from oracle.fp8 import e4m3fn_decode, e4m3fn_encode
from oracle.mxfp4 import (dequant_rows, e2m1_decode, e2m1_encode, e8m0_decode,
                          mla_decode_ref_mxfp4, quantize_rows, shared_exponent, unpack_codes)
from mla_decode_attention_08_gb300.inputs import bf16_bits_to_f32, normal_bf16_rows

# OCP MX v1.0, FP4 E2M1 value table: codes 0..7 (positive), 8..15 the negatives.
SPEC_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_matches_spec_table():
    vals = e2m1_decode(np.arange(16))
    assert list(vals[:8]) == SPEC_E2M1
    assert list(vals[8:]) == [-v for v in SPEC_E2M1]
    assert np.signbit(vals[8])  # code 8 is -0


def test_e8m0_decode_matches_torch():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = e8m0_decode(b)
    assert np.array_equal(np.isnan(got), np.isnan(ref)) and np.isnan(got[255])
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert e8m0_decode(127) == 1.0


def _rne_step_encode(y):
    """Second rounding algorithm: scale by the binade's step, rint (ties to even)."""
    a = np.minimum(np.abs(np.asarray(y, np.float64)), 6.0)
    _, ex = np.frexp(np.maximum(a, 1.0))
    step = np.where(a < 1.0, 0.5, np.exp2((ex - 2).astype(np.float64)))
    return np.minimum(np.rint(a / step) * step, 6.0) * np.where(np.signbit(y), -1.0, 1.0)


def test_e2m1_encode_two_algorithms_agree():
    rng = np.random.default_rng(5)
    y = np.concatenate([rng.uniform(-8, 8, 200_000), np.arange(-7, 7.0001, 0.125),
                        rng.normal(0, 2, 100_000)])
    got = e2m1_decode(e2m1_encode(y))
    assert np.array_equal(got, _rne_step_encode(y))


def test_e2m1_encode_ties_saturation_sign():
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for y, v in ties.items():
        assert e2m1_decode(e2m1_encode(y)) == v
        assert e2m1_decode(e2m1_encode(-y)) == -v
    assert e2m1_decode(e2m1_encode(7.0)) == 6.0 and e2m1_decode(e2m1_encode(-1e30)) == -6.0
    assert e2m1_encode(-0.0) == 8 and e2m1_encode(0.0) == 0
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(e2m1_encode(e2m1_decode(codes)), codes)


def test_shared_exponent_examples():
    amax = np.array([6.0, 4.0, 7.99, 1.0, 0.99, 0.0, 2.0 ** -130, 1.5 * 2.0 ** 127])
    assert list(shared_exponent(amax)) == [0, 0, 0, -2, -3, -127, -127, 125]


def test_packing_order_low_nibble_first():
    x = np.zeros((1, 576))
    x[0, 0] = 0.5   # block 0 amax 6 -> scale 1: element 0 code 1
    x[0, 1] = -6.0  # element 1 code 0xF
    packed, scales = quantize_rows(x)
    assert packed[0, 0] == 0xF1 and scales[0, 0] == 127
    assert scales[0, 1] == 0  # all-zero block: exponent -127
    assert np.array_equal(unpack_codes(packed)[0, :2], [1, 15])


def test_representable_blocks_are_exact():
    rng = np.random.default_rng(6)
    n = 300
    k = rng.integers(-20, 20, size=(n, 18))
    codes = rng.integers(0, 16, size=(n, 18, 32))
    codes[:, :, 0] = rng.choice([6, 7, 14, 15], size=(n, 18))  # |value| 4 or 6 sets amax's binade
    x = (e2m1_decode(codes) * np.exp2(k.astype(np.float64))[..., None]).reshape(n, 576)
    packed, scales = quantize_rows(x)
    assert np.array_equal(scales.astype(np.int64) - 127, k)
    assert np.array_equal(dequant_rows(packed, scales, np.arange(n)), x)


def test_quantiser_brute_force_and_error_bound():
    x = bf16_bits_to_f32(normal_bf16_rows(21, 40)).astype(np.float64)
    packed, scales = quantize_rows(x)
    deq = dequant_rows(packed, scales, np.arange(40))
    for r in range(0, 40, 7):
        for blk in range(18):
            seg = x[r, 32 * blk:32 * blk + 32]
            amax = np.abs(seg).max()
            e = math.floor(math.log2(amax)) - 2
            assert scales[r, blk] == e + 127
            X = 2.0 ** e
            for i in range(32):
                # nearest grid value (ties: even code) by exhaustive search
                cands = [(abs(abs(seg[i]) / X - g), c % 2, g) for c, g in enumerate(SPEC_E2M1)]
                g = min(cands)[2]
                want = math.copysign(g * X, seg[i])
                assert deq[r, 32 * blk + i] == want
    X = np.exp2(scales.astype(np.float64) - 127).repeat(32, axis=1)
    assert np.all(np.abs(deq - x) <= 2 * X)


def _bf16(x):
    from mla_decode_attention_08_gb300.inputs import f32_to_bf16_bits
    return bf16_bits_to_f32(f32_to_bf16_bits(np.asarray(x, np.float32))).astype(np.float64)


def test_decode_brute_force_tiny():
    rng = np.random.default_rng(7)
    lengths = [3, 1, 5]
    kv_indptr = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    qo_indptr = np.arange(4, dtype=np.int32)
    N = int(kv_indptr[-1])
    q = _bf16(rng.normal(size=(3, 16, 576)))
    packed, scales = quantize_rows(rng.normal(size=(N, 576)) * 3)
    out = mla_decode_ref_mxfp4(q, packed, scales, qo_indptr, kv_indptr)
    for b in range(3):
        toks = range(kv_indptr[b], kv_indptr[b + 1])
        rows = []
        for j in toks:  # element by element from the nibbles and scale bytes
            row = []
            for d in range(576):
                byte = int(packed[j, d // 2])
                nib = byte & 0xF if d % 2 == 0 else byte >> 4
                mag = SPEC_E2M1[nib & 7]
                row.append((-mag if nib & 8 else mag) * 2.0 ** (int(scales[j, d // 32]) - 127))
            rows.append(row)
        k = np.array(rows)
        for h in range(16):
            z = [sum(q[b, h, d] * k[t, d] for d in range(576)) * SM_SCALE for t in range(len(rows))]
            w = [math.exp(v) for v in z]
            s = sum(w)
            o = [sum(w[t] * k[t, d] for t in range(len(rows))) / s for d in range(0, 512, 37)]
            assert np.allclose(out[b, h, 0:512:37], o, rtol=1e-12, atol=1e-14)


def test_equals_e4m3_step_on_exactly_representable_cache():
    # MXFP4 values e2m1 * 2^k with k in [-8, 6] are exact e4m3fn codes at scale 1,
    # so both decode steps see identical float64 caches.
    rng = np.random.default_rng(8)
    N, B = 96, 4
    k = rng.integers(-8, 7, size=(N, 18))
    codes = rng.integers(0, 16, size=(N, 18, 32))
    codes[:, :, 0] = 7
    x = (e2m1_decode(codes) * np.exp2(k.astype(np.float64))[..., None]).reshape(N, 576)
    packed, scales = quantize_rows(x)
    e4 = e4m3fn_encode(x.astype(np.float32))
    assert np.array_equal(e4m3fn_decode(e4), x)
    kv_indptr = np.array([0, 10, 40, 41, 96], np.int32)
    qo_indptr = np.arange(B + 1, dtype=np.int32)
    q = _bf16(rng.normal(size=(B, 16, 576)))
    a = mla_decode_ref_mxfp4(q, packed, scales, qo_indptr, kv_indptr)
    b = mla_decode_ref(q, e4, np.float32(1.0), qo_indptr, kv_indptr)
    assert np.array_equal(a, b)


def test_one_token_and_constant_score():
    rng = np.random.default_rng(9)
    x = rng.normal(size=(8, 576))
    packed, scales = quantize_rows(x)
    deq = dequant_rows(packed, scales, np.arange(8))
    q = _bf16(rng.normal(size=(2, 16, 576)))
    out = mla_decode_ref_mxfp4(q, packed, scales, np.arange(3, dtype=np.int32),
                               np.array([0, 1, 1], np.int32))
    assert np.array_equal(out[0], np.broadcast_to(deq[0, :512], (16, 512)))
    assert not out[1].any()  # empty row: zeros
    # constant score: q's latent part zero, every row the same rope dims
    x[:, 512:] = x[0, 512:]
    packed, scales = quantize_rows(x)
    deq = dequant_rows(packed, scales, np.arange(8))
    q[:, :, :512] = 0.0
    out = mla_decode_ref_mxfp4(q[:1], packed, scales, np.arange(2, dtype=np.int32),
                               np.array([0, 8], np.int32))
    assert np.allclose(out[0], deq[:, :512].mean(axis=0), rtol=0, atol=1e-14)
