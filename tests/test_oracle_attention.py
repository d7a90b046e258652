"""Pins of the oracle's decode attention: brute force, closed forms, invariants."""
import math

import numpy as np
import pytest

from oracle.attention import (SM_SCALE, bf16_bits_to_f64, combine_partials, mla_decode_ref,
                              mla_decode_split_ref, mla_decode_weights, split_partial)
from oracle.fp8 import e4m3fn_decode
from oracle.schedule import token_segments
from mla_decode_attention_08_gb300.inputs import f32_to_bf16_bits


def random_case(rng, lengths, paged=False):
    batch = len(lengths)
    q = bf16_bits_to_f64(f32_to_bf16_bits(rng.standard_normal((batch, 16, 576)).astype(np.float32)))
    total = int(sum(lengths))
    pool = total + 5
    codes = rng.integers(0, 256, size=(pool, 576), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C          # no NaN codes in a cache
    scale = np.float32(rng.uniform(0.001, 0.02))
    kv_indptr = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    qo_indptr = np.arange(batch + 1, dtype=np.int32)
    idx = rng.permutation(pool)[:total].astype(np.int32) if paged else None
    return q, codes, scale, qo_indptr, kv_indptr, idx


def brute_force(q, codes, scale, qo_indptr, kv_indptr, idx):
    """Definition written with scalar loops: no max shift, math.exp, sm_scale = 1/24."""
    batch = len(qo_indptr) - 1
    out = np.zeros((q.shape[0], 16, 512))
    for b in range(batch):
        t = int(qo_indptr[b])
        toks = range(int(kv_indptr[b]), int(kv_indptr[b + 1]))
        slots = [int(idx[j]) if idx is not None else j for j in toks]
        for h in range(16):
            weights = []
            for s in slots:
                k = [float(v) * float(scale) for v in e4m3fn_decode(codes[s])]
                dot = sum(q[t, h, d] * k[d] for d in range(576))
                weights.append(math.exp(dot / 24.0))      # sqrt(576) = 24
            total = sum(weights)
            for w, s in zip(weights, slots):
                v = e4m3fn_decode(codes[s][:512]) * float(scale)
                out[t, h] += (w / total) * v
    return out


@pytest.mark.parametrize("lengths,paged", [([1, 3, 7], False), ([5, 2], True), ([4], False)])
def test_brute_force_tiny(lengths, paged):
    rng = np.random.default_rng(sum(lengths) + 10 * paged)
    case = random_case(rng, lengths, paged)
    q, codes, scale = case[0], case[1], case[2]
    q *= 0.05   # keep exp() of unshifted scores finite in the brute force
    ref = mla_decode_ref(q, codes, scale, *case[3:5], kv_indices=case[5])
    bf = brute_force(q, codes, scale, *case[3:])
    np.testing.assert_allclose(ref, bf, rtol=1e-10, atol=1e-12)


def test_sm_scale_is_one_over_24():
    assert SM_SCALE == 1.0 / 24.0


def test_two_token_closed_form_rope_dims_score_but_do_not_carry_value():
    # Only dim 520 (a rope dim) of q is non-zero, so the scores come from the rope
    # part alone; V (dims < 512) is read from the same rows.
    q = np.zeros((1, 16, 576))
    q[0, :, 520] = np.arange(16) * 0.5                 # head h: 0.5 h
    codes = np.zeros((2, 576), dtype=np.uint8)
    codes[0, 520], codes[1, 520] = 0x38, 0x40          # k = 1.0 and 2.0 (times scale 1)
    codes[0, :512], codes[1, :512] = 0x38, 0xB8        # v = +1 and -1
    out = mla_decode_ref(q, codes, np.float32(1.0), [0, 1], [0, 2])
    for h in range(16):
        z0, z1 = 0.5 * h * 1.0 / 24.0, 0.5 * h * 2.0 / 24.0
        w1 = math.exp(z1) / (math.exp(z0) + math.exp(z1))
        np.testing.assert_allclose(out[0, h], (1 - w1) - w1, rtol=0, atol=1e-15)


def test_weights_sum_to_one_and_empty_row_is_zero():
    rng = np.random.default_rng(5)
    q, codes, scale, qo, kv, idx = random_case(rng, [9, 0, 300], paged=True)
    for b in (0, 2):
        w = mla_decode_weights(q, codes, scale, qo, kv, b, kv_indices=idx)
        assert np.all(np.abs(w.sum(axis=1) - 1.0) < 1e-12)
        assert np.all(w >= 0)
    out = mla_decode_ref(q, codes, scale, qo, kv, kv_indices=idx)
    assert np.all(out[1] == 0.0)


def test_one_token_returns_v_exactly():
    rng = np.random.default_rng(6)
    q, codes, scale, qo, kv, idx = random_case(rng, [1, 1], paged=True)
    out = mla_decode_ref(q, codes, scale, qo, kv, kv_indices=idx)
    for b in range(2):
        v = e4m3fn_decode(codes[idx[b], :512]) * float(scale)
        assert np.array_equal(out[b], np.broadcast_to(v, (16, 512)))


def test_constant_score_gives_mean_of_v():
    rng = np.random.default_rng(7)
    q, codes, scale, qo, kv, _ = random_case(rng, [37])
    q[:, :, :512] = 0.0                 # scores depend on rope dims only ...
    codes[:, 512:] = codes[0, 512:]     # ... which every row shares
    out = mla_decode_ref(q, codes, scale, qo, kv)
    mean_v = (e4m3fn_decode(codes[:37, :512]) * float(scale)).mean(axis=0)
    np.testing.assert_allclose(out[0], np.broadcast_to(mean_v, (16, 512)), rtol=0, atol=1e-15)


def test_permutation_invariance():
    rng = np.random.default_rng(8)
    q, codes, scale, qo, kv, _ = random_case(rng, [50])
    perm = rng.permutation(50).astype(np.int32)
    a = mla_decode_ref(q, codes, scale, qo, kv)
    b = mla_decode_ref(q, codes, scale, qo, kv, kv_indices=perm)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)


def test_split_combine_equals_unsplit():
    rng = np.random.default_rng(9)
    lengths = [700, 1, 129, 0, 256]
    q, codes, scale, qo, kv, idx = random_case(rng, lengths, paged=True)
    full = mla_decode_ref(q, codes, scale, qo, kv, kv_indices=idx)
    for grid in (1, 3, 7, 11):
        segs = token_segments(kv, grid)
        split = mla_decode_split_ref(q, codes, scale, qo, kv, segs, kv_indices=idx)
        np.testing.assert_allclose(split, full, rtol=1e-11, atol=1e-13)


def test_combine_with_empty_split_and_single_split():
    rng = np.random.default_rng(10)
    q = rng.standard_normal((16, 576))
    k = rng.standard_normal((20, 576))
    o, lse = split_partial(q, k)
    z, zl = split_partial(q, k[:0])
    assert np.all(z == 0) and np.all(np.isneginf(zl))
    np.testing.assert_array_equal(combine_partials([o, z], [lse, zl]), o)
    np.testing.assert_allclose(combine_partials([o], [lse]), o, rtol=0, atol=0)
    assert np.all(combine_partials([z], [zl]) == 0)


def test_rejects_multi_token_queries():
    with pytest.raises(ValueError):
        mla_decode_ref(np.zeros((2, 16, 576)), np.zeros((4, 576), np.uint8), 1.0, [0, 2], [0, 4])
