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


def test_rejects_rows_without_query_tokens():
    with pytest.raises(ValueError):
        mla_decode_ref(np.zeros((2, 16, 576)), np.zeros((4, 576), np.uint8), 1.0, [0, 2, 2], [0, 4, 4])


# ------------------------------------------------------------------ multi-token rows
def multi_token_case(rng, lengths, n, paged=False):
    """Rows of n query tokens each (qo_indptr = n * arange), small query values."""
    q, codes, scale, _, kv_indptr, idx = random_case(rng, lengths, paged)
    batch = len(lengths)
    q = bf16_bits_to_f64(f32_to_bf16_bits(
        (0.05 * rng.standard_normal((batch * n, 16, 576))).astype(np.float32)))
    qo_indptr = (n * np.arange(batch + 1)).astype(np.int32)
    return q, codes, scale, qo_indptr, kv_indptr, idx


def brute_force_positions(q, codes, scale, qo_indptr, kv_indptr, idx):
    """Multi-token decode with scalar loops, phrased by sequence positions: a
    row's cache holds positions 0..L-1, its n query tokens are the last n of
    them (positions L-n..L-1), and a query at position p sees positions <= p."""
    out = np.zeros((q.shape[0], 16, 512))
    for b in range(len(qo_indptr) - 1):
        n = int(qo_indptr[b + 1] - qo_indptr[b])
        length = int(kv_indptr[b + 1] - kv_indptr[b])
        for i in range(n):
            t = int(qo_indptr[b]) + i
            pos = length - n + i
            slots = []
            for j in range(length):
                if j <= pos:
                    g = int(kv_indptr[b]) + j
                    slots.append(int(idx[g]) if idx is not None else g)
            for h in range(16):
                weights = []
                for sl in slots:
                    k = [float(v) * float(scale) for v in e4m3fn_decode(codes[sl])]
                    weights.append(math.exp(sum(q[t, h, d] * k[d] for d in range(576)) / 24.0))
                total = sum(weights)
                for w, sl in zip(weights, slots):
                    out[t, h] += (w / total) * (e4m3fn_decode(codes[sl][:512]) * float(scale))
    return out


@pytest.mark.parametrize("lengths,n,paged", [([3, 5], 2, False), ([4, 1, 6], 2, True), ([5], 3, False),
                                             ([2], 4, False)])
def test_multi_token_brute_force(lengths, n, paged):
    rng = np.random.default_rng(1000 + 7 * n + sum(lengths))
    case = multi_token_case(rng, lengths, n, paged)
    ref = mla_decode_ref(*case[:5], kv_indices=case[5])
    np.testing.assert_allclose(ref, brute_force_positions(*case), rtol=1e-10, atol=1e-12)


def test_multi_token_full_row_is_causal_attention():
    """With as many query tokens as cached tokens the step is plain causal
    attention over the row: a lower-triangular mask on the score matrix."""
    rng = np.random.default_rng(77)
    length = 9
    q, codes, scale, qo, kvp, idx = multi_token_case(rng, [length], length)
    ref = mla_decode_ref(q, codes, scale, qo, kvp)
    k = e4m3fn_decode(codes[:length]) * float(scale)
    for h in range(16):
        z = (q[:, h, :] @ k.T) / 24.0
        z[np.triu(np.ones((length, length), dtype=bool), 1)] = -np.inf
        w = np.exp(z - z.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        np.testing.assert_allclose(ref[:, h, :], w @ k[:, :512], rtol=1e-12, atol=1e-14)


def test_multi_token_last_token_is_plain_decode_and_early_tokens_see_less():
    rng = np.random.default_rng(78)
    lengths, n = [7, 3, 12], 3
    q, codes, scale, qo, kvp, idx = multi_token_case(rng, lengths, n, paged=True)
    ref = mla_decode_ref(q, codes, scale, qo, kvp, kv_indices=idx)
    for b, length in enumerate(lengths):
        for i in range(n):
            # token i alone, as a one-token row over the first L - n + 1 + i tokens
            vis = length - n + 1 + i
            one = mla_decode_ref(q[[n * b + i]], codes, scale, [0, 1], [0, vis],
                                 kv_indices=idx[kvp[b]:kvp[b] + vis])
            np.testing.assert_array_equal(ref[n * b + i], one[0])


def test_multi_token_tokens_that_see_nothing_are_zero():
    rng = np.random.default_rng(79)
    q, codes, scale, qo, kvp, idx = multi_token_case(rng, [1, 2], 3)
    ref = mla_decode_ref(q, codes, scale, qo, kvp)
    # row 0 (L=1): tokens 0 and 1 see nothing, token 2 sees one; row 1 (L=2): token 0 sees nothing
    assert np.all(ref[[0, 1, 3]] == 0) and all(np.any(ref[t] != 0) for t in (2, 4, 5))
    np.testing.assert_array_equal(ref[2], e4m3fn_decode(codes[0, :512])[None, :].repeat(16, 0) * float(scale))


def test_multi_token_split_equals_unsplit():
    rng = np.random.default_rng(80)
    lengths, n = [300, 129, 5], 2
    case = multi_token_case(rng, lengths, n, paged=True)
    ref = mla_decode_ref(*case[:5], kv_indices=case[5])
    for grid in (1, 3, 7):
        segs = token_segments(case[4], grid)
        got = mla_decode_split_ref(*case[:5], segs, kv_indices=case[5])
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ bf16 cache
def bf16_value(bits: int) -> float:
    """A bf16 bit pattern is the upper half of a float32 (decoded through struct)."""
    import struct
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def brute_force_bf16(q, kv_bits, qo_indptr, kv_indptr, idx):
    """The bf16-cache step with scalar loops over positions (multi-token aware)."""
    out = np.zeros((q.shape[0], 16, 512))
    for b in range(len(qo_indptr) - 1):
        n = int(qo_indptr[b + 1] - qo_indptr[b])
        length = int(kv_indptr[b + 1] - kv_indptr[b])
        for i in range(n):
            t = int(qo_indptr[b]) + i
            slots = []
            for j in range(length - n + i + 1):
                g = int(kv_indptr[b]) + j
                slots.append(int(idx[g]) if idx is not None else g)
            rows = {s: [bf16_value(v) for v in kv_bits[s]] for s in slots}
            for h in range(16):
                weights = [math.exp(sum(q[t, h, d] * rows[s][d] for d in range(576)) / 24.0)
                           for s in slots]
                total = sum(weights)
                for w, s in zip(weights, slots):
                    out[t, h] += (w / total) * np.array(rows[s][:512])
    return out


def bf16_case(rng, lengths, n=1, paged=False):
    batch = len(lengths)
    q = bf16_bits_to_f64(f32_to_bf16_bits(
        (0.05 * rng.standard_normal((batch * n, 16, 576))).astype(np.float32)))
    total = int(sum(lengths))
    kv_bits = f32_to_bf16_bits(rng.standard_normal((total + 3, 576)).astype(np.float32))
    kv_indptr = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    qo_indptr = (n * np.arange(batch + 1)).astype(np.int32)
    idx = rng.permutation(total + 3)[:total].astype(np.int32) if paged else None
    return q, kv_bits, qo_indptr, kv_indptr, idx


@pytest.mark.parametrize("lengths,n,paged", [([1, 3, 7], 1, False), ([5, 2], 1, True),
                                             ([4, 1, 6], 2, True), ([3], 3, False)])
def test_bf16_cache_brute_force_tiny(lengths, n, paged):
    from oracle.attention import mla_decode_ref_bf16kv
    rng = np.random.default_rng(2000 + 11 * n + sum(lengths) + paged)
    q, kv_bits, qo, kvp, idx = bf16_case(rng, lengths, n, paged)
    ref = mla_decode_ref_bf16kv(q, kv_bits, qo, kvp, kv_indices=idx)
    np.testing.assert_allclose(ref, brute_force_bf16(q, kv_bits, qo, kvp, idx), rtol=1e-10, atol=1e-12)


def test_bf16_cache_of_fp8_values_equals_the_fp8_step():
    """A bf16 cache holding exactly the e4m3 values times a power-of-two scale
    (three mantissa bits fit in bf16's seven) gives the fp8 step bit for bit."""
    from oracle.attention import mla_decode_ref_bf16kv
    rng = np.random.default_rng(2100)
    q, codes, _, qo, kvp, idx = random_case(rng, [40, 0, 3, 129], paged=True)
    scale = np.float32(2.0 ** -5)
    vals = e4m3fn_decode(codes) * float(scale)
    bits = f32_to_bf16_bits(vals.astype(np.float32))
    assert np.array_equal(bf16_bits_to_f64(bits), vals)
    a = mla_decode_ref(q, codes, scale, qo, kvp, kv_indices=idx)
    b = mla_decode_ref_bf16kv(q, bits, qo, kvp, kv_indices=idx)
    assert np.array_equal(a, b)


def test_bf16_cache_one_token_returns_its_v():
    from oracle.attention import mla_decode_ref_bf16kv
    rng = np.random.default_rng(2200)
    q, kv_bits, qo, kvp, idx = bf16_case(rng, [1, 1], paged=True)
    out = mla_decode_ref_bf16kv(q, kv_bits, qo, kvp, kv_indices=idx)
    for b in range(2):
        want = [bf16_value(v) for v in kv_bits[idx[b], :512]]
        assert np.array_equal(out[b], np.broadcast_to(want, (16, 512)))
