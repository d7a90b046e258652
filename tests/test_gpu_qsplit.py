"""Stage 1's two-term e4m3 operands against the oracle, bit for bit (GPU).

The kernel's own operand code (``prepare_q`` for one and two query tokens per
CTA, ``split_p_16``) runs through the test hooks ``mla_debug_q_operand`` and
``mla_debug_p_split`` of the C ABI; ``oracle.qsplit`` restates the reading.
The codes must be identical; the query's scale factor must be exactly
2^-k2 * kv_scale * log2(e) / 24 up to the one float32 rounding of the last
product.
"""
import numpy as np
import pytest
import torch

from mla_decode_attention_08_gb300 import binding
from mla_decode_attention_08_gb300.inputs import WORKLOADS, workload_query_bits
from oracle.qsplit import bf16_bits_to_f32, p_split_e4m3, q_operand_tokens

from .gpu_util import bits_to_bf16

pytestmark = pytest.mark.gpu

LOG2E_OVER_24 = 1.4426950408889634 / 24.0


def run_q(q_bits: np.ndarray, per_cta: int, kv_scale: float = 1.0):
    q = bits_to_bf16(q_bits)
    scale = torch.tensor([kv_scale], dtype=torch.float32, device="cuda")
    codes, qk = binding.mla_debug_q_operand(q, scale, per_cta)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), qk.cpu().numpy().astype(np.float64)


def check_q(q_bits: np.ndarray, per_cta: int, kv_scale: float = 1.0):
    codes, qk = run_q(q_bits, per_cta, kv_scale)
    hi, lo, k2 = q_operand_tokens(q_bits)
    assert np.array_equal(codes[:, 0], hi), np.argwhere(codes[:, 0] != hi)[:5]
    assert np.array_equal(codes[:, 1], lo), np.argwhere(codes[:, 1] != lo)[:5]
    # qk = float32(2^-k2 * kv_scale * c) within float32 rounding (the constant's and
    # the product's; the spacing 2^-149 where it is subnormal, as for clamped tokens),
    # which pins k2: a wrong exponent is off by a factor of two
    exact = np.exp2(-k2.astype(np.float64)) * np.float64(np.float32(kv_scale)) * LOG2E_OVER_24
    assert np.all(np.abs(qk - exact) <= 2.0 ** -23 * exact + 2.0 ** -149), (qk, exact, k2)


@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("per_cta", [1, 2])
def test_workload_queries_bit_exact(name, per_cta):
    check_q(workload_query_bits(name), per_cta)


def test_real_kv_scale():
    check_q(workload_query_bits("bs32_kv1024"), 1, kv_scale=float(np.float32(4.71 / 448.0)))


def _tokens_from(values: np.ndarray, amax_bits: int) -> np.ndarray:
    per = 16 * 576 - 1
    n = (values.size + per - 1) // per
    out = np.zeros((n, 16 * 576), dtype=np.uint16)
    for t in range(n):
        chunk = values[t * per:(t + 1) * per]
        out[t, :chunk.size] = chunk
        out[t, -1] = amax_bits
    return out.reshape(n, 16, 576)


@pytest.mark.parametrize("per_cta", [1, 2])
def test_every_bf16_below_the_maximum(per_cta):
    # every finite bf16 of magnitude <= 1.75, both signs, at the fixed exponent k2 = 8
    mags = np.arange(0x0000, 0x3FE1, dtype=np.uint16)
    toks = _tokens_from(np.concatenate([mags, mags | np.uint16(0x8000)]), 0x3FE0)
    check_q(toks, per_cta)


@pytest.mark.parametrize("per_cta", [1, 2])
def test_edge_tokens(per_cta):
    rng = np.random.default_rng(11)
    toks = []
    toks.append(np.zeros((16, 576), np.uint16))                          # all zero
    toks.append(np.full((16, 576), 0x8000, np.uint16))                   # all -0
    t = rng.integers(0, 0x7F80, (16, 576)).astype(np.uint16)             # every binade
    t[5, 100] = 0x7F7F                                                   # largest finite bf16
    toks.append(t)
    toks.append(rng.integers(1, 0x0080, (16, 576)).astype(np.uint16))    # subnormals only (clamped k2)
    toks.append((rng.integers(1, 0x0080, (16, 576)).astype(np.uint16) | np.uint16(0x8000)))
    for e in (-120, -20, -6, 0, 1, 7, 40, 120):                          # amax at the window's top
        base = (rng.standard_normal((16, 576)) * 0.3 * 2.0 ** e).astype(np.float32)
        bits = (base.view(np.uint32) >> 16).astype(np.uint16)
        bits[0, 0] = (np.float32(0.875 * 2.0 ** (e + 1)).view(np.uint32) >> 16).astype(np.uint16)
        toks.append(bits)
        above = bits.copy()
        above[0, 0] += 1                                                 # one bf16 step above it
        toks.append(above)
    q = np.stack(toks)
    check_q(q, per_cta)
    check_q(q[:-1], per_cta)  # an odd count: the last two-token CTA holds one token
    assert bf16_bits_to_f32(q).dtype == np.float32


def test_p_split_bit_exact():
    halves = np.arange(0x0000, 0x5C01, dtype=np.uint16).view(np.float16).astype(np.float32)
    rng = np.random.default_rng(4)
    rand = rng.uniform(0, 256, 200_000).astype(np.float32)
    # floats exactly half-way between adjacent halves (ties of the float -> half rounding)
    h = np.arange(0x0400, 0x5BFF, 97, dtype=np.uint16).view(np.float16).astype(np.float64)
    nxt = (np.arange(0x0400, 0x5BFF, 97, dtype=np.uint16) + 1).view(np.float16).astype(np.float64)
    ties = ((h + nxt) / 2).astype(np.float32)
    p = np.concatenate([halves, rand, ties, np.float32([0.0, 256.0, 2.0 ** -24, 2.0 ** -30])])
    p = np.concatenate([p, np.zeros((-p.size) % 16, np.float32)])
    hi, lo = binding.mla_debug_p_split(torch.from_numpy(p).cuda())
    torch.cuda.synchronize()
    ohi, olo = p_split_e4m3(p)
    assert np.array_equal(hi.cpu().numpy(), ohi)
    assert np.array_equal(lo.cpu().numpy(), olo)
