"""The MXFP4-cache decode step (mla_decode_fwd_mxfp4) and the MXFP4 quantiser
(mla_mxfp4_quantize) through the C ABI against the float64 oracle.

The caches the decode step reads in these tests are made by the oracle's
quantiser from the seeded bf16 source (the workload-sized ones by the GPU
quantiser, checked code for code against the oracle's on every row the
reference uses).  The kernel converts each block to e4m3 exactly (block scales
in its window), so K and V are exact and the arithmetic is the e4m3 cache's:
Q and P split into two e4m3 terms (about 8 significant bits), float32
accumulation, a bf16 output; the tolerance is the e4m3 path's.
"""
import numpy as np
import pytest
import torch

from mla_decode_attention_08_gb300 import binding
from mla_decode_attention_08_gb300.inputs import (bf16_bits_to_f32, f32_to_bf16_bits,
                                                  make_from_lengths, make_inputs,
                                                  normal_bf16_rows)
from oracle.attention import bf16_bits_to_f64
from oracle.mxfp4 import dequant_rows, mla_decode_ref_mxfp4, quantize_rows

from .gpu_util import assert_close, bits_to_bf16, num_sms

pytestmark = pytest.mark.gpu

MLA_DERR_MX_SCALE = 16


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    binding.load_library(built_library)


def oracle_quantize(kv_bits: np.ndarray, chunk: int = 2048):
    """The oracle's MXFP4 of bf16 rows, in row chunks (bounded host memory)."""
    n = kv_bits.shape[0]
    fp4 = np.empty((n, 288), np.uint8)
    sc = np.empty((n, 18), np.uint8)
    for r0 in range(0, n, chunk):
        fp4[r0:r0 + chunk], sc[r0:r0 + chunk] = quantize_rows(
            bf16_bits_to_f32(kv_bits[r0:r0 + chunk]).astype(np.float64))
    return fp4, sc


def gpu_quantize(kv_bits: np.ndarray):
    src = bits_to_bf16(kv_bits)
    n = kv_bits.shape[0]
    fp4 = torch.empty((n, 288), dtype=torch.uint8, device="cuda")
    sc = torch.empty((n, 18), dtype=torch.uint8, device="cuda")
    binding.mla_mxfp4_quantize(src, fp4, sc)
    torch.cuda.synchronize()
    return fp4, sc


class MxCase:
    """Inputs on the GPU with an MXFP4 cache (given, or made by the oracle)."""

    def __init__(self, inp, fp4=None, scales=None, scale_bias=0):
        self.inp = inp
        if fp4 is None:
            bits = inp.kv_bits if inp.kv_bits.shape[0] else np.zeros((1, 576), np.uint16)
            fp4, scales = oracle_quantize(bits)
        self.fp4_host, self.sc_host = fp4, scales
        self.fp4 = torch.from_numpy(fp4).cuda()
        self.sc = torch.from_numpy(scales).cuda()
        self.scale_bias = scale_bias
        self.q = bits_to_bf16(inp.q_bits)
        self.qo_indptr = torch.from_numpy(inp.qo_indptr).cuda()
        self.kv_indptr = torch.from_numpy(inp.kv_indptr).cuda()
        self.out = torch.empty((inp.batch, 16, 512), dtype=torch.bfloat16, device="cuda")

    def plan(self, sms=None):
        return binding.mla_decode_plan(self.inp.batch, self.inp.max_kv_len, sms or num_sms())

    def run(self, sms=None, plan=None, workspace=None):
        plan = plan or self.plan(sms)
        ws = workspace if workspace is not None else binding.new_workspace(plan)
        binding.mla_decode_fwd_mxfp4(self.q, self.fp4, self.sc, self.qo_indptr, self.kv_indptr,
                                     self.out, plan=plan, workspace=ws,
                                     scale_bias=self.scale_bias)
        torch.cuda.synchronize()
        return self.out.float().cpu().numpy(), binding.mla_decode_read_error(ws), plan, ws

    def reference(self, rows=None):
        inp = self.inp
        return mla_decode_ref_mxfp4(bf16_bits_to_f64(inp.q_bits), self.fp4_host, self.sc_host,
                                    inp.qo_indptr, inp.kv_indptr, rows=rows)


def test_quantiser_matches_oracle_bit_for_bit():
    rows = bf16_bits_to_f32(normal_bf16_rows(31, 3000))
    rows[5] = 0.0                                             # all-zero row
    rows[6] *= 2.0 ** -128                                    # tiny (bf16 subnormals)
    rows[7] *= 2.0 ** 100                                     # large
    # a block of exact ties after scaling (block amax 6 -> scale 1), saturation, -0
    rows[8, :16] = [6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, -1.25, -1.75, -2.5,
                    -3.5, -5, -0.0]
    rows[8, 32:36] = [7.5, -7.5, 1e-3, -1e-3]                 # amax 7.5 -> scale 1, saturate
    bits = f32_to_bf16_bits(rows)
    fp4, sc = gpu_quantize(bits)
    want_fp4, want_sc = oracle_quantize(bits)
    assert np.array_equal(sc.cpu().numpy(), want_sc)
    assert np.array_equal(fp4.cpu().numpy(), want_fp4)


CASES = [
    ("one_tile", [128]),
    ("tails", [1, 127, 128, 129, 255, 257, 1000]),
    ("empty_rows", [0, 300, 0, 1, 0]),
    ("short_rows", [3, 129, 700, 64, 1]),
    ("long_row", [5000]),
    ("many_rows", list(range(1, 400, 13))),
]


@pytest.mark.parametrize("name,lengths", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("sms", [1, 5, None])
def test_mxfp4_cache_matches_oracle(name, lengths, sms):
    inp = make_from_lengths(lengths, seed=1200 + len(lengths))
    case = MxCase(inp)
    gpu, err, _, _ = case.run(sms=sms)
    assert err == 0
    assert_close(gpu, case.reference())


def test_mxfp4_cache_one_token_rows_return_v_exactly():
    """One cached token: the output is that row's dequantised V (exact in bf16)."""
    inp = make_from_lengths([1, 1, 1], seed=1209)
    case = MxCase(inp)
    gpu, err, _, _ = case.run()
    assert err == 0
    for b in range(3):
        v = dequant_rows(case.fp4_host, case.sc_host, np.array([b]))[0, :512]
        assert np.array_equal(gpu[b], np.broadcast_to(v, (16, 512))), b


def test_mxfp4_cache_sharp_scores_exercise_rescaling():
    inp = make_from_lengths([2000, 517, 4096], seed=1210)
    inp.q_bits = (inp.q_bits.view(np.uint16).astype(np.uint32) + (4 << 7)).astype(np.uint16)  # q x 16
    case = MxCase(inp)
    gpu, err, _, _ = case.run(sms=3)
    assert err == 0
    assert_close(gpu, case.reference())


def test_mxfp4_cache_separate_stages_give_the_same_bits():
    inp = make_from_lengths([300, 1000, 17, 4500, 129, 0, 2000], seed=1211)
    case = MxCase(inp)
    plan = case.plan(7)
    ws = binding.new_workspace(plan)
    gpu, err, _, _ = case.run(plan=plan, workspace=ws)
    assert err == 0
    out2 = torch.full_like(case.out, float("nan"))
    binding.mla_decode_stage1_mxfp4(case.q, case.fp4, case.sc, case.qo_indptr, case.kv_indptr,
                                    out2, plan=plan, workspace=ws)
    binding.mla_decode_stage2(case.qo_indptr, out2, plan=plan, workspace=ws)
    torch.cuda.synchronize()
    assert binding.mla_decode_read_error(ws) == 0
    assert np.array_equal(out2.float().cpu().numpy(), gpu)


def test_mxfp4_scale_bias_moves_the_window():
    """A cache scaled by 2^12 lies outside the bias-0 window (flagged) and inside
    the bias-8 one (exact again, matching the oracle)."""
    inp = make_from_lengths([700, 129, 2000], seed=1212)
    rows = bf16_bits_to_f32(inp.kv_bits) * np.float32(2.0 ** 12)
    fp4, sc = oracle_quantize(f32_to_bf16_bits(rows))
    case = MxCase(inp, fp4, sc, scale_bias=8)
    gpu, err, _, _ = case.run()
    assert err == 0
    assert_close(gpu, case.reference())
    case.scale_bias = 0
    gpu, err, _, _ = case.run()
    assert err == MLA_DERR_MX_SCALE and np.isfinite(gpu).all()


def test_mxfp4_zero_blocks_do_not_flag():
    """All-zero blocks carry the smallest scale; they stay zero and raise nothing."""
    inp = make_from_lengths([300, 5], seed=1213)
    rows = bf16_bits_to_f32(inp.kv_bits)
    rows[::3, 64:160] = 0.0
    fp4, sc = oracle_quantize(f32_to_bf16_bits(rows))
    assert (sc == 0).any()
    case = MxCase(inp, fp4, sc)
    gpu, err, _, _ = case.run()
    assert err == 0
    assert_close(gpu, case.reference())


@pytest.mark.parametrize("name", ["bs4_kv1024", "bs32_kv1024", "bs64_kv8192", "bs256_kv8192"])
def test_mxfp4_cache_workloads(name):
    """The contiguous benchmark shapes over their MXFP4 cache (made on the GPU):
    every row of the small ones, sampled rows of the large ones, whose codes are
    first checked against the oracle's quantiser."""
    inp = make_inputs(name)
    fp4_d, sc_d = gpu_quantize(inp.kv_bits)
    full = inp.batch * inp.max_kv_len <= 32 * 1024
    rows = list(range(inp.batch)) if full else sorted({0, 1, inp.batch // 2, inp.batch - 2,
                                                       inp.batch - 1})
    fp4_ref = np.zeros((inp.kv_bits.shape[0], 288), np.uint8)
    sc_ref = np.zeros((inp.kv_bits.shape[0], 18), np.uint8)
    for b in rows:
        j0, j1 = int(inp.kv_indptr[b]), int(inp.kv_indptr[b + 1])
        fp4_ref[j0:j1], sc_ref[j0:j1] = oracle_quantize(inp.kv_bits[j0:j1])
        assert np.array_equal(fp4_d[j0:j1].cpu().numpy(), fp4_ref[j0:j1]), b
        assert np.array_equal(sc_d[j0:j1].cpu().numpy(), sc_ref[j0:j1]), b
    case = MxCase(inp, fp4_ref[:1], sc_ref[:1])
    case.fp4, case.sc = fp4_d, sc_d
    case.fp4_host, case.sc_host = fp4_ref, sc_ref
    gpu, err, plan, _ = case.run()
    assert err == 0 and np.isfinite(gpu).all()
    ref = case.reference(None if full else rows)
    st = assert_close(gpu, ref, None if full else rows)
    print(name, "grid", plan.grid, st)


def test_mxfp4_more_rows_than_prologue_threads():
    """1,000 rows (several per thread of the 512-thread prologue), lengths 0..300."""
    rng = np.random.default_rng(1214)
    lengths = rng.integers(0, 301, size=1000)
    inp = make_from_lengths(lengths, seed=1214)
    case = MxCase(inp)
    gpu, err, _, _ = case.run()
    assert err == 0
    assert_close(gpu, case.reference())


@pytest.mark.parametrize("k", range(4))
def test_mxfp4_randomised_shapes(k):
    rng = np.random.default_rng(1300 + k)
    batch = int(rng.integers(1, 200))
    lengths = rng.integers(0, 3000, size=batch)
    lengths[rng.random(batch) < 0.1] = 0
    inp = make_from_lengths(lengths, seed=1300 + k)
    case = MxCase(inp)
    gpu, err, _, _ = case.run(sms=int(rng.integers(1, 153)))
    assert err == 0
    assert_close(gpu, case.reference())
