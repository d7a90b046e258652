"""The bf16-cache decode step (mla_decode_fwd_bf16kv) through the C ABI against
the float64 oracle over the same bf16 cache values.  The bf16 cache is read
contiguously (no page table).

K and V are the cache's bf16 values and the query is the bf16 value handed in;
the kernel rounds P to bf16 (relative error 2^-9) and accumulates in float32,
so besides the pages' tolerance the relative L2 error is held to 5e-3 (the
final rounding of the output to bf16 alone contributes about 1e-3)."""
import numpy as np
import pytest
import torch

from mla_decode_attention_08_gb300 import binding
from mla_decode_attention_08_gb300.inputs import make_from_lengths, make_inputs
from oracle.attention import bf16_bits_to_f64, mla_decode_ref_bf16kv

from .gpu_util import assert_close, bits_to_bf16, num_sms

pytestmark = pytest.mark.gpu

REL_L2_BF16 = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    binding.load_library(built_library)


class Bf16Case:
    """Inputs on the GPU with the bf16 cache used as it is."""

    def __init__(self, inp):
        self.inp = inp
        self.q = bits_to_bf16(inp.q_bits)
        bits = inp.kv_bits if inp.kv_bits.shape[0] else np.zeros((1, 576), np.uint16)
        self.kv = bits_to_bf16(bits)
        self.qo_indptr = torch.from_numpy(inp.qo_indptr).cuda()
        self.kv_indptr = torch.from_numpy(inp.kv_indptr).cuda()
        self.kv_indices = None if inp.kv_indices is None else torch.from_numpy(inp.kv_indices).cuda()
        self.out = torch.empty((inp.batch * inp.qo_len, 16, 512), dtype=torch.bfloat16, device="cuda")

    def plan(self, sms=None):
        return binding.mla_decode_plan(self.inp.batch, self.inp.max_kv_len, sms or num_sms(),
                                       qo_len=self.inp.qo_len)

    def run(self, sms=None, plan=None, workspace=None):
        plan = plan or self.plan(sms)
        ws = workspace if workspace is not None else binding.new_workspace(plan)
        binding.mla_decode_fwd_bf16kv(self.q, self.kv, self.qo_indptr, self.kv_indptr, self.out,
                                      plan=plan, workspace=ws, kv_indices=self.kv_indices)
        torch.cuda.synchronize()
        return self.out.float().cpu().numpy(), binding.mla_decode_read_error(ws), plan, ws

    def reference(self, rows=None):
        inp = self.inp
        return mla_decode_ref_bf16kv(bf16_bits_to_f64(inp.q_bits), inp.kv_bits, inp.qo_indptr,
                                     inp.kv_indptr, inp.kv_indices, rows=rows)


CASES = [
    ("one_tile", [128], 1),
    ("tails", [1, 127, 128, 129, 255, 257, 1000], 1),
    ("empty_rows", [0, 300, 0, 1, 0], 1),
    ("short_rows", [3, 129, 700, 64, 1], 1),
    ("long_row", [5000], 1),
    ("many_rows", list(range(1, 400, 13)), 1),
    ("two_token_tails", [2, 127, 128, 129, 130, 1000], 2),
    ("two_token_see_nothing", [1, 0, 2, 1], 2),
    ("two_token_mixed", [3, 129, 700, 64, 1, 2000], 2),
    ("three_tokens", [3, 4, 129, 1000, 0, 2], 3),
    ("four_tokens", [4, 5, 128, 131, 1000, 1], 4),
]


@pytest.mark.parametrize("name,lengths,qo_len", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("sms", [1, 5, None])
def test_bf16_cache_matches_oracle(name, lengths, qo_len, sms):
    inp = make_from_lengths(lengths, seed=900 + len(lengths) + qo_len, qo_len=qo_len)
    case = Bf16Case(inp)
    gpu, err, _, _ = case.run(sms=sms)
    assert err == 0
    assert_close(gpu, case.reference(), rel_l2_max=REL_L2_BF16)


def test_bf16_cache_sharp_scores_exercise_rescaling():
    inp = make_from_lengths([2000, 517, 4096], seed=908)
    inp.q_bits = (inp.q_bits.view(np.uint16).astype(np.uint32) + (4 << 7)).astype(np.uint16)  # q x 16
    case = Bf16Case(inp)
    gpu, err, _, _ = case.run(sms=3)
    assert err == 0
    assert_close(gpu, case.reference(), rel_l2_max=REL_L2_BF16)


def test_bf16_cache_one_token_rows_return_v_exactly():
    """One cached token: P = 1 and l = 1, so the output is that row's V bit for bit."""
    inp = make_from_lengths([1, 1, 1], seed=909)
    gpu, err, _, _ = Bf16Case(inp).run()
    assert err == 0
    for b in range(3):
        v = bf16_bits_to_f64(inp.kv_bits[b, :512])
        assert np.array_equal(gpu[b], np.broadcast_to(v, (16, 512))), b


def test_bf16_cache_separate_stages_give_the_same_bits():
    inp = make_from_lengths([300, 1000, 17, 4500, 129, 0, 2000], seed=910)
    case = Bf16Case(inp)
    plan = case.plan(7)
    ws = binding.new_workspace(plan)
    gpu, err, _, _ = case.run(plan=plan, workspace=ws)
    assert err == 0
    out2 = torch.full_like(case.out, float("nan"))
    binding.mla_decode_stage1_bf16kv(case.q, case.kv, case.qo_indptr, case.kv_indptr, out2,
                                     plan=plan, workspace=ws, kv_indices=case.kv_indices)
    binding.mla_decode_stage2(case.qo_indptr, out2, plan=plan, workspace=ws)
    torch.cuda.synchronize()
    assert binding.mla_decode_read_error(ws) == 0
    assert np.array_equal(out2.float().cpu().numpy(), gpu)
    assert_close(gpu, case.reference(), rel_l2_max=REL_L2_BF16)


def test_bf16_cache_rejects_a_page_table():
    inp = make_from_lengths([50, 60], seed=911, paged=True)
    case = Bf16Case(inp)
    with pytest.raises(binding.MlaError) as e:
        case.run()
    assert e.value.status == 2


@pytest.mark.parametrize("name", ["bs4_kv1024", "bs32_kv1024", "bs64_kv8192", "bs256_kv8192",
                                  "bs64_q2_kv8192", "bs64_q4_kv8192"])
def test_bf16_cache_workloads(name):
    """The contiguous benchmark shapes over their bf16 cache: every row of the
    small ones, sampled rows (first, last, a few in between) of the large ones."""
    inp = make_inputs(name)
    case = Bf16Case(inp)
    gpu, err, plan, _ = case.run()
    assert err == 0 and np.isfinite(gpu).all()
    full = inp.batch * inp.max_kv_len <= 32 * 1024
    rows = None if full else sorted({0, 1, inp.batch // 2, inp.batch - 2, inp.batch - 1})
    ref = case.reference(rows)
    n = inp.qo_len
    toks = None if rows is None else [n * b + i for b in rows for i in range(n)]
    st = assert_close(gpu, ref, toks, rel_l2_max=REL_L2_BF16)
    print(name, "grid", plan.grid, st)


@pytest.mark.parametrize("k", range(4))
def test_bf16_cache_randomised_shapes(k):
    rng = np.random.default_rng(1400 + k)
    batch = int(rng.integers(1, 200))
    qo_len = int(rng.integers(1, 5))
    lengths = rng.integers(0, 3000, size=batch)
    lengths[rng.random(batch) < 0.1] = 0
    inp = make_from_lengths(lengths, seed=1400 + k, qo_len=qo_len)
    case = Bf16Case(inp)
    gpu, err, _, _ = case.run(sms=int(rng.integers(1, 153)))
    assert err == 0
    assert_close(gpu, case.reference(), rel_l2_max=REL_L2_BF16)
