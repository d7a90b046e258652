"""Multi-token decode (qo_len = 2 to 4) through the C ABI against the float64 oracle.

Each row holds n query tokens; token i sees the row's first L - n + 1 + i
cached tokens (the oracle's causal, end-aligned reading).  One KV tile serves
two tokens' 16 heads (MMA N = 64); rows of three or four tokens are shared by
two sibling CTAs per worker (tokens 0-1 and 2-3)."""
import numpy as np
import pytest
import torch

from mla_decode_attention_08_gb300 import binding
from mla_decode_attention_08_gb300.inputs import make_from_lengths

from .gpu_util import DeviceCase, OracleCase, assert_close, num_sms

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    binding.load_library(built_library)


CASES = [
    ("one_tile", [128], False),
    ("tails", [2, 127, 128, 129, 130, 255, 257, 1000], False),
    ("tokens_that_see_nothing", [1, 0, 2, 1], False),
    ("paged_mixed", [3, 129, 700, 64, 1, 2000], True),
    ("long_row", [5000], False),
    ("many_rows", list(range(2, 400, 13)), True),
]


@pytest.mark.parametrize("name,lengths,paged", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("sms", [1, 5, None])
def test_two_token_decode_matches_oracle(name, lengths, paged, sms):
    inp = make_from_lengths(lengths, seed=500 + len(lengths), paged=paged, qo_len=2)
    gpu, err, plan, _ = DeviceCase(inp).run(sms=sms)
    assert err == 0 and plan.qo_len == 2
    assert_close(gpu, OracleCase(inp).reference())


def test_two_token_separate_stages_give_the_same_bits():
    inp = make_from_lengths([300, 1000, 17, 4500, 129, 0, 2000], seed=4343, paged=True, qo_len=2)
    dev = DeviceCase(inp)
    plan = binding.mla_decode_plan(inp.batch, inp.max_kv_len, 7, qo_len=2)
    ws = binding.new_workspace(plan)
    gpu, err, _, _ = dev.run(plan=plan, workspace=ws)
    assert err == 0
    out2 = torch.full_like(dev.out, float("nan"))
    binding.mla_decode_stage1(dev.q, dev.kv_codes, dev.kv_scale, dev.qo_indptr, dev.kv_indptr,
                              out2, plan=plan, workspace=ws, kv_indices=dev.kv_indices)
    binding.mla_decode_stage2(dev.qo_indptr, out2, plan=plan, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(out2.float().cpu().numpy(), gpu)
    assert_close(gpu, OracleCase(inp).reference())


def test_rows_of_one_token_are_rejected_by_a_two_token_plan():
    """qo_indptr must give every row two tokens: a one-token layout sets the
    query error bit and writes nothing it cannot place."""
    inp = make_from_lengths([300, 200], seed=12, qo_len=2)
    dev = DeviceCase(inp)
    dev.qo_indptr.copy_(torch.tensor([0, 1, 2], dtype=torch.int32))
    _, err, _, _ = dev.run(sms=3)
    assert err & 1


MANY = [
    ("tails", [3, 4, 127, 128, 129, 131, 257, 1000]),
    ("tokens_that_see_nothing", [1, 0, 2, 3, 4, 5]),
    ("long_row", [5000]),
]


@pytest.mark.parametrize("qo_len", [3, 4])
@pytest.mark.parametrize("name,lengths", MANY, ids=[c[0] for c in MANY])
@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("sms", [1, 5, None])
def test_three_and_four_token_decode_matches_oracle(qo_len, name, lengths, paged, sms):
    inp = make_from_lengths(lengths, seed=600 + 10 * qo_len + len(lengths), paged=paged,
                            qo_len=qo_len)
    dev = DeviceCase(inp)
    dev.out.fill_(float("nan"))
    gpu, err, plan, _ = dev.run(sms=sms)
    assert err == 0 and plan.qo_len == qo_len
    assert_close(gpu, OracleCase(inp).reference())


@pytest.mark.parametrize("qo_len", [3, 4])
def test_sibling_stages_give_the_same_bits(qo_len):
    """Rows of three or four tokens: two sibling CTAs per worker write one
    partial slot; stage 1 + stage 2 launched separately equal the fused call."""
    inp = make_from_lengths([300, 1000, 17, 4500, 129, 0, 2000], seed=4400 + qo_len, paged=True,
                            qo_len=qo_len)
    dev = DeviceCase(inp)
    plan = binding.mla_decode_plan(inp.batch, inp.max_kv_len, 14, qo_len=qo_len)
    assert plan.grid == 7
    ws = binding.new_workspace(plan)
    gpu, err, _, _ = dev.run(plan=plan, workspace=ws)
    assert err == 0
    out2 = torch.full_like(dev.out, float("nan"))
    binding.mla_decode_stage1(dev.q, dev.kv_codes, dev.kv_scale, dev.qo_indptr, dev.kv_indptr,
                              out2, plan=plan, workspace=ws, kv_indices=dev.kv_indices)
    binding.mla_decode_stage2(dev.qo_indptr, out2, plan=plan, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(out2.float().cpu().numpy(), gpu)
    assert_close(gpu, OracleCase(inp).reference())


def test_four_token_rows_of_three_are_flagged():
    inp = make_from_lengths([300, 200], seed=13, qo_len=4)
    dev = DeviceCase(inp)
    dev.qo_indptr.copy_(torch.tensor([0, 3, 8], dtype=torch.int32))
    _, err, _, _ = dev.run(sms=3)
    assert err & 1


def test_two_token_workload_sampled_rows():
    """bs64 x kv8192 with two query tokens (the measured two-token shape):
    sampled rows of both output paths against the oracle."""
    from mla_decode_attention_08_gb300.inputs import make_inputs
    inp = make_inputs("bs64_q2_kv8192")
    dev = DeviceCase(inp)
    gpu, err, plan, _ = dev.run()
    assert err == 0
    rows = [0, 1, 31, 62, 63]
    ref = OracleCase(inp).reference(rows=rows)
    toks = [2 * b + i for b in rows for i in range(2)]
    assert_close(gpu[toks], ref[toks])
