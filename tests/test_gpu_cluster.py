"""The cluster split of small batches against the float64 oracle (GPU).

A plan with ``cluster`` = s > 0 shares every row among the s CTAs of one
thread-block cluster, which meet at one cluster barrier and combine their
partials (written to the workspace, read back through L2), with no second
kernel.  These tests run shapes that make the plan pick
s = 8, 4 and 2 (ragged rows, rows with fewer tiles than CTAs, empty rows), the
bf16 cache, host-made input errors, the stall hook, a page table with a
cluster plan (which runs the persistent split), the two stages launched apart,
and repeat calls, through the C ABI.
"""
import time

import numpy as np
import pytest
import torch

from mla_decode_attention_08_gb300 import binding
from mla_decode_attention_08_gb300.inputs import make_from_lengths
from oracle.schedule import plan_cluster

from .gpu_util import DeviceCase, OracleCase, assert_close, num_sms

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    binding.load_library(built_library)


SHAPES = [
    # name, lengths, max_kv_len (None: the longest), sms, cluster size the plan takes
    ("bs4_uniform", [1024] * 4, None, 152, 8),
    ("ragged_8", [1000, 1, 0, 700, 129, 257], None, 152, 8),
    ("ranks_without_tiles", [130, 5, 1024], None, 152, 8),
    ("all_rows_empty", [0, 0, 0], 1024, 152, 8),
    ("bs32_ragged", list(np.random.default_rng(3).integers(0, 1025, 32)), 1024, 152, 4),
    ("three_tiles", [300, 300, 257], None, 152, 2),
    ("small_gpu", [1000, 513, 1024, 7, 900], 1024, 40, 4),
    ("one_row", [1024], None, 152, 8),
]


@pytest.mark.parametrize("name,lengths,max_len,sms,size", SHAPES, ids=[s[0] for s in SHAPES])
def test_cluster_split_matches_oracle(name, lengths, max_len, sms, size):
    inp = make_from_lengths(lengths, seed=500 + len(lengths), max_kv_len=max_len)
    dev = DeviceCase(inp)
    dev.out.fill_(float("nan"))
    gpu, err, plan, _ = dev.run(sms=sms)
    assert plan.cluster == size == plan_cluster(inp.batch, 1, inp.max_kv_len, sms)
    assert err == 0
    ref = OracleCase(inp).reference()
    assert_close(gpu, ref)
    # the persistent split of the same plan agrees with the oracle too
    gpu_p, err_p, plan_p, _ = dev.run(sms=sms, persistent=True)
    assert plan_p.cluster == 0 and err_p == 0
    assert_close(gpu_p, ref)


def test_sharp_scores_across_the_cluster():
    """Scores scaled up so that the CTAs' log-sum-exps differ by many binades:
    the combine weights then span a wide range, and each CTA's own rescaling runs."""
    inp = make_from_lengths([1024, 900, 640, 1000], seed=61)
    inp.q_bits = (np.ascontiguousarray(inp.q_bits).view(np.uint16).astype(np.uint32) + (3 << 7)).astype(np.uint16)
    dev = DeviceCase(inp)
    gpu, err, plan, _ = dev.run()
    assert plan.cluster == 8 and err == 0
    assert_close(gpu, OracleCase(inp).reference())


def test_repeat_calls_give_the_same_bits():
    inp = make_from_lengths([1024, 333, 1024, 77], seed=62)
    dev = DeviceCase(inp)
    a, err, plan, ws = dev.run()
    b, err2, _, _ = dev.run(plan=plan, workspace=ws)
    assert plan.cluster == 8 and err == 0 and err2 == 0
    assert np.array_equal(a, b)


def test_stages_apart_equal_the_fused_call():
    """With a cluster plan, stage 1 does the whole step and a separately
    launched stage 2 finds no work: the pair gives the fused call's bits."""
    inp = make_from_lengths([800, 1024, 1, 600], seed=63)
    dev = DeviceCase(inp)
    fused, err, plan, ws = dev.run()
    assert plan.cluster == 8 and err == 0
    out2 = torch.full_like(dev.out, float("nan"))
    binding.mla_decode_stage1(dev.q, dev.kv_codes, dev.kv_scale, dev.qo_indptr, dev.kv_indptr,
                              out2, plan=plan, workspace=ws)
    binding.mla_decode_stage2(dev.qo_indptr, out2, plan=plan, workspace=ws)
    torch.cuda.synchronize()
    assert binding.mla_decode_read_error(ws) == 0
    assert np.array_equal(out2.float().cpu().numpy(), fused)


def test_page_table_with_a_cluster_plan_runs_the_persistent_split():
    inp = make_from_lengths([1000, 20, 1024, 500], seed=64, paged=True)
    dev = DeviceCase(inp)
    gpu, err, plan, _ = dev.run()
    assert plan.cluster == 8 and err == 0
    assert_close(gpu, OracleCase(inp).reference())


def test_bf16_cache_cluster_split():
    from .test_gpu_bf16kv import REL_L2_BF16, Bf16Case
    for lengths in ([1024] * 4, [1000, 1, 0, 700, 129, 257], list(range(3, 1024, 37))):
        inp = make_from_lengths(lengths, seed=65 + len(lengths), max_kv_len=1024)
        case = Bf16Case(inp)
        gpu, err, plan, _ = case.run()
        assert plan.cluster > 0 and err == 0
        assert_close(gpu, case.reference(), rel_l2_max=REL_L2_BF16)


def test_bad_query_row_is_flagged_and_not_written():
    inp = make_from_lengths([200, 300, 100], seed=14)
    dev = DeviceCase(inp)
    dev.qo_indptr = torch.tensor([0, 2, 2, 3], dtype=torch.int32, device="cuda")
    dev.out.fill_(7.0)
    gpu, err, plan, _ = dev.run(sms=152)
    assert plan.cluster > 0 and err & 1
    ref = OracleCase(make_from_lengths([200, 300, 100], seed=14)).reference()
    assert_close(gpu[2:3], ref[2:3])
    assert np.all(gpu[1] == 7.0)  # row 1's span [2, 2) is empty: not written


def test_decreasing_kv_indptr_gives_zeros_and_flag():
    inp = make_from_lengths([200, 300], seed=15, max_kv_len=1024)
    dev = DeviceCase(inp)
    dev.kv_indptr = torch.tensor([0, 300, 200], dtype=torch.int32, device="cuda")
    dev.out.fill_(7.0)
    gpu, err, plan, _ = dev.run()
    assert plan.cluster > 0 and err & 2 and np.all(gpu == 0)


def test_stalled_stream_times_out_and_the_context_survives():
    inp = make_from_lengths([700, 300, 1024, 5], seed=31)
    dev = DeviceCase(inp)
    plan = binding.mla_decode_plan(inp.batch, inp.max_kv_len, num_sms())
    assert plan.cluster > 0
    ws = binding.new_workspace(plan)
    t0 = time.time()
    binding.mla_decode_fwd_stall_stream(dev.q, dev.kv_codes, dev.kv_scale, dev.qo_indptr,
                                        dev.kv_indptr, dev.out, plan=plan, workspace=ws)
    torch.cuda.synchronize()
    assert binding.mla_decode_read_error(ws) == 8  # MLA_DERR_TIMEOUT
    assert time.time() - t0 < 30.0
    gpu, err, _, _ = dev.run(plan=plan, workspace=ws)
    assert err == 0
    assert_close(gpu, OracleCase(inp).reference())


def test_a_forged_cluster_size_is_refused():
    inp = make_from_lengths([1024] * 4, seed=66)
    dev = DeviceCase(inp)
    plan = binding.mla_decode_plan(inp.batch, inp.max_kv_len, num_sms())
    plan.cluster = 4  # not what the plan rule gives for this shape
    with pytest.raises(binding.MlaError):
        dev.run(plan=plan)
