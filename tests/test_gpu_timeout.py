"""The bounded waits, made to run out on the GPU without a fault.

mla_decode_fwd_stall_stream launches the decode with producers that never
load the cache, so the waits on those loads (a flag nothing sets) reach their
time limit.  The kernel must report MLA_DERR_TIMEOUT in the workspace error
word, return, and leave the context usable: the next call on the same
workspace gives the right answer.  Both the contiguous and the page-table
kernels, with one, two and four query tokens (two sibling CTAs per worker),
and the MXFP4 kernel (whose converter warps wait on the missing loads) are
covered.
"""
import time

import pytest
import torch

from mla_decode_attention_08_gb300 import binding
from mla_decode_attention_08_gb300.inputs import make_from_lengths

from .gpu_util import DeviceCase, OracleCase, assert_close

pytestmark = pytest.mark.gpu

MLA_DERR_TIMEOUT = 8


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    binding.load_library(built_library)


@pytest.mark.parametrize("paged,qo_len", [(False, 1), (True, 1), (False, 2), (True, 2), (False, 4),
                                          (True, 4)])
def test_stalled_stream_times_out_and_the_context_survives(paged, qo_len):
    inp = make_from_lengths([700, 300, 2000, 5], seed=31, paged=paged, qo_len=qo_len)
    dev = DeviceCase(inp)
    plan = binding.mla_decode_plan(inp.batch, inp.max_kv_len, 6, qo_len=qo_len)
    ws = binding.new_workspace(plan)
    t0 = time.time()
    binding.mla_decode_fwd_stall_stream(dev.q, dev.kv_codes, dev.kv_scale, dev.qo_indptr,
                                        dev.kv_indptr, dev.out, plan=plan, workspace=ws,
                                        kv_indices=dev.kv_indices)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    err = binding.mla_decode_read_error(ws)  # reads and clears
    assert err == MLA_DERR_TIMEOUT, err
    assert elapsed < 30.0
    # the same workspace and context, a normal call
    gpu, err, _, _ = dev.run(plan=plan, workspace=ws)
    assert err == 0
    assert_close(gpu, OracleCase(inp).reference())


def test_mxfp4_stalled_stream_times_out_and_the_context_survives():
    from oracle.mxfp4 import mla_decode_ref_mxfp4
    from oracle.attention import bf16_bits_to_f64
    from .test_gpu_mxfp4 import MxCase
    inp = make_from_lengths([700, 300, 2000, 5], seed=32)
    case = MxCase(inp)
    plan = binding.mla_decode_plan(inp.batch, inp.max_kv_len, 6)
    ws = binding.new_workspace(plan)
    t0 = time.time()
    binding.mla_decode_fwd_mxfp4_stall_stream(case.q, case.fp4, case.sc, case.qo_indptr,
                                              case.kv_indptr, case.out, plan=plan, workspace=ws)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    err = binding.mla_decode_read_error(ws)
    assert err == MLA_DERR_TIMEOUT, err
    assert elapsed < 30.0
    gpu, err, _, _ = case.run(plan=plan, workspace=ws)
    assert err == 0
    assert_close(gpu, mla_decode_ref_mxfp4(bf16_bits_to_f64(inp.q_bits), case.fp4_host, case.sc_host,
                                           inp.qo_indptr, inp.kv_indptr))
