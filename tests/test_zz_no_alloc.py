"""The decode entry point that allocates nothing (mla_decode_fwd_static_scratch).

Some callers cannot allocate device memory themselves: a plugin inside a host
application that owns every device allocation, or a serving loop where an
allocation could synchronise the device.  For them the library keeps its own
fixed scratch array on each GPU.  These tests call that entry point through the
C ABI and check it against the workspace entry point on the same plan (the
same bits: the output is deterministic for a plan) and against the oracle, on
calls in a row whose plans, grids and split rows differ, so that whatever an
earlier call left in the shared array cannot decide a later call's result.  The
file is named to run after every other test; it passes alone as well.
"""
import ctypes

import numpy as np
import pytest
import torch

from mla_decode_attention_08_gb300 import binding
from mla_decode_attention_08_gb300.inputs import make_from_lengths

from .gpu_util import DeviceCase, OracleCase, assert_close

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 12 * 1024 * 1024


@pytest.fixture(scope="module")
def lib(built_library):
    return binding.load_library(built_library)


def static_call(dev: DeviceCase, plan) -> np.ndarray:
    out = torch.full_like(dev.out, float("nan"))
    binding.mla_decode_fwd_static_scratch(dev.q, dev.kv_codes, dev.kv_scale, dev.qo_indptr,
                                          dev.kv_indptr, out, plan=plan, kv_indices=dev.kv_indices)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def check_against_both(dev: DeviceCase, plan, ref: np.ndarray) -> None:
    got = static_call(dev, plan)
    want, err, _, _ = dev.run(plan=plan)
    assert err == 0
    assert np.array_equal(got, want)      # the same plan gives the same bits
    assert_close(got, ref)
    assert binding.mla_decode_static_scratch_read_error(clear=True) == 0


def test_static_scratch_calls_in_a_row(lib):
    binding.mla_decode_static_scratch_read_error(clear=True)
    # Call 1: a contiguous batch on a 152-worker grid (many split rows, every slot used).
    a = make_from_lengths([4000, 129, 7000, 1, 2500, 3000], seed=90)
    plan_a = binding.mla_decode_plan(a.batch, a.max_kv_len, 152)
    dev_a = DeviceCase(a)
    check_against_both(dev_a, plan_a, OracleCase(a).reference())

    # Calls 2 and 3: another shape, a page table and a 7-worker grid: split rows,
    # a whole row, an empty row, twice in a row.
    b = make_from_lengths([300, 1000, 17, 0, 4500], seed=91, paged=True)
    plan_b = binding.mla_decode_plan(b.batch, b.max_kv_len, 7)
    assert plan_b.grid != plan_a.grid and plan_b.ws_bytes <= STATIC_SCRATCH_BYTES
    dev_b = DeviceCase(b)
    ref_b = OracleCase(b).reference()
    for _ in range(2):
        check_against_both(dev_b, plan_b, ref_b)

    # Call 4: the same plan with other row lengths in the same buffers (within the
    # plan's max_kv_len): other split rows and combine jobs than call 3 left behind.
    c = make_from_lengths([4400, 5, 0, 1200, 200], seed=92, paged=True, max_kv_len=b.max_kv_len)
    dev_c = DeviceCase(c)
    check_against_both(dev_c, plan_b, OracleCase(c).reference())

    # Call 5: back to the first plan after the others.
    check_against_both(dev_a, plan_a, OracleCase(a).reference())


def test_static_scratch_error_word(lib):
    binding.mla_decode_static_scratch_read_error(clear=True)
    inp = make_from_lengths([200, 300, 100], seed=14)
    dev = DeviceCase(inp)
    plan = binding.mla_decode_plan(inp.batch, inp.max_kv_len, 2)
    good = dev.qo_indptr
    dev.qo_indptr = torch.tensor([0, 2, 2, 3], dtype=torch.int32, device="cuda")  # row 0 holds two tokens
    static_call(dev, plan)
    assert binding.mla_decode_static_scratch_read_error(clear=True) & 1  # MLA_DERR_QO_INDPTR
    assert binding.mla_decode_static_scratch_read_error(clear=False) == 0
    dev.qo_indptr = good
    got = static_call(dev, plan)
    assert binding.mla_decode_static_scratch_read_error(clear=True) == 0
    assert_close(got, OracleCase(inp).reference())


def test_static_scratch_rejects_plans_beyond_its_size(lib):
    big = binding.mla_decode_plan(2_000_000, 8192, 152)
    assert big.ws_bytes > STATIC_SCRATCH_BYTES
    status = lib.mla_decode_fwd_static_scratch(None, None, None, None, None, None, None,
                                               ctypes.byref(big), None, 0, 1)
    assert status == 3  # MLA_ERR_WORKSPACE_TOO_SMALL, before anything is launched
