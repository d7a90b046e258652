"""The decode entry point that allocates nothing (mla_decode_fwd_static_scratch).

Some callers cannot allocate device memory themselves: a plugin inside a host
application that owns every device allocation, or a serving loop where an
allocation could synchronise the device.  For them the library keeps its own
fixed scratch array on each GPU.  These tests call that entry point through the
C ABI and check it against the workspace entry point, on two calls in a row
(the array keeps the previous call's contents, which must not leak into the
next call's result).  The file is named to run after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from mla_decode_attention_08_gb300 import binding
from mla_decode_attention_08_gb300.inputs import make_from_lengths

from .gpu_util import ATOL, RTOL, DeviceCase

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 12 * 1024 * 1024


@pytest.fixture(scope="module")
def lib(built_library):
    return binding.load_library(built_library)


def test_static_scratch_matches_workspace_entry_point(lib):
    # Split rows (partials and the combine stage), a whole row, an empty row, paged cache.
    inp = make_from_lengths([300, 1000, 17, 0, 4500], seed=91, paged=True)
    dev = DeviceCase(inp)
    plan = binding.mla_decode_plan(inp.batch, inp.max_kv_len, 7)
    assert plan.ws_bytes <= STATIC_SCRATCH_BYTES
    want, err, _, _ = dev.run(plan=plan)
    assert err == 0
    for _ in range(2):
        out = torch.full_like(dev.out, float("nan"))
        binding.mla_decode_fwd_static_scratch(dev.q, dev.kv_codes, dev.kv_scale, dev.qo_indptr,
                                              dev.kv_indptr, out, plan=plan,
                                              kv_indices=dev.kv_indices)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.isfinite(got).all()
        assert np.all(np.abs(got - want) <= ATOL + RTOL * np.abs(want))


def test_static_scratch_rejects_plans_beyond_its_size(lib):
    big = binding.mla_decode_plan(2_000_000, 8192, 152)
    assert big.ws_bytes > STATIC_SCRATCH_BYTES
    status = lib.mla_decode_fwd_static_scratch(None, None, None, None, None, None, None,
                                               ctypes.byref(big), None, 0, 1)
    assert status == 3  # MLA_ERR_WORKSPACE_TOO_SMALL, before anything is launched
