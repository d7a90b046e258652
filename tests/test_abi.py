"""The C ABI on the CPU: exports, plan, host schedule vs the oracle, host-side errors."""
import ctypes
import os
import re

import numpy as np
import pytest

from mla_decode_attention_08_gb300 import binding
from mla_decode_attention_08_gb300.build import ROOT
from oracle.schedule import plan_cluster, plan_grid, worker_table
from oracle.schedule import schedule as oracle_schedule

HEADER = os.path.join(ROOT, "include", "mla_decode.h")


@pytest.fixture(scope="module")
def lib(built_library):
    return binding.load_library(built_library)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert "mla_decode_fwd" in names and len(names) >= 9
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(binding.SIGNATURES)


def test_abi_version_and_status_strings(lib):
    assert lib.mla_decode_abi_version() == 5
    for s in range(5):
        assert lib.mla_status_string(s)


@pytest.mark.parametrize("batch,max_len,sms", [(4, 1024, 152), (32, 1024, 152), (64, 8192, 152),
                                               (256, 8192, 152), (128, 8192, 148), (1, 0, 152),
                                               (7, 129, 10)])
def test_plan_matches_oracle_grid(lib, batch, max_len, sms):
    plan = binding.mla_decode_plan(batch, max_len, sms)
    assert plan.grid == plan_grid(batch, max_len, sms)
    assert plan.tile_tokens == 128 and plan.batch == batch
    g = plan.grid
    assert plan.ws_prefix_offset >= 4 and plan.ws_prefix_offset % 256 == 0
    assert plan.ws_workers_offset >= plan.ws_prefix_offset + 4 * (batch + 1)
    assert plan.ws_lse_offset >= plan.ws_workers_offset + 32 * g
    assert plan.ws_partial_offset >= plan.ws_lse_offset + 4 * 32 * g
    assert plan.ws_bytes >= plan.ws_partial_offset + 2 * 2 * g * 16 * 512
    assert all(o % 256 == 0 for o in (plan.ws_workers_offset, plan.ws_lse_offset,
                                      plan.ws_partial_offset, plan.ws_bytes))


@pytest.mark.parametrize("seed", range(12))
def test_host_schedule_bit_exact_vs_oracle(lib, seed):
    rng = np.random.default_rng(100 + seed)
    batch = int(rng.integers(1, 300))
    lengths = rng.integers(0, int(rng.integers(1, 9000)) + 1, size=batch)
    lengths[rng.random(batch) < 0.15] = 0
    indptr = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    grid = int(rng.integers(1, 200))
    workers, prefix = binding.mla_decode_schedule_host(indptr, grid)
    assert np.array_equal(workers, worker_table(indptr, grid))
    assert prefix.tolist() == oracle_schedule(indptr, grid)["prefix"]


def test_host_schedule_workload_shapes(lib):
    for batch, length in [(4, 1024), (32, 1024), (64, 8192), (256, 8192)]:
        indptr = np.arange(batch + 1, dtype=np.int32) * length
        grid = plan_grid(batch, length, 152)
        workers, _ = binding.mla_decode_schedule_host(indptr, grid)
        assert np.array_equal(workers, worker_table(indptr, grid))


def test_host_side_argument_errors(lib):
    plan = binding.mla_decode_plan(4, 1024, 152)
    p = ctypes.byref(plan)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the checks fail first
    assert lib.mla_decode_fwd(None, fake, fake, fake, fake, fake, None, p, None, 0, 4096,
                              fake, plan.ws_bytes) == 1
    bad = binding.mla_plan_t.from_buffer_copy(plan)
    bad.abi_version = 99
    assert lib.mla_decode_fwd(fake, fake, fake, fake, fake, fake, None, ctypes.byref(bad), None,
                              0, 4096, fake, plan.ws_bytes) == 1
    # misaligned q
    assert lib.mla_decode_fwd(ctypes.c_void_p((1 << 20) + 2), fake, fake, fake, fake, fake, None,
                              p, None, 0, 4096, fake, plan.ws_bytes) == 1
    # kv_rows out of range
    assert lib.mla_decode_fwd(fake, fake, fake, fake, fake, fake, None, p, None, 0, 0,
                              fake, plan.ws_bytes) == 1
    # workspace too small
    assert lib.mla_decode_fwd(fake, fake, fake, fake, fake, fake, None, p, None, 0, 4096,
                              fake, plan.ws_bytes - 1) == 3
    assert lib.mla_decode_plan(0, 10, 152, ctypes.byref(binding.mla_plan_t())) == 1
    assert lib.mla_decode_plan(3, -1, 152, ctypes.byref(binding.mla_plan_t())) == 1
    assert lib.mla_decode_schedule_host(None, 3, 3, None, None) == 1
    # the bf16-cache entry points take no scale and check the same arguments
    assert lib.mla_decode_fwd_bf16kv(fake, fake, fake, fake, fake, None, p, None, 0, 4096,
                                     fake, plan.ws_bytes - 1) == 3
    assert lib.mla_decode_fwd_bf16kv(fake, None, fake, fake, fake, None, p, None, 0, 4096,
                                     fake, plan.ws_bytes) == 1
    assert lib.mla_decode_stage1_bf16kv(fake, fake, fake, fake, ctypes.c_void_p((1 << 20) + 8),
                                        None, p, None, 0, 4096, fake, plan.ws_bytes) == 1
    # a bf16 cache is read contiguously: a page table is unsupported
    assert lib.mla_decode_fwd_bf16kv(fake, fake, fake, fake, fake, None, p, fake, 4096, 4096,
                                     fake, plan.ws_bytes) == 2


def test_mxfp4_host_side_argument_errors(lib):
    plan = binding.mla_decode_plan(4, 1024, 152)
    p = ctypes.byref(plan)
    fake = ctypes.c_void_p(1 << 20)
    ws = plan.ws_bytes

    def fwd(*, scales=fake, bias=0, rows=4096, plan_ref=p, ws_bytes=ws, fn=lib.mla_decode_fwd_mxfp4):
        return fn(fake, fake, scales, bias, fake, fake, fake, None, plan_ref, rows, fake, ws_bytes)

    assert fwd(scales=None) == 1
    assert fwd(scales=ctypes.c_void_p((1 << 20) + 2)) == 1          # scales not 16-byte aligned
    assert fwd(bias=101) == 1 and fwd(bias=-101) == 1
    assert fwd(rows=119_304_420) == 1                               # scale bytes past 2^31
    assert fwd(rows=0) == 1
    assert fwd(ws_bytes=ws - 1) == 3
    assert fwd(fn=lib.mla_decode_stage1_mxfp4, ws_bytes=ws - 1) == 3
    plan2 = binding.mla_decode_plan(4, 1024, 152, qo_len=2)
    assert fwd(plan_ref=ctypes.byref(plan2), ws_bytes=plan2.ws_bytes) == 2  # one query token only
    assert lib.mla_mxfp4_quantize(None, 4, fake, fake, None) == 1
    assert lib.mla_mxfp4_quantize(fake, 0, fake, fake, None) == 1
    assert lib.mla_mxfp4_quantize(fake, 4, ctypes.c_void_p((1 << 20) + 4), fake, None) == 1


def test_binding_refuses_cpu_tensors(lib):
    import torch
    plan = binding.mla_decode_plan(1, 128, 152)
    q = torch.zeros(1, 16, 576, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        binding.mla_decode_fwd(q, q, q, q, q, q, plan=plan, workspace=q)


@pytest.mark.parametrize("qo_len", [1, 2, 3, 4])
def test_plan_mtp_sizes_the_partials_by_query_tokens(lib, qo_len):
    plan = binding.mla_decode_plan(64, 8192, 152, qo_len=qo_len)
    # rows of three or four tokens take two sibling CTAs per worker
    workers = plan_grid(64, 8192, 152 if qo_len <= 2 else 76)
    assert plan.qo_len == qo_len and plan.grid == workers
    g = plan.grid
    assert plan.ws_partial_offset >= plan.ws_lse_offset + 4 * 2 * g * qo_len * 16
    assert plan.ws_bytes >= plan.ws_partial_offset + 2 * 2 * g * qo_len * 16 * 512


def test_plan_mtp_rejects_unsupported_token_counts(lib):
    plan = binding.mla_plan_t()
    for n in (0, 5, 8, -1):
        assert lib.mla_decode_plan_mtp(8, n, 1024, 152, ctypes.byref(plan)) == 1


@pytest.mark.parametrize("kv", [
    lambda torch: torch.zeros((8, 576), dtype=torch.bfloat16),   # a bf16 cache
    lambda torch: torch.zeros((8, 576), dtype=torch.float32),
    lambda torch: torch.zeros((8, 288), dtype=torch.uint8),      # MXFP4 elements
])
def test_binding_refuses_a_cache_that_is_not_e4m3(lib, kv):
    torch = pytest.importorskip("torch")
    cache = kv(torch)
    q = torch.zeros((1, 16, 576), dtype=torch.bfloat16)
    ind = torch.zeros(2, dtype=torch.int32)
    out = torch.zeros((1, 16, 512), dtype=torch.bfloat16)
    plan = binding.mla_decode_plan(1, 8, 152)
    err = TypeError if cache.dtype != torch.uint8 else ValueError
    with pytest.raises(err):
        binding.mla_decode_fwd(q, cache, torch.ones(1), ind, ind, out, plan=plan,
                               workspace=torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(err):
        binding.mla_decode_fwd_static_scratch(q, cache, torch.ones(1), ind, ind, out, plan=plan)


@pytest.mark.parametrize("qo_len", [1, 2])
def test_plan_cluster_matches_oracle(lib, qo_len):
    for sms in (152, 148, 40, 7, 1):
        for batch in (1, 2, 3, 4, 5, 8, 15, 16, 32, 33, 34, 64, 76, 77, 256):
            for max_len in (0, 1, 128, 129, 300, 512, 1024, 2048, 4096, 8192):
                plan = binding.mla_decode_plan(batch, max_len, sms, qo_len=qo_len)
                assert plan.cluster == plan_cluster(batch, qo_len, max_len, sms), (batch, max_len, sms)
                assert plan.grid == plan_grid(batch, max_len, sms if qo_len <= 2 else sms // 2)


def test_trace_table_sizes_match_the_header():
    """The binding sizes the host arrays of mla_decode_trace_read from the
    header's MLA_TRACE_* constants; a drift would make the call write past
    them.  The trace summariser's event indices stay inside the table."""
    text = open(os.path.join(ROOT, "include", "mla_decode.h")).read()
    want = {name: int(re.search(rf"#define {name} (\d+)", text).group(1))
            for name in ("MLA_TRACE_CTAS", "MLA_TRACE_EVENTS", "MLA_TRACE2_BLOCKS")}
    assert (binding.TRACE_CTAS, binding.TRACE_EVENTS, binding.TRACE2_BLOCKS) == (
        want["MLA_TRACE_CTAS"], want["MLA_TRACE_EVENTS"], want["MLA_TRACE2_BLOCKS"])
    from mla_decode_attention_08_gb300 import trace
    assert all(0 < ev < want["MLA_TRACE_EVENTS"] for ev, _ in trace.EVENTS)
