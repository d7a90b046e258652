"""The decode step under the stream semantics the C ABI states: calls with
their own workspaces run concurrently on different streams, the output is
deterministic for a fixed plan, and the step can be captured once into a CUDA
graph and replayed while the query and the cache lengths change between steps
(the schedule is derived on the device from kv_indptr, so nothing the host
computed goes stale)."""
import numpy as np
import pytest
import torch

from mla_decode_attention_08_gb300 import binding
from mla_decode_attention_08_gb300.inputs import Inputs, f32_to_bf16_bits, make_from_lengths

from .gpu_util import DeviceCase, OracleCase, assert_close, bits_to_bf16, num_sms

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    binding.load_library(built_library)


def fwd(dev, plan, ws, stream=None, kv_indptr=None, kv_indices="case"):
    binding.mla_decode_fwd(dev.q, dev.kv_codes, dev.kv_scale, dev.qo_indptr,
                           dev.kv_indptr if kv_indptr is None else kv_indptr, dev.out, stream,
                           plan=plan, workspace=ws,
                           kv_indices=dev.kv_indices if kv_indices == "case" else kv_indices)


def test_concurrent_calls_on_two_streams_with_their_own_workspaces():
    """Two problems decoded at once on two streams give, bit for bit, what each
    gives alone, and so does every repeat."""
    cases = [DeviceCase(make_from_lengths([3000, 17, 800, 129, 0, 4096], seed=77, paged=True)),
             DeviceCase(make_from_lengths(list(range(1, 600, 7)), seed=78))]
    alone = []
    for c in cases:
        out, err, _, _ = c.run()
        assert err == 0
        alone.append(out)
    plans = [binding.mla_decode_plan(c.inp.batch, c.inp.max_kv_len, num_sms()) for c in cases]
    wss = [binding.new_workspace(p) for p in plans]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(3):
        for c in cases:
            c.out.fill_(float("nan"))
        torch.cuda.synchronize()
        for c, p, ws, s in zip(cases, plans, wss, streams):
            fwd(c, p, ws, s)
        torch.cuda.synchronize()
        for c, ws, want in zip(cases, wss, alone):
            assert binding.mla_decode_read_error(ws) == 0
            assert np.array_equal(c.out.float().cpu().numpy(), want)


@pytest.mark.parametrize("paged", [False, True])
def test_graph_replay_follows_new_queries_and_lengths(paged):
    """Capture one call, then replay it as a decode loop would: the same
    inputs give the eager bits; a new query with every row one token longer
    (same buffers, kv_indptr rewritten in place) gives the oracle's output for
    the new problem."""
    grown = np.array([1001, 4, 130, 1, 2501, 257])
    base = make_from_lengths(grown, seed=83, paged=paged)   # cache and page table of the longer step
    n_rows = int(grown.sum())

    def step(lengths, q_seed):
        ind = np.zeros(len(lengths) + 1, np.int32)
        np.cumsum(lengths, out=ind[1:])
        q = np.random.default_rng(q_seed).standard_normal((len(lengths), 16, 576), dtype=np.float32)
        idx = None if base.kv_indices is None else base.kv_indices[:int(ind[-1])]
        return Inputs(q_bits=f32_to_bf16_bits(q), kv_bits=base.kv_bits, qo_indptr=base.qo_indptr,
                      kv_indptr=ind, kv_indices=idx, max_kv_len=base.max_kv_len)

    first, second = step(grown - 1, 84), step(grown, 85)
    dev = DeviceCase(base)                 # the cache (all rows) and the page table's buffer
    assert dev.kv_codes.shape[0] == n_rows
    plan = binding.mla_decode_plan(base.batch, base.max_kv_len, num_sms())
    ws = binding.new_workspace(plan)
    kv_indptr = torch.from_numpy(first.kv_indptr).cuda()
    dev.q.copy_(bits_to_bf16(first.q_bits))
    fwd(dev, plan, ws, kv_indptr=kv_indptr)
    torch.cuda.synchronize()
    assert binding.mla_decode_read_error(ws) == 0
    eager = dev.out.float().cpu().numpy()
    assert_close(eager, OracleCase(first).reference())

    g = torch.cuda.CUDAGraph()
    dev.out.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fwd(dev, plan, ws, kv_indptr=kv_indptr)
    g.replay()
    torch.cuda.synchronize()
    assert binding.mla_decode_read_error(ws) == 0
    assert np.array_equal(dev.out.float().cpu().numpy(), eager)

    dev.q.copy_(bits_to_bf16(second.q_bits))
    kv_indptr.copy_(torch.from_numpy(second.kv_indptr))
    dev.out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert binding.mla_decode_read_error(ws) == 0
    assert_close(dev.out.float().cpu().numpy(), OracleCase(second).reference())
