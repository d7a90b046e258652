"""Parity of the CUDA path (through the C ABI) with the float64 oracle."""
import numpy as np
import pytest
import torch

from mla_decode_attention_08_gb300 import binding
from mla_decode_attention_08_gb300.inputs import WORKLOADS, make_from_lengths, make_inputs
from oracle.fp8 import e4m3fn_decode
from oracle.schedule import plan_grid, worker_table
from oracle.schedule import schedule as oracle_schedule

from .gpu_util import DeviceCase, OracleCase, assert_close, num_sms

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    binding.load_library(built_library)


# ------------------------------------------------------------------ small shapes
SMALL = [
    ("one_tile", [128], False),
    ("tails", [1, 127, 128, 129, 255, 257, 1000], False),
    ("empty_rows", [0, 300, 0, 1, 0], False),
    ("paged_tails", [3, 129, 700, 64, 1], True),
    ("long_row", [5000], False),
    ("many_rows", list(range(1, 400, 13)), True),
]


@pytest.mark.parametrize("name,lengths,paged", SMALL, ids=[s[0] for s in SMALL])
@pytest.mark.parametrize("sms", [1, 5, None])
@pytest.mark.parametrize("persistent", [False, True], ids=["planned", "persistent"])
def test_small_shapes(name, lengths, paged, sms, persistent):
    inp = make_from_lengths(lengths, seed=777 + len(lengths), paged=paged)
    dev = DeviceCase(inp)
    gpu, err, plan, ws = dev.run(sms=sms, persistent=persistent)
    assert err == 0
    ref = OracleCase(inp).reference()
    assert_close(gpu, ref)
    if plan.cluster and not paged:
        return  # the cluster split writes no persistent schedule (tests/test_gpu_cluster.py)
    # the schedule the kernel used, bit for bit
    views = binding.workspace_views(plan, ws)
    assert np.array_equal(views["workers"].cpu().numpy(), worker_table(inp.kv_indptr, plan.grid))
    assert views["prefix"].cpu().numpy().tolist() == oracle_schedule(inp.kv_indptr, plan.grid)["prefix"]
    assert np.array_equal(views["jobs"].cpu().numpy(), expected_jobs(inp, plan.grid))


def expected_jobs(inp, grid):
    """Combine job per worker from the oracle's schedule: a split row is
    combined by the entry of its second worker (the first worker boundary inside
    it), holding (query row, first worker, last worker, first worker's slot)."""
    sch = oracle_schedule(inp.kv_indptr, grid)
    jobs = np.zeros((grid, 4), dtype=np.int64)
    jobs[:, 0] = -1
    first_slot = {(sg["worker"], sg["row"]): sg["slot"] for sg in sch["segments"]}
    for b, ws in sch["covers"].items():
        if len(ws) > 1:
            jobs[ws[1]] = (int(inp.qo_indptr[b]), ws[0], ws[-1], first_slot[(ws[0], b)])
    return jobs


def test_grid_larger_than_tile_count():
    # 3 tiles over a grid of 8: most workers have empty ranges.
    inp = make_from_lengths([130, 1, 0, 120], seed=5)
    gpu, err, plan, _ = DeviceCase(inp).run(plan=binding.mla_decode_plan(4, 8192, 8))
    assert plan.grid == 8 and err == 0
    assert_close(gpu, OracleCase(inp).reference())


def test_all_rows_empty():
    inp = make_from_lengths([0, 0, 0], seed=6, max_kv_len=64)
    gpu, err, _, _ = DeviceCase(inp).run()
    assert err == 0 and np.all(gpu == 0)


def test_sharp_scores_exercise_rescaling():
    inp = make_from_lengths([2000, 517, 4096], seed=8)
    inp.q_bits = (inp.q_bits.view(np.uint16).astype(np.uint32) + (4 << 7)).astype(np.uint16)  # q x 16
    gpu, err, _, _ = DeviceCase(inp).run(sms=3)
    assert err == 0
    assert_close(gpu, OracleCase(inp).reference())


def test_one_token_rows_return_v():
    inp = make_from_lengths([1, 1, 1], seed=9, paged=True)
    dev = DeviceCase(inp)
    gpu, err, _, _ = dev.run()
    assert err == 0
    codes = dev.kv_codes.cpu().numpy()
    scale = np.float32(dev.kv_scale.item())
    for b in range(3):
        slot = inp.kv_indices[b]
        v32 = (e4m3fn_decode(codes[slot, :512]).astype(np.float32) * scale).astype(np.float32)
        want = torch.from_numpy(v32).to(torch.bfloat16).float().numpy()
        assert np.array_equal(gpu[b], np.broadcast_to(want, (16, 512))), b


def test_constant_scores_return_mean_of_v():
    inp = make_from_lengths([300, 77], seed=10)
    q = inp.q_bits.reshape(2, 16, 576).copy()
    q[:, :, :512] = 0
    inp.q_bits = q
    kv = inp.kv_bits.copy()
    kv[:, 512:] = kv[0, 512:]
    inp.kv_bits = kv
    dev = DeviceCase(inp)
    gpu, err, _, _ = dev.run(sms=4)
    assert err == 0
    codes = dev.kv_codes.cpu().numpy().astype(np.uint8)
    scale = float(dev.kv_scale.item())
    for b, (j0, j1) in enumerate([(0, 300), (300, 377)]):
        mean_v = (e4m3fn_decode(codes[j0:j1, :512]) * scale).mean(axis=0)
        np.testing.assert_allclose(gpu[b], np.broadcast_to(mean_v, (16, 512)), rtol=1e-2, atol=1e-3)


def test_permuted_cache_matches_contiguous():
    inp = make_from_lengths([900, 33, 1500], seed=11)
    a, err_a, _, _ = DeviceCase(inp).run(sms=7)
    perm = np.random.default_rng(3).permutation(inp.kv_bits.shape[0])
    paged = make_from_lengths([900, 33, 1500], seed=11)
    paged.kv_bits = np.empty_like(inp.kv_bits)
    paged.kv_bits[perm] = inp.kv_bits          # token j now lives in cache row perm[j]
    paged.kv_indices = perm.astype(np.int32)
    b, err_b, _, _ = DeviceCase(paged).run(sms=7)
    assert err_a == 0 and err_b == 0
    np.testing.assert_allclose(a, b, rtol=1e-2, atol=2e-3)


def test_split_count_invariance():
    inp = make_from_lengths([3000, 1024, 17], seed=12, paged=True)
    dev = DeviceCase(inp)
    ref = OracleCase(inp).reference()
    for sms in (1, 2, 3, 9, 40, 152):
        gpu, err, _, _ = dev.run(sms=sms)
        assert err == 0
        assert_close(gpu, ref)


# ------------------------------------------------------------------ codec
def test_fp8_quantize_bit_exact():
    inp = make_from_lengths([3000, 1], seed=13)
    dev, ora = DeviceCase(inp), OracleCase(inp)
    assert np.float32(dev.kv_scale.item()) == ora.scale
    assert np.array_equal(dev.kv_codes.cpu().numpy(), ora.codes())


def test_fp8_quantize_every_bf16_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 7) & 0xFF
    bits = bits[exp != 0xFF]                   # finite values only
    src = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    codes = torch.empty(bits.size, dtype=torch.uint8, device="cuda")
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    binding.mla_fp8_quantize_per_tensor(src, codes, scale, torch.empty(16, dtype=torch.uint8, device="cuda"))
    from mla_decode_attention_08_gb300.inputs import bf16_bits_to_f32
    from oracle.quant import quantize_per_tensor
    want_codes, want_scale = quantize_per_tensor(bf16_bits_to_f32(bits))
    assert np.float32(scale.item()) == want_scale
    assert np.array_equal(codes.cpu().numpy(), want_codes)


# ------------------------------------------------------------------ host-made input errors
def test_bad_query_row_is_flagged_and_skipped():
    inp = make_from_lengths([200, 300, 100], seed=14)
    dev = DeviceCase(inp)
    dev.qo_indptr = torch.tensor([0, 2, 2, 3], dtype=torch.int32, device="cuda")
    dev.out.fill_(7.0)
    gpu, err, _, _ = dev.run(sms=2)
    assert err & 1
    ref = OracleCase(make_from_lengths([200, 300, 100], seed=14)).reference()
    assert_close(gpu[2:3], ref[2:3])


def test_decreasing_kv_indptr_gives_zeros_and_flag():
    inp = make_from_lengths([200, 300], seed=15)
    dev = DeviceCase(inp)
    dev.kv_indptr = torch.tensor([0, 300, 200], dtype=torch.int32, device="cuda")
    gpu, err, _, _ = dev.run()
    assert err & 2 and np.all(gpu == 0)


def test_out_of_range_page_index_is_flagged():
    inp = make_from_lengths([50, 60], seed=16, paged=True)
    dev = DeviceCase(inp)
    bad = dev.kv_indices.clone()
    bad[5] = 10 ** 6
    dev.kv_indices = bad
    _, err, _, _ = dev.run()
    assert err & 4


# ------------------------------------------------------------------ the benchmark workloads
def _sample_rows(inp, plan, k=6):
    """First, last, and rows split across workers (both kinds of output path)."""
    sch = oracle_schedule(inp.kv_indptr, plan.grid)
    split = [b for b, ws in sch["covers"].items() if len(ws) > 1]
    whole = [b for b, ws in sch["covers"].items() if len(ws) == 1]
    rows = {0, inp.batch - 1}
    rows.update(split[:k // 2])
    rows.update(whole[:k // 2])
    return sorted(rows)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_parity(name):
    inp = make_inputs(name)
    dev = DeviceCase(inp)
    gpu, err, plan, ws = dev.run()
    assert err == 0
    assert np.isfinite(gpu).all()
    ora = OracleCase(inp)
    full = inp.batch * inp.max_kv_len <= 32 * 1024
    rows = None if full else _sample_rows(inp, plan)
    ref = ora.reference(rows)
    n = inp.qo_len  # output rows of batch row b: n b .. n b + n - 1
    toks = None if rows is None else [n * b + i for b in rows for i in range(n)]
    st = assert_close(gpu, ref, toks)
    print(name, "grid", plan.grid, st)
    # the cache codes the kernel read, bit-exact on the sampled cache rows
    check = np.arange(min(4096, inp.kv_bits.shape[0]))
    assert np.float32(dev.kv_scale.item()) == ora.scale
    assert np.array_equal(dev.kv_codes[: check.size].cpu().numpy(), ora.codes(check))
    if plan.cluster == 0 or inp.kv_indices is not None:
        views = binding.workspace_views(plan, ws)
        assert np.array_equal(views["workers"].cpu().numpy(), worker_table(inp.kv_indptr, plan.grid))
    # rows of three or four query tokens take two sibling CTAs per worker
    sms = num_sms() if inp.qo_len <= 2 else num_sms() // 2
    assert plan.grid == plan_grid(inp.batch, inp.max_kv_len, sms)


# ------------------------------------------------------------------ split partials
def test_split_partials_and_lse_match_oracle():
    """Stage 1's normalised partial and base-2 log-sum-exp of every split segment
    against the oracle's split_partial over the same token range (the combine
    inputs, checked before the combine can hide an error in one of them)."""
    from oracle.attention import _row_tokens, dequant_rows, split_partial

    from .gpu_util import ATOL, RTOL

    inp = make_from_lengths([300, 1000, 17, 4500, 129, 0, 2000], seed=4242, paged=True)
    dev = DeviceCase(inp)
    plan = binding.mla_decode_plan(inp.batch, inp.max_kv_len, 7)
    ws = binding.new_workspace(plan)
    # The two-kernel form writes every piece's partial (the fused call lets the
    # worker that completes a row skip its own).
    binding.mla_decode_stage1(dev.q, dev.kv_codes, dev.kv_scale, dev.qo_indptr, dev.kv_indptr,
                              dev.out, plan=plan, workspace=ws, kv_indices=dev.kv_indices)
    binding.mla_decode_stage2(dev.qo_indptr, dev.out, plan=plan, workspace=ws)
    torch.cuda.synchronize()
    assert binding.mla_decode_read_error(ws) == 0
    gpu = dev.out.float().cpu().numpy()
    views = binding.workspace_views(plan, ws)
    part = views["partial"].float().cpu().numpy()[:, 0]  # [slot][head][dim] (one query token)
    lse = views["lse"].cpu().numpy()[:, 0]       # [slot][head]
    orc = OracleCase(inp)
    codes = orc.codes()
    checked = 0
    for s in oracle_schedule(inp.kv_indptr, plan.grid)["segments"]:
        if not s["split"]:
            continue
        b = s["row"]
        length = int(inp.kv_indptr[b + 1] - inp.kv_indptr[b])
        j0, j1 = s["tile_begin"] * 128, min(length, s["tile_end"] * 128)
        slots = _row_tokens(b, inp.kv_indptr, inp.kv_indices)[j0:j1]
        o, l = split_partial(orc.q[int(inp.qo_indptr[b])], dequant_rows(codes, orc.scale, slots))
        got = part[s["slot"]].astype(np.float64)
        assert np.all(np.abs(got - o) <= ATOL + RTOL * np.abs(o)), (s, np.abs(got - o).max())
        assert np.all(np.abs(lse[s["slot"]] - l) <= 2e-2), (s, lse[s["slot"]], l)
        checked += 1
    assert checked >= 6
    assert_close(gpu, orc.reference())


# ------------------------------------------------------------------ combine edge cases
COMBINE_CASES = [
    ("split_paged", [300, 1000, 17, 4500, 129, 0, 2000], True, 7),
    ("many_pieces", [4000, 1, 4000], False, 40),  # rows split over up to ~30 workers
    ("empty_workers", [130, 1, 0, 120], False, 8),  # grid larger than the tile count
    ("all_empty", [0, 0, 0], False, 5),
    ("zero_rows_between_splits", [0, 900, 0, 0, 700, 0], True, 11),
]


@pytest.mark.parametrize("qo_len", [1, 2, 3])
@pytest.mark.parametrize("name,lengths,paged,sms", COMBINE_CASES, ids=[c[0] for c in COMBINE_CASES])
def test_combine_edge_cases_and_separate_stages(name, lengths, paged, sms, qo_len):
    """Rows split over many workers, workers with no tiles, rows without cached
    tokens, with one to three query tokens per row (stage 2's four- and
    eight-head kernels, sibling CTAs): mla_decode_fwd matches the oracle, and
    launching its two kernels through mla_decode_stage1 / mla_decode_stage2
    gives the same bits."""
    inp = make_from_lengths(lengths, seed=99 + len(lengths), paged=paged, max_kv_len=max(max(lengths), 1),
                            qo_len=qo_len)
    dev = DeviceCase(inp)
    plan = binding.mla_decode_plan(inp.batch, inp.max_kv_len, sms, qo_len=qo_len)
    ws = binding.new_workspace(plan)
    dev.out.fill_(float("nan"))
    gpu, err, _, _ = dev.run(plan=plan, workspace=ws)
    assert err == 0
    assert_close(gpu, OracleCase(inp).reference())
    out2 = torch.full_like(dev.out, float("nan"))
    binding.mla_decode_stage1(dev.q, dev.kv_codes, dev.kv_scale, dev.qo_indptr, dev.kv_indptr,
                              out2, plan=plan, workspace=ws, kv_indices=dev.kv_indices)
    binding.mla_decode_stage2(dev.qo_indptr, out2, plan=plan, workspace=ws)
    torch.cuda.synchronize()
    assert binding.mla_decode_read_error(ws) == 0
    assert np.array_equal(out2.float().cpu().numpy(), gpu)


# ------------------------------------------------------------------ larger and randomised shapes
def test_more_rows_than_prologue_threads():
    """1000 rows: each prologue thread scans several rows (the rows-per-thread
    path of the block scan), with empty and one-token rows among them."""
    rng = np.random.default_rng(71)
    lengths = rng.integers(0, 300, size=1000)
    lengths[rng.random(1000) < 0.05] = 0
    lengths[rng.random(1000) < 0.05] = 1
    for paged in (False, True):
        inp = make_from_lengths(lengths, seed=72 + paged, paged=paged)
        dev = DeviceCase(inp)
        gpu, err, plan, ws = dev.run()
        assert err == 0
        assert_close(gpu, OracleCase(inp).reference())
        views = binding.workspace_views(plan, ws)
        assert np.array_equal(views["workers"].cpu().numpy(), worker_table(inp.kv_indptr, plan.grid))
        assert np.array_equal(views["jobs"].cpu().numpy(), expected_jobs(inp, plan.grid))


def test_one_very_long_row_among_short_ones():
    """A 100,000-token row split over every worker next to short rows."""
    inp = make_from_lengths([100_000, 3, 0, 129], seed=73)
    dev = DeviceCase(inp)
    gpu, err, plan, _ = dev.run()
    assert err == 0 and plan.grid == plan_grid(inp.batch, inp.max_kv_len, num_sms()) >= 140
    assert_close(gpu, OracleCase(inp).reference())


@pytest.mark.parametrize("seed", range(8))
def test_randomised_shapes(seed):
    """Random batch, lengths (with empty rows), page table, query tokens per
    row (1 to 4) and grid, against the oracle."""
    rng = np.random.default_rng(9000 + seed)
    batch = int(rng.integers(1, 300))
    lengths = rng.integers(0, int(rng.integers(2, 1500)), size=batch)
    lengths[rng.random(batch) < 0.1] = 0
    qo_len = int(rng.integers(1, 5))
    paged = bool(rng.random() < 0.5)
    sms = int(rng.integers(1, 153))
    inp = make_from_lengths(lengths, seed=9100 + seed, paged=paged, qo_len=qo_len)
    dev = DeviceCase(inp)
    dev.out.fill_(float("nan"))
    gpu, err, plan, _ = dev.run(sms=sms)
    assert err == 0, (batch, qo_len, paged, sms)
    assert_close(gpu, OracleCase(inp).reference())
