"""CUDA path (through the C ABI) against the oracle.

Scores within |err| <= 1e-3 + 2e-3 |ref|; the fused first-digit histogram equal
to a count of the stored scores; selection on identical scores bit-exact; the
fused launch equal to selection on its own scores, and within the allowed-swap
rule of the oracle's end-to-end selection."""
import zlib

import numpy as np
import pytest
import torch

import workloads
from tests import gpu_util, parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    import sparse_attention_indexer_launch_gb300 as lib
    return lib


SMALL = [
    # name, lengths, rows per request, kv, extra build args
    ("one_key", [1], [1], "e4m3", {}),
    ("ragged_e4m3", [63, 64, 65, 127, 129, 300, 1000, 2500], [1, 2, 3, 4, 1, 2, 3, 4], "e4m3", {}),
    ("ragged_bf16", [63, 64, 65, 127, 129, 300, 1000, 2500], [1, 2, 3, 4, 1, 2, 3, 4], "bf16", {}),
    ("chain_8_rows", [3000], [8], "e4m3", {}),
    ("mixture_dups", [5000, 4097], [4, 2], "e4m3", {"key_dist": "mixture", "dup_frac": 0.02}),
    ("rows_out_of_order", [700, 900], [3, 2], "e4m3", {"row_order": [3, 0, 4, 1, 2]}),
    ("around_k", [2047, 2048, 2049, 4096], [1, 1, 1, 1], "e4m3", {}),
    ("around_k_bf16", [2047, 2048, 2049, 4100], [2, 1, 3, 1], "bf16", {}),
    # 600 rows in 150 requests: the plan's passes and group records span several blocks of rows
    ("many_rows", [(i * 97) % 2900 + 64 for i in range(150)], [4] * 150, "e4m3", {}),
    # more rows than one block of the planning pass: the plan's group records go
    # through global memory between its two passes
    ("rows_over_1024", [(i * 53) % 600 + 1 for i in range(280)], [4] * 280, "e4m3", {}),
    # one long request among many short ones: most CTAs of the rows x slices
    # selection grid find their slice past the row's end
    ("long_among_short", [60000] + [(i * 37) % 2000 + 1 for i in range(99)], [2] * 100, "e4m3", {}),
]


@pytest.mark.parametrize("name,lengths,rows,kv,extra", SMALL, ids=[c[0] for c in SMALL])
def test_small_problems(lib, orc, name, lengths, rows, kv, extra):
    prob = workloads.build(name, lengths, rows, kv, seed=zlib.crc32(name.encode()) % 1000, **extra)
    dp, scores, hist, st = gpu_util.run_score(lib, prob)
    assert st == lib.IDX_OK, lib.status_string(st)
    ref, _ = gpu_util.check_scores_vs_oracle(orc, prob, scores, hist)
    for K in (1, 7, 100, 2048):
        out = dp.topk(torch.from_numpy(scores).cuda(), K=K).cpu().numpy()
        gpu_util.check_selection(orc, out, scores, prob.row_bound, K)
        out2 = dp.topk(torch.from_numpy(scores).cuda(), hist=torch.from_numpy(hist.view(np.int32)).cuda(),
                       K=K).cpu().numpy()
        assert np.array_equal(out, out2), "histogram given vs computed"
    out = dp.launch().cpu().numpy()
    assert dp.status() == lib.IDX_OK
    gpu_util.check_selection(orc, out, scores, prob.row_bound, prob.K)
    O = orc.topk(ref.astype(np.float32), prob.row_bound, prob.K)
    parity.check_endtoend(out, ref, O, prob.row_bound, prob.K)


def test_zero_bound_rows_and_padding(lib, orc):
    prob = workloads.build("pad", [5, 3000], [2, 3], "e4m3", seed=3, bounds=[[0, 5], [0, 1, 2999]])
    dp, scores, hist, st = gpu_util.run_score(lib, prob)
    assert st == lib.IDX_OK
    gpu_util.check_scores_vs_oracle(orc, prob, scores, hist)
    out = dp.launch().cpu().numpy()
    assert np.all(out[0] == -1) and np.all(out[2] == -1)
    assert out[3, 0] == 0 and np.all(out[3, 1:] == -1)
    gpu_util.check_selection(orc, out, scores, prob.row_bound, prob.K)


def _equal_keys_problem(L, rows, zero=False):
    prob = workloads.build("equal", [L], [rows], "e4m3", seed=9)
    if zero:
        prob.k_cache[:] = 0
    else:
        prob.k_cache[:] = prob.k_cache[0, 0]
        prob.k_scale[:] = prob.k_scale[0, 0]
    return prob


@pytest.mark.parametrize("L,zero", [(3000, False), (10000, False), (20000, True)])
def test_all_equal_scores(lib, orc, L, zero):
    """Every score equal: the k-th value has thousands of ties (more than the
    candidate buffer for L >= 10000), and the lowest positions must win."""
    prob = _equal_keys_problem(L, 2, zero)
    dp, scores, hist, st = gpu_util.run_score(lib, prob)
    assert st == lib.IDX_OK
    gpu_util.check_scores_vs_oracle(orc, prob, scores, hist)
    out = dp.launch().cpu().numpy()
    gpu_util.check_selection(orc, out, scores, prob.row_bound, prob.K)
    b = prob.row_bound
    for r in range(prob.R):
        if len(np.unique(scores[r, :b[r]])) == 1:
            assert list(out[r]) == list(range(min(prob.K, b[r]))) + [-1] * (prob.K - min(prob.K, b[r]))


def test_two_value_scores(lib, orc):
    """Half the keys share one score, half another: the threshold bin is huge."""
    prob = workloads.build("two", [12000], [1], "e4m3", seed=10)
    pt = prob.page_table[0]
    for t in range(12000):
        src = (0, 0) if (t * 7919) % 2 else (0, 1)
        prob.k_cache[pt[t // 64], t % 64] = prob.k_cache[src]
        prob.k_scale[pt[t // 64], t % 64] = prob.k_scale[src]
    dp, scores, hist, st = gpu_util.run_score(lib, prob)
    gpu_util.check_scores_vs_oracle(orc, prob, scores, hist)
    out = dp.launch().cpu().numpy()
    gpu_util.check_selection(orc, out, scores, prob.row_bound, prob.K)


def test_negative_scales(lib, orc):
    """ReLU(s * d) with s < 0 keeps the negative products: the epilogue's other branch."""
    prob = workloads.build("neg", [1000], [2], "e4m3", seed=11)
    prob.k_scale[::3] *= -1.0
    dp, scores, hist, st = gpu_util.run_score(lib, prob)
    gpu_util.check_scores_vs_oracle(orc, prob, scores, hist)


def test_topk_given_adversarial_scores(lib, orc):
    """Selection alone on crafted scores: +-0, duplicates, one hot bin, negatives."""
    rng = np.random.default_rng(12)
    R, L = 6, 30000
    s = np.empty((R, L), np.float32)
    s[0] = rng.standard_normal(L)
    s[1] = 0.0
    s[1, ::2] = -0.0
    s[2] = rng.integers(-5, 5, L)
    s[3] = 1.0 + rng.integers(0, 8, L) * np.float32(2 ** -20)     # one exponent, few values
    s[4] = -np.abs(rng.standard_normal(L)) * 1e-30
    s[5] = rng.standard_normal(L) * 1e30
    bounds = np.array([L, L, L - 1, 2049, 2048, 17], np.int32)
    dev_s = torch.from_numpy(s).cuda()
    dev_b = torch.from_numpy(bounds).cuda()
    ws = lib.alloc_bytes(64 << 20)
    for K in (1, 2, 2047, 2048):
        out = torch.empty((R, K), dtype=torch.int32, device="cuda")
        lib.idx_topk(dev_s, L, dev_b, R, L, K, None, out, ws)
        gpu_util.check_selection(orc, out.cpu().numpy(), s, bounds, K)


def _check_whole_problem(lib, orc, prob, label):
    """Every visible score against the oracle, the fused histogram, exact selection
    on the GPU's scores (idx_topk and the fused launch), and the end-to-end rule."""
    dp, scores, hist, st = gpu_util.run_score(lib, prob)
    assert st == lib.IDX_OK, lib.status_string(st)
    R, b = prob.R, prob.row_bound
    # histogram: exact count of the stored scores
    assert np.array_equal(hist, orc.first_digit_hist(scores, b))
    # selection on identical scores
    out = dp.topk(torch.from_numpy(scores).cuda()).cpu().numpy()
    gpu_util.check_selection(orc, out, scores, b, prob.K)
    launch = dp.launch().cpu().numpy()
    assert dp.status() == lib.IDX_OK
    assert np.array_equal(launch, out), "fused launch differs from selection on its own scores"
    # scores: every visible score of the oracle (full rows)
    ref = orc.score(prob, ld=scores.shape[1])
    worst, where = parity.score_errors(scores, ref, b)
    assert worst <= 1.0, (worst, where)
    O = orc.topk(ref.astype(np.float32), b, prob.K)
    swaps = parity.check_endtoend(launch, ref, O, b, prob.K)
    print(f"{label}: worst score error {worst:.3f} of tolerance, {swaps} allowed swaps")


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4, "3b"])
def test_configs_full_size(lib, orc, cfg):
    """The five workloads at full size, in the launch configuration the benchmark
    times."""
    _check_whole_problem(lib, orc, workloads.make_config(cfg), f"cfg{cfg}")


LARGEST = [
    # 8,192 rows (2,048 requests of four): the plan's passes over many row blocks,
    # the selection over thousands of short rows
    ("rows_8192", [(i * 131) % 300 + 1 for i in range(2048)], [4] * 2048, "e4m3", {}),
    # a request of 1,572,864 keys (24,576 pages) read by a row and its neighbour
    ("keys_1_5m", [1_572_864], [2], "e4m3", {"key_dist": "mixture"}),
]


@pytest.mark.parametrize("name,lengths,rows,kv,extra", LARGEST, ids=[c[0] for c in LARGEST])
def test_largest_shapes(lib, orc, name, lengths, rows, kv, extra):
    """Shapes well past the benchmark's: many more rows, three times the keys."""
    prob = workloads.build(name, lengths, rows, kv, seed=zlib.crc32(name.encode()) % 1000, **extra)
    _check_whole_problem(lib, orc, prob, name)


def test_bad_page_id_is_reported(lib, orc):
    prob = workloads.build("badpage", [640], [2], "e4m3", seed=13)
    prob.page_table[0, 3] = prob.P + 5           # out of range
    dp = lib.DeviceProblem(prob)
    dp.score()
    assert dp.status() == lib.IDX_EDEVICE
    good = workloads.build("good", [640], [2], "e4m3", seed=13)
    dp2, scores, hist, st = gpu_util.run_score(lib, good)
    assert st == lib.IDX_OK


HINT_CASES = [
    # name, lengths, rows per request, kv, extra build args
    ("lone_rows_e4m3", [20000, 9000, 300, 64], [1, 1, 1, 1], "e4m3", {}),
    ("row_pairs_e4m3", [12000, 700, 5000], [2, 2, 1], "e4m3", {"key_dist": "mixture", "dup_frac": 0.02}),
    ("row_pairs_bf16", [9000, 4097], [2, 1], "bf16", {}),
    ("mixed_rows_e4m3", [6000, 3000, 2000, 129], [4, 1, 3, 2], "e4m3", {}),
    ("negative_scales", [3000, 1000], [1, 2], "e4m3", {"negate_every": 3}),
]


@pytest.mark.parametrize("name,lengths,rows,kv,extra", HINT_CASES, ids=[c[0] for c in HINT_CASES])
def test_rows_hint_never_changes_the_result(lib, orc, name, lengths, rows, kv, extra):
    """idx_problem.rows_hint picks the scan: 1 or 2 the batched one (several tiles
    per accumulator, every epilogue warp busy), anything else the plain one.
    Scores, fused histogram and selection must be identical for every hint, also
    for hints below the true row count, and match the oracle."""
    extra = dict(extra)
    negate = extra.pop("negate_every", 0)
    prob = workloads.build(name, lengths, rows, kv, seed=zlib.crc32(name.encode()) % 1000, **extra)
    if negate:
        prob.k_scale[::negate] *= -1.0
    got = {}
    for hint in (0, 1, 2, 4):
        dp = lib.DeviceProblem(prob, rows_hint=hint)
        scores, hist = dp.score()
        out = dp.launch()
        assert dp.status() == lib.IDX_OK, hint
        got[hint] = (scores.cpu().numpy(), hist.cpu().numpy().view(np.uint32), out.cpu().numpy())
    s0, h0, o0 = got[0]
    gpu_util.check_scores_vs_oracle(orc, prob, s0, h0)
    gpu_util.check_selection(orc, o0, s0, prob.row_bound, prob.K)
    for hint, (s, h, o) in got.items():
        for r in range(prob.R):
            b = int(prob.row_bound[r])
            assert np.array_equal(s[r, :b], s0[r, :b]), (hint, r)
        assert np.array_equal(h, h0), hint
        assert np.array_equal(o, o0), hint


def test_wait_limit_in_the_batched_scan(lib, orc):
    """The batched scan (a lone row, hint 1) held back at its first hand-off also
    ends in IDX_ETIMEOUT and leaves the context usable."""
    prob = workloads.build("stall_lone", [6000], [1], "e4m3", seed=15)
    dp = lib.DeviceProblem(prob, rows_hint=1)
    prev = lib.debug_set(lib.IDX_DEBUG_WAIT_LIMIT_NS, 20_000_000)
    try:
        lib.debug_set(lib.IDX_DEBUG_STALL_SCORE_MMA, 1)
        dp.score()
        assert dp.status() == lib.IDX_ETIMEOUT
    finally:
        lib.debug_set(lib.IDX_DEBUG_STALL_SCORE_MMA, 0)
        lib.debug_set(lib.IDX_DEBUG_WAIT_LIMIT_NS, prev)
    scores, hist = dp.score()
    assert dp.status() == lib.IDX_OK
    gpu_util.check_scores_vs_oracle(orc, prob, scores.cpu().numpy(), hist.cpu().numpy().view(np.uint32))


def test_wait_limit_reports_timeout_and_context_survives(lib, orc):
    """A scoring launch told to hold back its first accumulator hand-off: the
    epilogue's wait runs out (limit 20 ms), the kernel records IDX_ETIMEOUT and
    returns; a normal launch afterwards still matches the oracle."""
    prob = workloads.build("stall", [4096], [4], "e4m3", seed=14)
    dp = lib.DeviceProblem(prob)
    prev = lib.debug_set(lib.IDX_DEBUG_WAIT_LIMIT_NS, 20_000_000)
    try:
        lib.debug_set(lib.IDX_DEBUG_STALL_SCORE_MMA, 1)
        dp.score()
        assert dp.status() == lib.IDX_ETIMEOUT
    finally:
        lib.debug_set(lib.IDX_DEBUG_STALL_SCORE_MMA, 0)
        lib.debug_set(lib.IDX_DEBUG_WAIT_LIMIT_NS, prev)
    dp2, scores, hist, st = gpu_util.run_score(lib, prob)
    assert st == lib.IDX_OK
    gpu_util.check_scores_vs_oracle(orc, prob, scores, hist)


@pytest.mark.parametrize("lengths,rows", [([3000, 700], [4, 1]), ([5000, 900], [1, 1])], ids=["rows4", "lone_rows"])
def test_launch_from_host_buffers(lib, orc, lengths, rows):
    """idx_launch_host (hint 0: the library counts the rows per request from the
    host row map, so lone rows take the batched scan) equal to idx_launch."""
    prob = workloads.build("host", lengths, rows, "e4m3", seed=15)
    host = {k: torch.from_numpy(getattr(prob, k)).pin_memory()
            for k in ("q", "w", "k_cache", "k_scale", "page_table", "row_req", "row_bound")}
    hp = lib.make_problem(host["q"], host["w"], host["k_cache"], host["k_scale"], host["page_table"],
                          host["row_req"], host["row_bound"], prob.max_bound, lib.IDX_KV_E4M3)
    arena = lib.alloc_bytes(lib.host_arena_size(hp, prob.K))
    out = torch.empty((prob.R, prob.K), dtype=torch.int32).pin_memory()
    lib.idx_launch_host(hp, prob.K, out, arena)
    torch.cuda.synchronize()
    dp = lib.DeviceProblem(prob)
    assert np.array_equal(out.numpy(), dp.launch().cpu().numpy())


def test_launch_replays_from_a_cuda_graph(lib, orc):
    """idx_launch captured into a CUDA graph (its four kernels and their
    programmatic dependencies) replays to the direct call's result, twice in a row,
    and its status word reads clean."""
    prob = workloads.build("graph", [7000, 3000], [4, 1], "e4m3", seed=16)
    dp = lib.DeviceProblem(prob)
    want = dp.launch().cpu().numpy()
    out = torch.full((prob.R, prob.K), -5, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        dp.launch(out, stream=side)       # one-time setup happens outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    out.fill_(-5)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dp.launch(out, stream=torch.cuda.current_stream())
    for _ in range(2):
        out.fill_(-5)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), want)
    assert dp.status() == lib.IDX_OK


def test_concurrent_launches_on_two_streams(lib, orc):
    """Two problems with their own workspaces, launched back to back on two
    streams so that their kernels can overlap, give the results each gives alone
    (the library keeps no state of a launch outside the caller's workspace)."""
    pa = workloads.build("stream_a", [9000, 4000], [4, 2], "e4m3", seed=17)
    pb = workloads.build("stream_b", [12000], [1], "bf16", seed=18)
    da, db = lib.DeviceProblem(pa), lib.DeviceProblem(pb)
    want_a, want_b = da.launch().cpu().numpy(), db.launch().cpu().numpy()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    oa = torch.empty((pa.R, pa.K), dtype=torch.int32, device="cuda")
    ob = torch.empty((pb.R, pb.K), dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):
        oa.fill_(-9)
        ob.fill_(-9)
        torch.cuda.synchronize()
        da.launch(oa, stream=sa)
        db.launch(ob, stream=sb)
        torch.cuda.synchronize()
        assert np.array_equal(oa.cpu().numpy(), want_a)
        assert np.array_equal(ob.cpu().numpy(), want_b)
    assert da.status(sa) == lib.IDX_OK and db.status(sb) == lib.IDX_OK


@pytest.mark.parametrize("K", [1, 100, 2047])
def test_launch_at_other_k(lib, orc, K):
    """The fused launch at K other than 2048, against the oracle's selection of
    the same K on the GPU's own scores."""
    prob = workloads.build("other_k", [5000, 1500, 90], [4, 2, 1], "e4m3", seed=19)
    dp = lib.DeviceProblem(prob, K=K)
    scores, _ = dp.score()
    out = dp.launch().cpu().numpy()
    assert out.shape == (prob.R, K) and dp.status() == lib.IDX_OK
    gpu_util.check_selection(orc, out, scores.cpu().numpy(), prob.row_bound, K)


@pytest.mark.parametrize("nreq", [3, 12], ids=["rows12", "rows48"])
def test_bad_bounds_and_requests_are_reported(lib, orc, nreq):
    """A row bound past max_bound is clamped to it and a request id outside [0, Q)
    reads nothing; both are reported as IDX_EDEVICE.  The other rows are scored
    and selected as usual."""
    prob = workloads.build("badbound", [900] * nreq, [4] * nreq, "e4m3", seed=20)
    mb = int(prob.max_bound)
    bad_bound = prob.row_bound.copy()
    bad_bound[1] = mb + 50
    for kind in ("bound", "request"):
        p = workloads.build("badbound", [900] * nreq, [4] * nreq, "e4m3", seed=20)
        if kind == "bound":
            p.row_bound[:] = bad_bound
        else:
            p.row_req[2] = p.page_table.shape[0] + 3
        dp = lib.DeviceProblem(p, max_bound=mb, rows_hint=0)
        scores, _ = dp.score()
        assert dp.status() == lib.IDX_EDEVICE, kind
        out = dp.launch().cpu().numpy()
        assert dp.status() == lib.IDX_EDEVICE, kind
        scores = scores.cpu().numpy()
        ref = p
        if kind == "bound":
            ref.row_bound[1] = mb                      # what the library scores: the clamped bound
        else:
            ref.row_bound[2] = 0                       # the bad row reads nothing
            ref.row_req[2] = 0
            assert (out[2] == -1).all()
        gpu_util.check_scores_vs_oracle(orc, ref, scores)
        gpu_util.check_selection(orc, out, scores, ref.row_bound, ref.K)
