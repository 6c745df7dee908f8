"""The key-sharded indexer on one GPU: a request's pages split into S shards,
each shard scored and ranked by idx_launch_scored on its own cache and page
table, the lists merged by idx_merge_topk.  The merge must equal the unsharded
idx_launch bit for bit (the union of the shards' top-K holds the global top-K,
and a key's score does not depend on the shard it is read in), and the merged
scores must equal the unsharded scores at those positions.  Shards that hold no
key of a row, rows with a bound below K and both caches are covered."""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    import sparse_attention_indexer_launch_gb300 as lib
    return lib


CASES = [
    ("e4m3_mixed", [20000, 9000, 3000, 700], [4, 2, 1, 3], "e4m3", {"bounds": None}),
    ("bf16_mixed", [12000, 5000], [3, 4], "bf16", {"bounds": None}),
    ("ties", [9000], [2], "e4m3", {"dup_frac": 0.2}),
]


@pytest.mark.parametrize("parts", [1, 2, 3, 8])
@pytest.mark.parametrize("name,lengths,rows,kv,extra", CASES, ids=[c[0] for c in CASES])
def test_sharded_launch_merges_to_the_unsharded_selection(lib, orc, name, lengths, rows, kv, extra, parts):
    from sparse_attention_indexer_launch_gb300 import shard
    extra = {k: v for k, v in extra.items() if v is not None}
    prob = workloads.build(name, lengths, rows, kv, seed=61 + parts, **extra)
    full = lib.DeviceProblem(prob)
    want = full.launch().cpu().numpy()
    scores, _ = full.score()
    scores = scores.cpu().numpy()
    assert full.status() == lib.IDX_OK
    idx_parts, score_parts, offs = [], [], []
    for sp, off in shard.split(prob, parts):
        dp = lib.DeviceProblem(sp, K=prob.K, max_bound=max(int(sp.row_bound.max(initial=0)), 0))
        i, s = dp.launch_scored()
        assert dp.status() == lib.IDX_OK
        idx_parts.append(i)
        score_parts.append(s)
        offs.append(off)
    assert offs == shard.offsets(int(prob.page_table.shape[1]), parts)
    pi, ps = torch.stack(idx_parts), torch.stack(score_parts)
    out = torch.empty((prob.R, prob.K), dtype=torch.int32, device="cuda")
    out_s = torch.empty((prob.R, prob.K), dtype=torch.float32, device="cuda")
    lib.idx_merge_topk(pi, ps, offs, prob.K, out, out_s)
    got, got_s = out.cpu().numpy(), out_s.cpu().numpy()
    assert np.array_equal(got, want), "merged selection differs from the unsharded launch"
    for r in range(prob.R):
        n = int((got[r] >= 0).sum())
        assert np.array_equal(got_s[r, :n], scores[r, got[r, :n]]), f"row {r}: merged scores"   # -0.0 == +0.0
        assert np.all(np.isneginf(got_s[r, n:]))
    # the oracle's merge of the same lists agrees
    assert np.array_equal(orc.merge_topk(pi.cpu().numpy(), ps.cpu().numpy(), np.array(offs, np.int32), prob.K), got)


def test_merge_rejects_bad_arguments(lib):
    pi = torch.zeros((9, 2, 16), dtype=torch.int32, device="cuda")
    ps = torch.zeros((9, 2, 16), dtype=torch.float32, device="cuda")
    out = torch.empty((2, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(lib.IdxError) as e:
        lib.idx_merge_topk(pi, ps, [0] * 9, 16, out)          # more parts than the merge takes
    assert e.value.status == lib.IDX_EUNSUPPORTED
    with pytest.raises(lib.IdxError) as e:
        lib.idx_merge_topk(pi[:2], ps[:2], [0, -64], 16, out)   # negative offset
    assert e.value.status == lib.IDX_EINVAL


def _ranked_parts(orc, scores, bounds, cuts, Kin):
    """Each part [cuts[s], cuts[s+1]) of every row ranked on its own by the oracle:
    positions in the part's numbering (-1 padded) and their scores."""
    R = scores.shape[0]
    S = len(cuts) - 1
    pi = np.full((S, R, Kin), -1, np.int32)
    ps = np.zeros((S, R, Kin), np.float32)
    for s in range(S):
        a, b = cuts[s], cuts[s + 1]
        sub = np.ascontiguousarray(scores[:, a:b])
        idx = orc.topk(sub, np.clip(bounds - a, 0, b - a).astype(np.int32), Kin)
        pi[s] = idx
        for r in range(R):
            ok = idx[r] >= 0
            ps[s, r, ok] = sub[r, idx[r, ok]]
    return pi, ps


@pytest.mark.parametrize("Kin,K", [(64, 64), (64, 100), (300, 32), (2048, 2048)])
def test_merge_matches_the_oracle_on_crafted_lists(lib, orc, Kin, K):
    """Integer scores (ties within and across parts, -0.0 against +0.0), a part
    that holds no key of some rows, parts shorter than Kin, and K above or below
    the lists' length; compared with the oracle's merge of the same lists,
    positions and scores."""
    rng = np.random.default_rng(71 + Kin + K)
    R, L = 6, 5000
    scores = rng.integers(-6, 6, (R, L)).astype(np.float32)
    scores[scores == 0] = -0.0
    scores[0, ::3] = 0.0
    scores[1] = rng.standard_normal(L).astype(np.float32)
    bounds = np.array([L, 40, 0, 1300, L - 3, 2001], np.int32)    # row 1: only the first part
    cuts = [0, 1000, 1003, 2000, L]                                # a 3-key part
    pi, ps = _ranked_parts(orc, scores, bounds, cuts, Kin)
    want = orc.merge_topk(pi, ps, np.array(cuts[:-1], np.int32), K)
    out = torch.full((R, K), -7, dtype=torch.int32, device="cuda")
    out_s = torch.full((R, K), 7.0, dtype=torch.float32, device="cuda")
    lib.idx_merge_topk(torch.from_numpy(pi).cuda(), torch.from_numpy(ps).cuda(), cuts[:-1], K, out, out_s)
    got, got_s = out.cpu().numpy(), out_s.cpu().numpy()
    assert np.array_equal(got, want)
    for r in range(R):
        n = int((got[r] >= 0).sum())
        assert np.array_equal(got_s[r, :n], scores[r, got[r, :n]]), r
        assert np.all(np.isneginf(got_s[r, n:])), r
    assert (got[2] == -1).all()                                    # bound 0: all padding
