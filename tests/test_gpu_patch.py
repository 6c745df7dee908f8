"""idx_patch_new_keys (each decode row's new key into the paged cache) against the
oracle: the written codes and scales bit-exact, nothing else touched, and the
launch that follows scores the new keys for every row of the request."""
import numpy as np
import pytest
import torch

import workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    import sparse_attention_indexer_launch_gb300 as lib
    return lib


def _new_keys(seed, R, scale=1.0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((R, 128)) * scale).astype(np.float32)
    x[0, :5] = 0.0                       # zeros, a signed zero and tiny values in one key
    x[0, 5] = -0.0
    x[0, 6:10] = 1e-7
    if R > 1:
        x[1] = 0.0                       # an all-zero key: scale 1
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("kv", ["e4m3", "bf16"])
def test_patch_writes_the_new_keys_and_the_launch_scores_them(lib, orc, kv):
    # rows of a request at consecutive positions (a draft chain), a lone row, a
    # zero-bound row, and positions on both sides of a page edge
    prob = workloads.build("patch", [3000, 64, 129, 5000], [4, 1, 2, 3], kv, seed=41,
                           bounds=[[2997, 2998, 2999, 3000], [64], [0, 129], [4031, 4032, 4033]])
    k_new = _new_keys(42, prob.R, scale=3.0)
    dp = lib.DeviceProblem(prob)
    lib.idx_patch_new_keys(dp.problem, torch.from_numpy(k_new.view(np.int16)).cuda())
    ref = orc.patch_new_keys(prob, k_new)
    if kv == "e4m3":
        got_cache = dp.k_cache.cpu().numpy()
        assert np.array_equal(got_cache, ref.k_cache), "cache bytes differ from the oracle's encoding"
        assert np.array_equal(dp.k_scale.cpu().numpy().view(np.uint32), ref.k_scale.view(np.uint32))
    else:
        got_cache = dp.k_cache.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got_cache, ref.k_cache)
    # the launch on the patched cache: its scores and selection against the oracle's
    out = dp.launch().cpu().numpy()
    assert dp.status() == lib.IDX_OK
    scores, _ = dp.score()
    scores = scores.cpu().numpy()
    ref_scores = orc.score(ref, ld=scores.shape[1])
    worst, where = parity.score_errors(scores, ref_scores, prob.row_bound)
    assert worst <= 1.0, (worst, where)
    O = orc.topk(ref_scores.astype(np.float32), prob.row_bound, prob.K)
    parity.check_endtoend(out, ref_scores, O, prob.row_bound, prob.K)


def test_patch_of_a_large_batch_matches_the_oracle(lib, orc):
    prob = workloads.make_config(2)          # 8 requests x 4 rows, shared shuffled pool
    k_new = _new_keys(43, prob.R, scale=0.01)
    dp = lib.DeviceProblem(prob)
    lib.idx_patch_new_keys(dp.problem, torch.from_numpy(k_new.view(np.int16)).cuda())
    ref = orc.patch_new_keys(prob, k_new)
    torch.cuda.synchronize()
    assert np.array_equal(dp.k_cache.cpu().numpy(), ref.k_cache)
    assert np.array_equal(dp.k_scale.cpu().numpy().view(np.uint32), ref.k_scale.view(np.uint32))


@pytest.mark.parametrize("kv", ["e4m3", "bf16"])
def test_launch_with_new_keys_equals_patch_then_launch(lib, orc, kv):
    """idx_launch_new_keys (the keys written by the launch's own first kernel)
    leaves the same cache as the oracle's patch and selects exactly what
    idx_patch_new_keys followed by idx_launch selects."""
    prob = workloads.build("fused_patch", [3000, 64, 129, 5000], [4, 1, 2, 3], kv, seed=45,
                           bounds=[[2997, 2998, 2999, 3000], [64], [0, 129], [4031, 4032, 4033]])
    k_new = torch.from_numpy(_new_keys(46, prob.R, scale=2.0).view(np.int16)).cuda()
    ref = orc.patch_new_keys(prob, k_new.cpu().numpy().view(np.uint16))
    fused = lib.DeviceProblem(prob)
    out = torch.empty((prob.R, prob.K), dtype=torch.int32, device="cuda")
    lib.idx_launch_new_keys(fused.problem, k_new, prob.K, out, fused.ws)
    assert fused.status() == lib.IDX_OK
    if kv == "e4m3":
        assert np.array_equal(fused.k_cache.cpu().numpy(), ref.k_cache)
        assert np.array_equal(fused.k_scale.cpu().numpy().view(np.uint32), ref.k_scale.view(np.uint32))
    else:
        assert np.array_equal(fused.k_cache.view(torch.int16).cpu().numpy().view(np.uint16), ref.k_cache)
    split = lib.DeviceProblem(prob)
    lib.idx_patch_new_keys(split.problem, k_new)
    assert np.array_equal(out.cpu().numpy(), split.launch().cpu().numpy())
