"""idx_topk_noalloc (top-K on the library's own scratch, no caller workspace)
against idx_topk and the oracle's selection on the same scores: two different
calls in a row, each equal to both, and the row limit refused before anything is
launched.

Collected last on purpose, so that it also runs after every other GPU test of
the session has used the device."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

MAX_ROWS = 8   # IDX_NOALLOC_MAX_ROWS in include/idx.h


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    import sparse_attention_indexer_launch_gb300 as lib
    return lib


def _scores(seed, R, L):
    """Crafted rows: normal scores, many exact ties, one narrow band of values,
    a short row and an empty row."""
    rng = np.random.default_rng(seed)
    s = rng.standard_normal((R, L)).astype(np.float32)
    s[1] = rng.integers(-3, 3, L).astype(np.float32)
    s[2] = 1.0 + rng.integers(0, 16, L).astype(np.float32) * np.float32(2 ** -20)
    bounds = np.full(R, L, np.int32)
    bounds[3] = 1500
    bounds[4] = 0
    bounds[R - 1] = L - 7
    return s, bounds


def _pair(lib, s, bounds, K):
    R, L = s.shape
    dev_s = torch.from_numpy(s).cuda()
    dev_b = torch.from_numpy(bounds).cuda()
    ref = torch.empty((R, K), dtype=torch.int32, device="cuda")
    ws = lib.alloc_bytes(64 << 20)
    lib.idx_topk(dev_s, L, dev_b, R, L, K, None, ref, ws)
    got = torch.full((R, K), -7, dtype=torch.int32, device="cuda")
    lib.idx_topk_noalloc(dev_s, L, dev_b, R, L, K, got)
    torch.cuda.synchronize()
    return ref.cpu().numpy(), got.cpu().numpy()


def test_noalloc_matches_idx_topk_on_two_calls_in_a_row(lib, orc):
    # first call: 8 rows (the limit), K = 2048
    s1, b1 = _scores(101, MAX_ROWS, 40000)
    ref1, got1 = _pair(lib, s1, b1, 2048)
    assert np.array_equal(got1, ref1)
    assert np.array_equal(got1, orc.topk(s1, b1, 2048))
    # second call right after, other shapes and scores: nothing may leak from the first
    s2, b2 = _scores(202, 6, 9000)
    ref2, got2 = _pair(lib, s2, b2, 100)
    assert np.array_equal(got2, ref2)
    assert np.array_equal(got2, orc.topk(s2, b2, 100))
    assert (got2[4] == -1).all()                       # the empty row is all padding


def test_noalloc_refuses_more_rows_than_its_scratch_holds(lib):
    R, L = MAX_ROWS + 1, 4096
    s = torch.zeros((R, L), dtype=torch.float32, device="cuda")
    b = torch.full((R,), L, dtype=torch.int32, device="cuda")
    out = torch.empty((R, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(lib.IdxError) as e:
        lib.idx_topk_noalloc(s, L, b, R, L, 16, out)
    assert e.value.status == lib.IDX_EUNSUPPORTED
