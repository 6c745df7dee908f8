"""The page's own top-k test matrix and query-magnitude stress cases, on the GPU
through the C ABI, against the oracle.

sglang PR 48224 page, section Accuracy Tests: the top-k check runs at positions
8447, 131071, 262143 and 524287 (bound = position + 1) with 2, 4 and 8 rows of
one request; the 2-row case is a live row with a pad row of the same request
(section Modifications, commit 1), the 8-row case the draft
chain of two groups of four.  Every visible score is compared with the oracle
within |err| <= 1e-3 + 2e-3 |ref|, the fused first-digit histogram exactly, the
selection bit-exactly on the GPU's own scores, the fused launch against that
selection, and the end-to-end index set under the allowed-swap rule.

The query cases stress the two-term E4M3 split of the bf16 query (the per-head
power-of-two prescale and its clamp, and the low term): rows scaled by 2^s for
s from -120 to +100, and heads with one large element among many small ones,
inside the split's exact range or so far below it that dropping them stays
within tolerance.  (A head whose small elements sit between those two, such as
2^-12 of its largest, loses up to about 2^-10.5 of the largest per element and
can exceed the absolute part of the tolerance: with elements at about 2^-12
and 2^-20 of the largest, scores near zero came out 14 and 4 times the
tolerance off.)"""
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


def _page_shapes():
    path = __file__.rsplit("/", 1)[0] + "/golden/page_test_shapes.txt"
    fields = {}
    for line in open(path):
        line = line.split("[")[0].strip()
        if line and not line.startswith("#"):
            k, v = line.split("=")
            fields[k.strip()] = [int(x) for x in v.split()]
    return fields["topk_positions"], fields["topk_rows"]


POSITIONS, ROWS = _page_shapes()
CASES = [(p + 1, n) for p in POSITIONS for n in ROWS]


def _check_all(lib, orc, prob):
    dp, scores, hist, st = gpu_util.run_score(lib, prob)
    assert st == lib.IDX_OK, lib.status_string(st)
    b = prob.row_bound
    ref = orc.score(prob, ld=scores.shape[1])
    worst, where = parity.score_errors(scores, ref, b)
    assert worst <= 1.0, (worst, where)
    assert np.array_equal(hist, orc.first_digit_hist(scores, b)), "fused first-digit histogram"
    out = dp.topk(torch.from_numpy(scores).cuda()).cpu().numpy()
    gpu_util.check_selection(orc, out, scores, b, prob.K)
    launch = dp.launch().cpu().numpy()
    assert dp.status() == lib.IDX_OK
    assert np.array_equal(launch, out), "fused launch differs from selection on its own scores"
    O = orc.topk(ref.astype(np.float32), b, prob.K)
    parity.check_endtoend(launch, ref, O, b, prob.K)
    return worst


@pytest.mark.parametrize("bound,rows", CASES, ids=[f"bound{b}_rows{n}" for b, n in CASES])
def test_page_topk_matrix(lib, orc, bound, rows):
    """One request holding `bound` keys; rows 2 = the live row and its pad row."""
    seed = (bound * 7 + rows) % 1000
    if rows == 2:
        prob = workloads.build(f"page_{bound}_{rows}", [bound], [2], "e4m3", seed=seed, key_dist="mixture",
                               bounds=[[bound, 0]])
    else:
        prob = workloads.build(f"page_{bound}_{rows}", [bound], [rows], "e4m3", seed=seed, key_dist="mixture")
    worst = _check_all(lib, orc, prob)
    print(f"bound {bound} rows {rows}: worst score error {worst:.3f} of tolerance")


def _bf16_bits(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("kv", ["e4m3", "bf16"])
def test_query_rows_at_extreme_magnitudes(lib, orc, kv):
    """Rows scaled by 2^s, s from -120 to 0: the prescale of the split takes each
    head's largest |q| to [128, 256), clamped at 2^120 (the row at 2^-120 meets
    the clamp), and the weights take the inverse, so scores span about 2^120
    between rows.  Larger scales are left out: there the scores reach 1e27, the
    tolerance is relative only, and a score that cancels to 2^-12 of its head
    terms carries fp32 accumulation error above it (any fp32 path would)."""
    prob = workloads.build("q_extreme", [3000, 1500], [4, 4], kv, seed=41)
    rng = np.random.default_rng(42)
    q = rng.standard_normal((prob.R, 64, 128)).astype(np.float32)
    row_exp = np.array([-120, -100, -60, -20, 0, -6, -40, -80], np.float32)
    for r in range(prob.R):
        q[r] *= np.float32(2.0 ** row_exp[r % len(row_exp)])
    prob.q = _bf16_bits(q)
    _check_all(lib, orc, prob)


@pytest.mark.parametrize("small_exp", [-1, -24, -40])
def test_query_heads_one_large_many_small(lib, orc, small_exp):
    """Per head one element of magnitude about 2^8 and 127 of magnitude about
    2^small_exp (uniform in [1, 2) x 2^small_exp, random sign).  At 2^-1 they lie
    inside the split's exact range (at least 2^-9.5 of the head's largest); at
    2^-24 and 2^-40 their terms underflow the E4M3 subnormals and are dropped,
    and their whole contribution stays far below the score tolerance."""
    prob = workloads.build("q_small", [4000], [4], "e4m3", seed=43)
    rng = np.random.default_rng(44)
    mag = (1.0 + rng.random((prob.R, 64, 128))) * 2.0 ** small_exp
    q = (rng.choice([-1.0, 1.0], size=mag.shape) * mag).astype(np.float32)
    big = rng.integers(0, 128, size=(prob.R, 64))
    sign = rng.choice([-1.0, 1.0], size=(prob.R, 64))
    for r in range(prob.R):
        q[r, np.arange(64), big[r]] = (sign[r] * (200.0 + rng.random(64) * 50.0)).astype(np.float32)
    prob.q = _bf16_bits(q)
    _check_all(lib, orc, prob)
