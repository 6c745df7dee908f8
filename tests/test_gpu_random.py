"""A seeded sweep of random problem shapes through the C ABI, against the oracle.

Each case draws its own batch: 1 to 6 requests with log-uniform lengths up to
40,000 keys, 1 to 4 rows a request (now and then 5 to 8, which the plan splits
into groups of at most four; every fourth case at most two, which selects the
batched scan instance), either cache type, normal or mixture keys, exact
duplicates, bounds drawn anywhere in [0, L] (zero and equal bounds included),
rows in scrambled order, and a top-K size from 1 to 2,048.  The library picks
the scan instance from the row map itself.  Every visible score must be within
the tolerance, the fused histogram must equal a count of the stored scores, the
fused launch must equal the oracle's selection on the GPU's scores bit for bit,
and the end-to-end rule must hold against the oracle's own scores."""
import math

import numpy as np
import pytest
import torch

import workloads
from tests import gpu_util, parity

pytestmark = pytest.mark.gpu

CASES = 24


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    import sparse_attention_indexer_launch_gb300 as lib
    return lib


def _random_problem(case: int):
    rng = np.random.default_rng(7000 + case)
    Q = int(rng.integers(1, 7))
    lengths = [int(math.floor(math.exp(rng.uniform(0.0, math.log(40000.0))))) for _ in range(Q)]
    if case % 4 == 3:   # at most two rows a request: the batched scan instance
        rows = [int(rng.integers(1, 3)) for _ in range(Q)]
    else:
        rows = [int(rng.integers(5, 9)) if rng.random() < 0.15 else int(rng.integers(1, 5)) for _ in range(Q)]
    kv = "bf16" if rng.random() < 0.35 else "e4m3"
    K = int(rng.choice([1, 5, 64, 700, 2048]))
    extra = {}
    if rng.random() < 0.4:
        extra["key_dist"] = "mixture"
    if rng.random() < 0.3:
        extra["dup_frac"] = 0.02
    if rng.random() < 0.4:
        extra["bounds"] = [[int(rng.integers(0, L + 1)) for _ in range(n)] for L, n in zip(lengths, rows)]
    R = sum(rows)
    if R > 1 and rng.random() < 0.3:
        extra["row_order"] = [int(x) for x in rng.permutation(R)]
    return workloads.build(f"random_{case}", lengths, rows, kv, seed=case, K=K, **extra)


@pytest.mark.parametrize("case", range(CASES))
def test_random_problem(lib, orc, case):
    prob = _random_problem(case)
    dp, scores, hist, st = gpu_util.run_score(lib, prob, K=prob.K)
    assert st == lib.IDX_OK, lib.status_string(st)
    ref, _ = gpu_util.check_scores_vs_oracle(orc, prob, scores, hist)
    out = dp.launch().cpu().numpy()
    assert dp.status() == lib.IDX_OK
    gpu_util.check_selection(orc, out, scores, prob.row_bound, prob.K)
    O = orc.topk(ref.astype(np.float32), prob.row_bound, prob.K)
    parity.check_endtoend(out, ref, O, prob.row_bound, prob.K)
