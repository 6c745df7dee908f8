"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare with the oracle under the rules of tests/parity.py."""
from __future__ import annotations

import numpy as np

from tests import parity


def run_score(lib, prob, K=None):
    dp = lib.DeviceProblem(prob, K=K)
    scores, hist = dp.score()
    st = dp.status()
    return dp, scores.cpu().numpy(), hist.cpu().numpy().view(np.uint32), st


def check_scores_vs_oracle(orc, prob, gpu_scores, gpu_hist=None):
    ref = orc.score(prob, ld=gpu_scores.shape[1])
    worst, where = parity.score_errors(gpu_scores, ref, prob.row_bound)
    assert worst <= 1.0, f"score outside tolerance: ratio {worst:.3g} at {where}"
    if gpu_hist is not None:
        assert np.array_equal(gpu_hist, orc.first_digit_hist(gpu_scores, prob.row_bound)), \
            "fused first-digit histogram differs from a count of the stored scores"
    return ref, worst


def check_selection(orc, gpu_idx, gpu_scores, row_bound, K):
    ref_idx = orc.topk(gpu_scores, row_bound, K)
    if not np.array_equal(gpu_idx, ref_idx):
        bad = np.argwhere(gpu_idx != ref_idx)
        r, j = bad[0]
        raise AssertionError(f"selection differs at row {r} slot {j}: gpu {gpu_idx[r, j]} oracle "
                             f"{ref_idx[r, j]} ({len(bad)} slots differ)")
