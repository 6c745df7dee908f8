"""Parity rules between the CUDA path and the oracle.

Scores: |gpu - ref| <= 1e-3 + 2e-3 * |ref| for every visible (row, position), ref
being the oracle's double-precision score.

Selection given identical scores: bit-exact, i.e. the CUDA top-k run on the
CUDA scores equals the oracle's top-k run on those same fp32 scores.

End to end: the CUDA index set G and the oracle's index set O (top-k of the
oracle's scores rounded to fp32) have the same size, and every position in their
symmetric difference has an oracle score within the score tolerance of the
oracle's k-th score.  The order of G is checked against the CUDA scores.
"""
from __future__ import annotations

import numpy as np

ATOL = 1e-3
RTOL = 2e-3


def tol(ref):
    return ATOL + RTOL * np.abs(ref)


def score_errors(gpu_scores, ref_scores, row_bound):
    """Max of |gpu - ref| / tol(ref) over the visible positions (<= 1 passes)."""
    worst = 0.0
    where = None
    for r, b in enumerate(np.asarray(row_bound)):
        b = int(b)
        if b == 0:
            continue
        g = np.asarray(gpu_scores[r, :b], dtype=np.float64)
        f = np.asarray(ref_scores[r, :b], dtype=np.float64)
        ratio = np.abs(g - f) / tol(f)
        i = int(np.argmax(ratio))
        if not np.isfinite(ratio[i]) or ratio[i] > worst:
            worst = float(ratio[i]) if np.isfinite(ratio[i]) else float("inf")
            where = (r, i, float(g[i]), float(f[i]))
    return worst, where


def check_index_rows(idx, row_bound, K):
    """Structural invariants: unique, in bound, count = min(K, bound), -1 padded."""
    idx = np.asarray(idx)
    assert idx.shape == (len(row_bound), K), idx.shape
    for r, b in enumerate(np.asarray(row_bound)):
        n = min(K, int(b))
        head, tail = idx[r, :n], idx[r, n:]
        assert np.all(tail == -1), f"row {r}: padding is not -1"
        assert np.all((head >= 0) & (head < b)), f"row {r}: index out of bound"
        assert np.unique(head).size == n, f"row {r}: duplicate indices"


def check_order(idx, scores, row_bound, K):
    """Selected positions ordered by score descending, then position ascending."""
    for r, b in enumerate(np.asarray(row_bound)):
        n = min(K, int(b))
        sel = np.asarray(idx[r, :n], dtype=np.int64)
        s = np.asarray(scores[r], dtype=np.float32)[sel]
        if n > 1:
            ds = np.diff(s.astype(np.float64))
            assert np.all(ds <= 0), f"row {r}: scores not non-increasing"
            ties = ds == 0
            assert np.all(np.diff(sel)[ties] > 0), f"row {r}: ties not by ascending position"


def check_endtoend(gpu_idx, ref_scores, oracle_idx, row_bound, K):
    """Allowed-swap rule; returns the number of swapped positions over all rows."""
    swaps = 0
    for r, b in enumerate(np.asarray(row_bound)):
        n = min(K, int(b))
        if n == 0:
            assert np.all(gpu_idx[r] == -1)
            continue
        G = set(int(x) for x in gpu_idx[r, :n])
        O = set(int(x) for x in oracle_idx[r, :n])
        assert len(G) == n and len(O) == n
        kth = float(ref_scores[r, int(oracle_idx[r, n - 1])])
        t = ATOL + RTOL * abs(kth)
        for p in G ^ O:
            d = abs(float(ref_scores[r, p]) - kth)
            assert d <= t, (f"row {r}: position {p} differs between the sets with oracle score "
                            f"{ref_scores[r, p]!r}, {d:.3g} from the k-th value {kth!r} (tol {t:.3g})")
        swaps += len(G ^ O) // 2
    return swaps
