"""Key-sharded indexer: host-side splitting and exchange.

Decode context parallelism (the "Release Test Suite - GLM-5.2-EXL3" page,
section Config change) shards a request's KV cache over GPUs and merges the
indexer's top-k at an owner GPU.  Here a shard is a contiguous range of each
request's pages.  Every shard runs idx_launch_scored on the keys it holds (its
positions numbered from 0), the shards' (position, score) lists are gathered,
and idx_merge_topk, with each shard's first position as its offset, gives
exactly the unsharded selection.

This module only moves data: it slices page tables and row bounds on the host
and gathers the shards' lists with torch.distributed.  Scoring, selection and
the merge run in the library's kernels.
"""
from __future__ import annotations

import numpy as np

PAGE = 64


def page_cuts(num_pages: int, parts: int):
    """Page boundaries of `parts` contiguous shards of a request's page range, as
    even as possible: [c_0 = 0, c_1, ..., c_parts = num_pages]."""
    if parts < 1:
        raise ValueError("parts must be >= 1")
    return [int(round(i * num_pages / parts)) for i in range(parts + 1)]


def shard_bounds(row_bound, page0: int, page1: int):
    """Row bounds within a shard holding pages [page0, page1) of each request:
    the keys of a row's prefix that fall in the shard, numbered from the shard's
    first position."""
    b = np.asarray(row_bound, dtype=np.int64) - page0 * PAGE
    return np.clip(b, 0, (page1 - page0) * PAGE).astype(np.int32)


def shard_problem(prob, page0: int, page1: int):
    """The shard of a workloads.Problem holding pages [page0, page1) of every
    request, as the GPU owning it would hold it: its own cache of just those
    pages, renumbered in order, and a page table over them.  Returns
    (shard Problem, position offset)."""
    import copy
    pt = np.asarray(prob.page_table)[:, page0:page1]
    ids = sorted(set(int(x) for x in pt.ravel() if x >= 0))
    remap = {old: new for new, old in enumerate(ids)}
    new_pt = np.full(pt.shape if pt.shape[1] > 0 else (pt.shape[0], 1), -1, np.int32)
    for (i, j), v in np.ndenumerate(pt):
        if v >= 0:
            new_pt[i, j] = remap[int(v)]
    sel = np.array(ids if ids else [0], dtype=np.int64)
    out = copy.copy(prob)
    out.name = f"{prob.name}[pages {page0}:{page1}]"
    out.k_cache = np.ascontiguousarray(prob.k_cache[sel])
    out.k_scale = None if prob.k_scale is None else np.ascontiguousarray(prob.k_scale[sel])
    out.page_table = new_pt
    out.row_bound = shard_bounds(prob.row_bound, page0, page1)
    return out, page0 * PAGE


def split(prob, parts: int):
    """Every shard of `prob` (see shard_problem) with its position offset."""
    cuts = page_cuts(int(prob.page_table.shape[1]), parts)
    return [shard_problem(prob, cuts[i], cuts[i + 1]) for i in range(parts)]


def exchange(local_idx, local_score, group=None):
    """All-gather of every rank's [R][K] (position, score) lists: returns
    [world][R][K] tensors on every rank (the owner merges them)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    idx = [torch.empty_like(local_idx) for _ in range(world)]
    score = [torch.empty_like(local_score) for _ in range(world)]
    dist.all_gather(idx, local_idx.contiguous(), group=group)
    dist.all_gather(score, local_score.contiguous(), group=group)
    return torch.stack(idx), torch.stack(score)


def offsets(num_pages: int, parts: int):
    """Every shard's first position (the merge's offsets), known to every rank
    from the shard layout alone."""
    return [c * PAGE for c in page_cuts(num_pages, parts)[:-1]]
