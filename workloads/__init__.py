"""Seeded synthetic inputs for the decode indexer.

This module only draws inputs: it holds none of the indexer's arithmetic, and
both the CUDA path's tests and benchmark and the CPU oracle's tests take their
inputs from here.  Shapes follow the indexer statement: q is bf16 [R][64][128],
w is fp32 [R][64], keys live in a paged cache of 64-token pages ([P][64][128]),
either FP8 E4M3 bytes with one fp32 scale per token ([P][64]) or bf16 values.
Page tables are [Q][pt_stride] int32 with -1 past each request's last page.

The five named workloads follow the indexer's stated configurations; the test
positions of the sglang PR 48224 page (section Accuracy Tests: ``--pos
8447,131071,262143,524287``, rows 2/4/8) give the bounds used by
``page_positions()``.  Where a configuration leaves a detail open the reading
taken here is: seed = configuration index; E4M3 quantisation by
round-to-nearest-even with the token's values first clamped to +-448; mixture
keys pick sigma in {1, 4} per token with probability 1/2; log-uniform lengths
are floor(exp(U(ln a, ln b))); the rows of a request are consecutive and see
bounds L-n+1 .. L.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

HEADS = 64
DIM = 128
PAGE = 64
TOPK = 2048


@dataclasses.dataclass
class Problem:
    name: str
    q: np.ndarray            # uint16 [R][64][128], bf16 bit patterns
    w: np.ndarray            # float32 [R][64]
    k_cache: np.ndarray      # uint8 [P][64][128] (e4m3) or uint16 [P][64][128] (bf16 bits)
    k_scale: np.ndarray | None  # float32 [P][64] for e4m3, None for bf16
    page_table: np.ndarray   # int32 [Q][pt_stride]
    row_req: np.ndarray      # int32 [R]
    row_bound: np.ndarray    # int32 [R]
    kv_dtype: str            # "e4m3" or "bf16"
    K: int = TOPK
    seed: int = 0
    recipe: str = ""

    @property
    def R(self) -> int:
        return int(self.row_bound.shape[0])

    @property
    def Q(self) -> int:
        return int(self.page_table.shape[0])

    @property
    def P(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def pt_stride(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def max_bound(self) -> int:
        return int(self.row_bound.max(initial=0))

    @property
    def key_rows(self) -> int:
        """Sum over rows of the keys each row scores (the metric's unit)."""
        return int(self.row_bound.astype(np.int64).sum())

    def request_keys(self) -> np.ndarray:
        """Keys read per request: the largest bound among its rows."""
        out = np.zeros(self.Q, dtype=np.int64)
        np.maximum.at(out, self.row_req.astype(np.int64), self.row_bound.astype(np.int64))
        return out

    @property
    def key_bytes(self) -> int:
        """Algorithmic key bytes: each request's keys read once."""
        per_key = DIM + 4 if self.kv_dtype == "e4m3" else 2 * DIM
        return int(self.request_keys().sum()) * per_key

    @property
    def mma_flops(self) -> int:
        return self.key_rows * 2 * HEADS * DIM


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def quantize_e4m3(x: np.ndarray):
    """fp32 tokens [n][128] -> (E4M3 codes uint8 [n][128], scale float32 [n]).

    The scale is the token's amax / 448; a token of zeros gets scale 1.  Values are
    divided by the scale, clamped to +-448 and rounded to nearest-even by torch's
    float8_e4m3fn cast, so no NaN code (0x7F, 0xFF) is ever produced."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    y = np.clip(x / scale[:, None], -448.0, 448.0).astype(np.float32)
    codes = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return np.ascontiguousarray(codes), scale


def _draw_keys(seed: int, n: int, kv_dtype: str, key_dist: str):
    """Keys in chunks of 2^16 tokens; chunk c draws from default_rng([seed, 7, c]) so
    the result does not depend on how many threads fill the chunks."""
    import concurrent.futures
    import os
    chunk = 1 << 16
    if kv_dtype == "e4m3":
        codes = np.empty((n, DIM), dtype=np.uint8)
        scales = np.empty(n, dtype=np.float32)
    else:
        codes = np.empty((n, DIM), dtype=np.uint16)
        scales = None

    def fill(c):
        s0 = c * chunk
        m = min(chunk, n - s0)
        rng = np.random.default_rng([seed, 7, c])
        x = rng.standard_normal((m, DIM), dtype=np.float32)
        if key_dist == "mixture":
            sigma = np.where(rng.random(m) < 0.5, np.float32(1.0), np.float32(4.0)).astype(np.float32)
            x *= sigma[:, None]
        elif key_dist != "normal":
            raise ValueError(key_dist)
        if kv_dtype == "e4m3":
            cq, sc = quantize_e4m3(x)
            codes[s0:s0 + m] = cq
            scales[s0:s0 + m] = sc
        else:
            codes[s0:s0 + m] = _bf16_bits(x)

    nchunks = (n + chunk - 1) // chunk
    workers = max(1, min(16, os.cpu_count() or 1, nchunks))
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(fill, range(nchunks)))
    return codes, scales


def build(name: str, lengths, rows_per_req, kv_dtype: str = "e4m3", seed: int = 0,
          key_dist: str = "normal", dup_frac: float = 0.0, bounds=None, K: int = TOPK,
          recipe: str = "", row_order=None) -> Problem:
    """General builder.

    lengths[q]       keys cached for request q (its pages are ceil(L/64));
    rows_per_req[q]  decode rows of request q, with bounds L-n+1..L unless
                     ``bounds`` (a list per request) is given;
    dup_frac         fraction of each request's positions overwritten by exact
                     copies (bytes and scale) of other positions of that request;
    row_order        optional permutation of the rows (to test non-consecutive
                     rows of one request)."""
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in lengths]
    rows_per_req = [int(x) for x in rows_per_req]
    Q = len(lengths)
    npages = [(L + PAGE - 1) // PAGE for L in lengths]
    P = max(1, sum(npages))
    pt_stride = max(1, max(npages) if npages else 1)
    R = sum(rows_per_req)

    q = _bf16_bits(rng.standard_normal((R, HEADS, DIM), dtype=np.float32))
    w = (rng.standard_normal((R, HEADS), dtype=np.float32) / np.float32(8.0)).astype(np.float32)

    codes, scales = _draw_keys(seed, P * PAGE, kv_dtype, key_dist)
    k_cache = codes.reshape(P, PAGE, DIM)
    k_scale = None if scales is None else scales.reshape(P, PAGE)

    perm = rng.permutation(P).astype(np.int32)
    page_table = np.full((max(Q, 1), pt_stride), -1, dtype=np.int32)
    cur = 0
    for qi in range(Q):
        page_table[qi, :npages[qi]] = perm[cur:cur + npages[qi]]
        cur += npages[qi]

    if dup_frac > 0:
        for qi in range(Q):
            L = lengths[qi]
            nd = int(round(dup_frac * L))
            if nd == 0 or L < 2:
                continue
            dst = rng.choice(L, size=nd, replace=False)
            src = rng.integers(0, L, size=nd)
            src = np.where(src == dst, (src + 1) % L, src)
            dp, ds = page_table[qi, dst // PAGE], dst % PAGE
            sp, ss = page_table[qi, src // PAGE], src % PAGE
            k_cache[dp, ds] = k_cache[sp, ss]
            if k_scale is not None:
                k_scale[dp, ds] = k_scale[sp, ss]

    row_req = np.empty(R, dtype=np.int32)
    row_bound = np.empty(R, dtype=np.int32)
    r = 0
    for qi in range(Q):
        n = rows_per_req[qi]
        L = lengths[qi]
        bq = bounds[qi] if bounds is not None else [max(0, L - n + 1 + j) for j in range(n)]
        for j in range(n):
            row_req[r] = qi
            row_bound[r] = int(bq[j])
            r += 1
    if row_order is not None:
        order = np.asarray(row_order)
        q, w, row_req, row_bound = q[order], w[order], row_req[order], row_bound[order]

    return Problem(name=name, q=np.ascontiguousarray(q), w=np.ascontiguousarray(w),
                   k_cache=np.ascontiguousarray(k_cache),
                   k_scale=None if k_scale is None else np.ascontiguousarray(k_scale),
                   page_table=page_table, row_req=row_req, row_bound=row_bound,
                   kv_dtype=kv_dtype, K=K, seed=seed, recipe=recipe)


def _log_uniform(rng, n, lo, hi):
    return [int(math.floor(math.exp(rng.uniform(math.log(lo), math.log(hi))))) for _ in range(n)]


CONFIG_NAMES = {
    0: "cfg0: 1 request x 1 row, 4,096 keys, E4M3",
    1: "cfg1: 1 request x 4 rows, 131,072 keys, E4M3, 1% duplicate keys",
    2: "cfg2: 8 requests x 4 rows, log-uniform 8K-256K keys, E4M3, shared shuffled pool",
    3: "cfg3: 2 requests x 4 rows, 524,288 keys each, E4M3, sigma 1/4 mixture keys",
    "3a": "cfg3a: 1 request x 4 rows, 524,288 keys, E4M3, sigma 1/4 mixture keys",
    "3b": "cfg3b: 1 request x 1 row at 524,288 keys and 1 pad row (bound 0), E4M3, sigma 1/4 mixture keys",
    4: "cfg4: 64 requests x 1-4 rows, log-uniform 1K-512K keys, bf16 cache",
}


def make_config(cfg, seed_offset: int = 0) -> Problem:
    """The named workloads (see CONFIG_NAMES).  A nonzero seed_offset draws the same
    shapes (lengths, rows, bounds) with other values and page permutations."""
    return _make_config(cfg, seed_offset)


def _make_config(cfg, off: int) -> Problem:
    if cfg == 0:
        return build(CONFIG_NAMES[0], [4096], [1], "e4m3", seed=0 + off,
                     bounds=[[4096]], recipe="q N(0,1) bf16; w N(0,1)/8; keys N(0,1) -> E4M3, scale amax/448")
    if cfg == 1:
        L = 131072
        return build(CONFIG_NAMES[1], [L], [4], "e4m3", seed=1 + off, dup_frac=0.01,
                     recipe="as cfg0; bounds L-3..L; 1% of positions exact copies of others")
    if cfg == 2:
        rng = np.random.default_rng(1002)
        lengths = _log_uniform(rng, 8, 8192, 262144)
        return build(CONFIG_NAMES[2], lengths, [4] * 8, "e4m3", seed=2 + off,
                     recipe=f"lengths {lengths}; bounds L-3..L; one globally shuffled page pool")
    if cfg == 3:
        return build(CONFIG_NAMES[3], [524288, 524288], [4, 4], "e4m3", seed=3 + off, key_dist="mixture",
                     recipe="keys sigma in {1,4} w.p. 1/2 per token -> E4M3; bounds L-3..L")
    if cfg == "3a":
        return build(CONFIG_NAMES["3a"], [524288], [4], "e4m3", seed=3 + off, key_dist="mixture",
                     recipe="first request of cfg3 alone")
    if cfg == "3b":
        return build(CONFIG_NAMES["3b"], [524288, 0], [1, 1], "e4m3", seed=3 + off, key_dist="mixture",
                     recipe="cfg3's first request with one row, and a pad row of an empty request")
    if cfg == 4:
        rng = np.random.default_rng(1004)
        rows = [int(x) for x in rng.integers(1, 5, size=64)]
        lengths = _log_uniform(rng, 64, 1024, 524288)
        return build(CONFIG_NAMES[4], lengths, rows, "bf16", seed=4 + off,
                     recipe="bf16 keys N(0,1); rows U{1..4}; lengths log-uniform 1K-512K")
    raise ValueError(cfg)


def page_positions():
    """The page's top-k test positions (pos = bound - 1) and row counts."""
    return [8447, 131071, 262143, 524287], [2, 4, 8]
