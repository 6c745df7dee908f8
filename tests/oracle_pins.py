"""Pins of the oracle to facts other than itself.

Each pin takes an ``oracle.Oracle`` so that the same checks can be run against
copies of oracle.c with planted mistakes (test_oracle.py checks that every such
copy fails at least one pin).  Expected values come from closed forms of the
constructed inputs, from library routines (torch's float8/bfloat16 casts,
Python's sorted, numpy), or from brute force; none is the oracle's formula
typed again.
"""
from __future__ import annotations

import itertools
import math
import struct

import numpy as np
import torch

import workloads

H, D, PG = 64, 128, 64


def e4m3_codes(values):
    """Library encoder (torch float8_e4m3fn) for exactly representable values."""
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.float8_e4m3fn)
    back = t.float().numpy()
    assert np.array_equal(back, np.asarray(values, dtype=np.float32)), "not exactly representable"
    return t.view(torch.uint8).numpy()


def bf16_bits(values):
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    assert np.array_equal(t.float().numpy(), np.asarray(values, dtype=np.float32))
    return t.view(torch.int16).numpy().view(np.uint16)


def blank_problem(lengths, rows_req, bounds, kv="e4m3", page_table=None, P=None):
    """All-zero inputs with the given shape; callers fill in the few values a case needs."""
    Q = len(lengths)
    npages = [(L + PG - 1) // PG for L in lengths]
    if page_table is None:
        P = sum(npages)
        stride = max(npages)
        page_table = np.full((Q, stride), -1, dtype=np.int32)
        cur = 0
        for qi in range(Q):
            page_table[qi, :npages[qi]] = np.arange(cur, cur + npages[qi])
            cur += npages[qi]
    page_table = np.asarray(page_table, dtype=np.int32)
    R = len(rows_req)
    kdt = np.uint8 if kv == "e4m3" else np.uint16
    return workloads.Problem(
        name="hand", q=np.zeros((R, H, D), np.uint16), w=np.zeros((R, H), np.float32),
        k_cache=np.zeros((P, PG, D), kdt),
        k_scale=np.ones((P, PG), np.float32) if kv == "e4m3" else None,
        page_table=page_table, row_req=np.asarray(rows_req, np.int32),
        row_bound=np.asarray(bounds, np.int32), kv_dtype=kv)


def set_key(prob, req, t, dim_values, scale=None):
    """Write the key of logical position t of request req through the page table."""
    page = prob.page_table[req, t // PG]
    slot = t % PG
    for d, v in dim_values.items():
        code = e4m3_codes([v])[0] if prob.kv_dtype == "e4m3" else bf16_bits([v])[0]
        prob.k_cache[page, slot, d] = code
    if scale is not None:
        prob.k_scale[page, slot] = scale


def set_q(prob, r, h, d, v):
    prob.q[r, h, d] = bf16_bits([v])[0]


# ---------------------------------------------------------------------------- decode


def pin_e4m3_all_codes(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = orc.e4m3_to_double(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def pin_e4m3_closed_forms(orc):
    # OCP E4M3 ("fn"): bias 7, 3 mantissa bits, subnormal step 2^-9, max 1.75 * 2^8.
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x3F: 1.875, 0x40: 2.0, 0x44: 3.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for code, val in cases.items():
        assert orc.e4m3_to_double([code])[0] == val, hex(code)
    assert math.isnan(orc.e4m3_to_double([0x7F])[0]) and math.isnan(orc.e4m3_to_double([0xFF])[0])
    z = orc.e4m3_to_double([0x80])[0]
    assert z == 0.0 and math.copysign(1.0, z) == -1.0


def pin_bf16_decode(orc):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = orc.bf16_to_double(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---------------------------------------------------------------------------- scores


def pin_relu_and_signed_weights(orc):
    # heads 0 and 1 read dim 0; key dim0 = 2, scale 1/2: both heads see 0.5*2 = 1.
    p = blank_problem([1], [0], [1])
    set_q(p, 0, 0, 0, 1.0)
    set_q(p, 0, 1, 0, 1.0)
    p.w[0, 0], p.w[0, 1] = 0.5, -0.25
    set_key(p, 0, 0, {0: 2.0}, scale=0.5)
    assert orc.score(p)[0, 0] == 0.5 * 1.0 - 0.25 * 1.0
    # head 1 now reads -dim0: its product is -1 and the ReLU removes it.
    set_q(p, 0, 1, 0, -1.0)
    assert orc.score(p)[0, 0] == 0.5
    # both heads negative: score 0.
    set_q(p, 0, 0, 0, -1.0)
    assert orc.score(p)[0, 0] == 0.0


def pin_head_dim_layout(orc):
    # key dims hold distinct integers 1..13 so any mix-up of (head, dim) changes the result.
    p = blank_problem([1], [0], [1])
    set_key(p, 0, 0, {d: float(d % 13 + 1) for d in range(D)}, scale=1.0)
    set_q(p, 0, 3, 5, 2.0)          # head 3, dim 5 -> 2 * (5 % 13 + 1) = 12
    p.w[0, :] = np.arange(H, dtype=np.float32) + 1.0   # every head weighted differently
    assert orc.score(p)[0, 0] == 4.0 * 12.0            # w[3] = 4


def pin_sum_over_heads_and_dims(orc):
    # q = 1 everywhere, key = 1 everywhere, scale 1/4: every head's product is 128/4 = 32.
    p = blank_problem([1], [0], [1])
    p.q[:] = bf16_bits([1.0])[0]
    set_key(p, 0, 0, {d: 1.0 for d in range(D)}, scale=0.25)
    p.w[0, :] = (np.arange(H, dtype=np.float32) - 32.0) / 64.0
    # sum_h (h - 32)/64 * 32 = (2016 - 2048) / 2 = -16
    assert orc.score(p)[0, 0] == -16.0


def pin_page_table_scale_and_bound(orc):
    # 200 positions over 4 pages, stored in the physical order 2, 0, 3, 1.
    L = 200
    p = blank_problem([L], [0, 0], [L, 150], page_table=[[2, 0, 3, 1]], P=4)
    set_q(p, 0, 0, 0, 1.0)
    set_q(p, 1, 0, 0, 1.0)
    p.w[:, 0] = 1.0
    val = lambda t: float((t * 7) % 15 + 1)
    scl = lambda t: 2.0 ** -(t % 4)
    for t in range(L):
        set_key(p, 0, t, {0: val(t)}, scale=scl(t))
    s = orc.score(p, ld=L + 1)
    for t in range(L):
        assert s[0, t] == val(t) * scl(t), t
    for t in range(150):
        assert s[1, t] == val(t) * scl(t), t
    assert np.isnan(s[0, L]), "position at the bound must not be scored"
    assert np.all(np.isnan(s[1, 150:])), "positions at or past the bound must not be scored"


def pin_long_page_table(orc):
    # 64 full pages in a shuffled physical order: position t holds value v(t) at dim 0.
    L = 64 * PG
    perm = np.random.default_rng(5).permutation(64).astype(np.int32)
    p = blank_problem([L], [0], [L], page_table=[perm], P=64)
    set_q(p, 0, 0, 0, 1.0)
    p.w[0, 0] = 1.0
    val = lambda t: float((3 * (t // PG) + t) % 16 + 1)   # depends on both page and slot
    codes = {v: e4m3_codes([v])[0] for v in range(1, 17)}
    for t in range(L):
        p.k_cache[perm[t // PG], t % PG, 0] = codes[int(val(t))]
    s = orc.score(p)
    assert np.array_equal(s[0], np.array([val(t) for t in range(L)]))


def pin_row_to_request(orc):
    # request 0 holds keys of value 1, request 1 of value 3; rows listed as [req 1, req 0].
    p = blank_problem([64, 64], [1, 0], [64, 64])
    for t in range(64):
        set_key(p, 0, t, {7: 1.0}, scale=1.0)
        set_key(p, 1, t, {7: 3.0}, scale=1.0)
    for r in range(2):
        set_q(p, r, 9, 7, 1.0)
        p.w[r, 9] = 1.0
    s = orc.score(p)
    assert np.all(s[0] == 3.0) and np.all(s[1] == 1.0)


def pin_bf16_cache(orc):
    # bf16 keys (scale 1, k_scale absent); 1 + 2^-7 is exact in bf16 but not in E4M3.
    p = blank_problem([3], [0], [3], kv="bf16")
    set_q(p, 0, 0, 0, 1.0)
    set_q(p, 0, 0, 1, 2.0)
    p.w[0, 0] = 1.0
    set_key(p, 0, 0, {0: 1.0 + 2.0 ** -7})
    set_key(p, 0, 1, {0: -1.0, 1: 1.5})
    set_key(p, 0, 2, {0: -4.0, 1: 1.0})
    s = orc.score(p)
    assert s[0, 0] == 1.0 + 2.0 ** -7
    assert s[0, 1] == -1.0 + 2.0 * 1.5
    assert s[0, 2] == 0.0


def pin_einsum_scorer(orc):
    # An independent implementation: torch decodes, numpy einsum contracts in float64.
    p = workloads.build("einsum", [300, 129, 64], [2, 1, 3], "e4m3", seed=11, dup_frac=0.05)
    got = orc.score(p)
    kd = torch.from_numpy(p.k_cache.copy()).view(torch.float8_e4m3fn).double().numpy()
    q = torch.from_numpy(p.q.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    for r in range(p.R):
        b = int(p.row_bound[r])
        t = np.arange(b)
        pages = p.page_table[p.row_req[r], t // PG]
        keys = kd[pages, t % PG]                       # [b][128]
        sc = p.k_scale[pages, t % PG].astype(np.float64)
        dots = np.einsum("hd,td->th", q[r], keys) * sc[:, None]
        ref = (np.maximum(dots, 0.0) * p.w[r].astype(np.float64)[None, :]).sum(axis=1)
        np.testing.assert_allclose(got[r, :b], ref, rtol=1e-12, atol=1e-12)


def pin_score_points(orc):
    p = workloads.build("pts", [500, 70], [3, 2], "e4m3", seed=12)
    full = orc.score(p)
    rows = np.array([0, 0, 1, 2, 3, 4, 4], np.int32)
    pos = np.array([0, 497, 250, 499, 0, 69, 3], np.int64)
    pos = np.minimum(pos, p.row_bound[rows] - 1)
    pts = orc.score_points(p, rows, pos)
    assert np.array_equal(pts, full[rows, pos])


# ---------------------------------------------------------------------------- selection


def _brute(scores, b, K):
    """Python's sorted on (-score, position): the definition by a library sort."""
    order = sorted(range(b), key=lambda t: (-float(scores[t]), t))
    out = [-1] * K
    for j in range(min(K, b)):
        out[j] = order[j]
    return out


def pin_topk_bruteforce(orc):
    rng = np.random.default_rng(13)
    for trial in range(40):
        R = 3
        ld = int(rng.integers(1, 80))
        kind = trial % 4
        if kind == 0:
            s = rng.standard_normal((R, ld)).astype(np.float32)
        elif kind == 1:
            s = rng.integers(-3, 4, size=(R, ld)).astype(np.float32)      # heavy ties
        elif kind == 2:
            s = np.zeros((R, ld), np.float32)
            s[:, ::2] = -0.0                                               # -0 == +0
        else:
            s = np.full((R, ld), 1.5, np.float32)                          # all equal
        bounds = rng.integers(0, ld + 1, size=R).astype(np.int32)
        for K in (1, 5, 64, 2048):
            got = orc.topk(s, bounds, K)
            for r in range(R):
                assert list(got[r]) == _brute(s[r], int(bounds[r]), K)


def pin_topk_exhaustive_small(orc):
    vals = [2.0, 1.0, 1.0, 0.0, -0.0, -1.0, 3.0]
    for n in range(1, 8):
        for perm in itertools.permutations(range(n)):
            s = np.array([[vals[i] for i in perm]], np.float32)
            for K in (1, 3, 8):
                got = orc.topk(s, np.array([n], np.int32), K)[0]
                assert list(got) == _brute(s[0], n, K)


def pin_topk_invariants(orc):
    rng = np.random.default_rng(14)
    s = (rng.standard_normal((4, 20000)) * 8).astype(np.float32)
    s[:, 100:200] = s[0, 50]                       # a block of equal scores
    bounds = np.array([20000, 19999, 2049, 2047], np.int32)
    K = 2048
    idx = orc.topk(s, bounds, K)
    for r in range(4):
        b, n = int(bounds[r]), min(K, int(bounds[r]))
        sel = idx[r, :n]
        assert np.all(idx[r, n:] == -1)
        assert np.unique(sel).size == n and sel.min() >= 0 and sel.max() < b
        ss = s[r, sel]
        assert np.all(np.diff(ss) <= 0)
        assert np.all(np.diff(sel)[np.diff(ss) == 0] > 0)
        rest = np.setdiff1d(np.arange(b), sel)
        if rest.size:
            kth = ss[-1]
            assert np.all(s[r, rest] <= kth)
            tied = rest[s[r, rest] == kth]
            assert tied.size == 0 or tied.min() > sel[ss == kth].max()


def pin_topk_padding(orc):
    s = np.arange(10, dtype=np.float32)[None, :].repeat(3, 0)
    idx = orc.topk(s, np.array([0, 3, 10], np.int32), 6)
    assert list(idx[0]) == [-1] * 6
    assert list(idx[1]) == [2, 1, 0, -1, -1, -1]
    assert list(idx[2]) == [9, 8, 7, 6, 5, 4]


# ---------------------------------------------------------------------------- radix key


def _f32(bits):
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def _sweep():
    vals = [0.0, -0.0, float("inf"), float("-inf")]
    for e in range(0, 255):
        for m in (0, 1, 0x2AAAAA, 0x7FFFFF):
            vals.append(_f32((e << 23) | m))
            vals.append(_f32(0x80000000 | (e << 23) | m))
    return np.array(vals, np.float32)


def pin_radix_key_monotone(orc):
    x = np.sort(_sweep().astype(np.float64)).astype(np.float32)
    k = orc.radix_key(x).astype(np.int64)
    for a, b, ka, kb in zip(x[:-1], x[1:], k[:-1], k[1:]):
        if a < b:
            assert ka < kb, (a, b)
        else:
            assert ka == kb, (a, b)            # includes -0.0 == +0.0


def closed_form_digit(x):
    """First digit from sign and biased exponent E: 32 + E//8 for x >= 0, 31 - E//8 below."""
    x = np.float32(x)
    if x == 0:
        return 32
    bits = struct.unpack("<I", struct.pack("<f", float(x)))[0]
    E = (bits >> 23) & 0xFF
    return 32 + (E >> 3) if x > 0 else 31 - (E >> 3)


def pin_radix_first_digit(orc):
    x = _sweep()
    k = orc.radix_key(x)
    for v, kv in zip(x, k):
        assert int(kv) >> 26 == closed_form_digit(v), v


def pin_first_digit_hist(orc):
    rng = np.random.default_rng(15)
    s = (rng.standard_normal((3, 5000)) * np.array([[1.0], [8.0], [1e-3]])).astype(np.float32)
    s[0, :10] = -0.0
    bounds = np.array([5000, 1234, 0], np.int32)
    hist = orc.first_digit_hist(s, bounds)
    for r in range(3):
        digits = [closed_form_digit(v) for v in s[r, :bounds[r]]]
        assert np.array_equal(hist[r], np.bincount(np.array(digits, dtype=np.int64), minlength=64))


def _top1_by_definition(row):
    """The top-1 by its statement, with Python's max: the largest value, NaN read as
    -1e30, the lowest index among equal values (max over (value, -index))."""
    vals = [(-1e30 if np.isnan(v) else float(v)) for v in row]
    j = max(range(len(vals)), key=lambda i: (vals[i], -i))
    return j, vals[j]


def pin_top1_bruteforce(orc):
    rng = np.random.default_rng(21)
    x = rng.integers(-4, 5, size=(40, 37)).astype(np.float32)    # many ties
    x[::7, 3] = np.nan
    idx, val = orc.top1(x)
    for r in range(x.shape[0]):
        j, v = _top1_by_definition(x[r])
        assert idx[r] == j and np.float32(val[r]) == np.float32(v), (r, idx[r], j)


def pin_top1_special_values(orc):
    rows = np.array([
        [np.nan, np.nan, np.nan, np.nan],            # all NaN: index 0, value -1e30
        [-np.inf, np.nan, -1e31, -np.inf],           # NaN (-1e30) beats -inf and -1e31
        [-0.0, 0.0, -1.0, -0.0],                     # -0.0 and +0.0 tie: index 0
        [1.0, np.inf, 3.0, np.inf],                  # +inf, lowest index
        [-1e30, np.nan, -2e30, -1e30],               # NaN ties with -1e30: index 0
    ], np.float32)
    idx, val = orc.top1(rows)
    assert list(idx) == [0, 1, 0, 1, 0], list(idx)
    assert val[0] == np.float32(-1e30) and val[1] == np.float32(-1e30) and val[2] == 0.0
    assert np.isinf(val[3]) and val[3] > 0 and val[4] == np.float32(-1e30)


def _lib_e4m3(x):
    """Library encoder: torch's float8_e4m3fn cast (round to nearest even) after
    clamping to the largest finite value."""
    x = np.clip(np.asarray(x, dtype=np.float32), -448.0, 448.0)
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pin_e4m3_encode_vs_library(orc):
    rng = np.random.default_rng(31)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = orc.e4m3_to_double(finite).astype(np.float32)
    pos = np.sort(vals[vals > 0])
    mids = ((pos[:-1].astype(np.float64) + pos[1:]) / 2).astype(np.float32)     # exact ties
    rand = (rng.choice([-1, 1], 4000) * np.exp(rng.uniform(np.log(1e-5), np.log(1e3), 4000))).astype(np.float32)
    x = np.concatenate([vals, mids, -mids, rand, np.array([0.0, -0.0, 448.0, 449.0, 1e9, -1e9], np.float32)])
    assert np.array_equal(orc.e4m3_encode(x), _lib_e4m3(x))


def pin_e4m3_encode_roundtrip(orc):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    back = orc.e4m3_encode(orc.e4m3_to_double(codes).astype(np.float32))
    assert np.array_equal(back, codes)


def pin_quantize_key(orc):
    rng = np.random.default_rng(32)
    for amp in (1.0, 1e-4, 300.0):
        x = (rng.standard_normal(128) * amp).astype(np.float32)
        bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
        scale = np.float32(np.abs(xb).max()) / np.float32(448.0)
        codes, sc = orc.quantize_key(bits)
        assert sc == scale
        assert np.array_equal(codes, _lib_e4m3(xb / scale))
        assert codes[np.argmax(np.abs(xb))] & 0x7F == 126          # the largest value maps to +-448
    codes, sc = orc.quantize_key(np.zeros(128, np.uint16))
    assert sc == np.float32(1.0) and not codes.any()


def pin_patch_position(orc):
    """New keys land at hand-worked cache cells.  Page table [[5, 2, 7], [0, 3, 1]]
    over 8 pages; a row's key goes to logical position bound - 1:
      request 0, bound 70  -> t = 69:  page index 1 -> page 2, slot 5
      request 0, bound 129 -> t = 128: page index 2 -> page 7, slot 0
      request 0, bound 1   -> t = 0:   page index 0 -> page 5, slot 0
      request 1, bound 64  -> t = 63:  page index 0 -> page 0, slot 63
      request 0, bound 0   -> no key
    Every other cell keeps its bytes (and scale)."""
    expect = {(2, 5): 0, (7, 0): 1, (5, 0): 2, (0, 63): 3}      # cell -> row whose key it holds
    rng = np.random.default_rng(34)
    for kv in ("e4m3", "bf16"):
        R, P = 5, 8
        k_new = torch.from_numpy((rng.standard_normal((R, 128)) + 0.5).astype(np.float32)).to(torch.bfloat16) \
            .view(torch.int16).numpy().view(np.uint16)
        prob = workloads.Problem(
            name="patch_literal", q=np.zeros((R, 64, 128), np.uint16), w=np.zeros((R, 64), np.float32),
            k_cache=np.zeros((P, 64, 128), np.uint8 if kv == "e4m3" else np.uint16),
            k_scale=np.full((P, 64), 0.5, np.float32) if kv == "e4m3" else None,
            page_table=np.array([[5, 2, 7], [0, 3, 1]], np.int32),
            row_req=np.array([0, 0, 0, 1, 0], np.int32), row_bound=np.array([70, 129, 1, 64, 0], np.int32),
            kv_dtype=kv)
        out = orc.patch_new_keys(prob, k_new)
        changed = {tuple(c) for c in np.argwhere((out.k_cache != prob.k_cache).any(axis=2)).tolist()}
        assert changed == set(expect), (kv, sorted(changed))
        for (page, slot), r in expect.items():
            if kv == "e4m3":
                codes, sc = orc.quantize_key(k_new[r])
                assert np.array_equal(out.k_cache[page, slot], codes) and out.k_scale[page, slot] == sc
            else:
                assert np.array_equal(out.k_cache[page, slot], k_new[r])
        if kv == "e4m3":
            moved = {tuple(c) for c in np.argwhere(out.k_scale != prob.k_scale).tolist()}
            assert moved <= set(expect), sorted(moved)


def _split_topk(orc, scores, bounds, cuts, K):
    """Each part [cuts[s], cuts[s+1]) of every row ranked on its own: positions in
    the part's numbering and their scores, as a key-sharded indexer produces them."""
    R = scores.shape[0]
    S = len(cuts) - 1
    pi = np.full((S, R, K), -1, np.int32)
    ps = np.zeros((S, R, K), np.float32)
    for si in range(S):
        a, b = cuts[si], cuts[si + 1]
        sub = np.ascontiguousarray(scores[:, a:b])
        sb = np.clip(bounds - a, 0, b - a).astype(np.int32)
        idx = orc.topk(sub, sb, K)
        pi[si] = idx
        for r in range(R):
            ok = idx[r] >= 0
            ps[si, r, ok] = sub[r, idx[r, ok]]
    return pi, ps


def pin_merge_equals_unsharded_topk(orc):
    """The merge of the parts' own top-K lists equals the top-K of the whole rows
    (a different path: oracle_topk over the scores), for 2, 3 and 8 parts, with
    ties across part edges and rows whose bound is below K or inside a part."""
    rng = np.random.default_rng(51)
    R, L, K = 4, 3000, 256
    scores = rng.integers(-40, 40, (R, L)).astype(np.float32)     # heavy ties
    scores[1] = rng.standard_normal(L).astype(np.float32)
    bounds = np.array([L, L - 17, 200, 1234], np.int32)
    full = orc.topk(scores, bounds, K)
    for cuts in ([0, 1500, L], [0, 64, 2000, L], list(np.linspace(0, L, 9).astype(int))):
        pi, ps = _split_topk(orc, scores, bounds, cuts, K)
        got = orc.merge_topk(pi, ps, np.array(cuts[:-1], np.int32), K)
        assert np.array_equal(got, full), cuts


def pin_merge_bruteforce(orc):
    """Tiny random parts against Python's sorted over the union (score descending,
    position ascending), including empty entries and equal scores."""
    rng = np.random.default_rng(52)
    for _ in range(30):
        S, R, Kin, K = int(rng.integers(1, 5)), 2, int(rng.integers(1, 6)), int(rng.integers(1, 9))
        offsets = np.cumsum(rng.integers(0, 20, S)).astype(np.int32)
        pi = np.full((S, R, Kin), -1, np.int32)
        ps = np.zeros((S, R, Kin), np.float32)
        for s_ in range(S):
            for r in range(R):
                n = int(rng.integers(0, Kin + 1))
                pos = rng.choice(20, size=n, replace=False)
                pi[s_, r, :n] = pos
                ps[s_, r, :n] = rng.integers(-3, 3, n)
        got = orc.merge_topk(pi, ps, offsets, K)
        for r in range(R):
            pairs = [(float(ps[s_, r, j]), int(pi[s_, r, j]) + int(offsets[s_]))
                     for s_ in range(S) for j in range(Kin) if pi[s_, r, j] >= 0]
            want = [p for _, p in sorted(pairs, key=lambda t: (-t[0], t[1]))][:K]
            want += [-1] * (K - len(want))
            assert list(got[r]) == want, (got[r], want)


ALL_PINS = [
    pin_e4m3_all_codes, pin_e4m3_closed_forms, pin_bf16_decode,
    pin_long_page_table, pin_page_table_scale_and_bound,
    pin_relu_and_signed_weights, pin_head_dim_layout, pin_sum_over_heads_and_dims,
    pin_row_to_request, pin_bf16_cache, pin_einsum_scorer,
    pin_score_points, pin_topk_bruteforce, pin_topk_exhaustive_small, pin_topk_invariants,
    pin_topk_padding, pin_radix_key_monotone, pin_radix_first_digit, pin_first_digit_hist,
    pin_top1_bruteforce, pin_top1_special_values,
    pin_e4m3_encode_vs_library, pin_e4m3_encode_roundtrip, pin_quantize_key, pin_patch_position,
    pin_merge_equals_unsharded_topk, pin_merge_bruteforce,
]
