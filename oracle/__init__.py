"""CPU oracle for the decode indexer: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and it
never calls the CUDA library; the two share no code.  The arithmetic lives in
``oracle.c`` (plain C, IEEE double); this module only compiles that file with
gcc into ``_build/liboracle.so`` and marshals numpy arrays to it.

What it computes is the method of the sglang PR 48224 page (sgl-amd-mono #86):
every cached key of each row scored (section Motivation, first paragraph),
positions from a row's bound on left out (section Modifications, commit 2), each
row's exact top-2048 selected (section Motivation; section Accuracy Tests), and
the first radix digit ``radix_key >> 26`` over 64 bins (section Modifications,
commit 4).  The score formula is sum_h w_h * ReLU(scale * <q_h, k>) over 64
heads of 128 dims.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

HEADS = 64
DIM = 128
PAGE = 64
KV_E4M3 = 0
KV_BF16 = 1


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (OpenMP, no target-specific flags)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    i32 = ctypes.c_int
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_score.argtypes = [p, p, p, i32, p, p, i64, p, p, i32, i64, p, i64]
    lib.oracle_score.restype = i32
    lib.oracle_score_points.argtypes = [p, p, p, i32, p, p, i64, p, p, i64, p, p, i64, p]
    lib.oracle_score_points.restype = i32
    lib.oracle_topk.argtypes = [p, i64, p, i32, i32, p]
    lib.oracle_topk.restype = i32
    lib.oracle_radix_key.argtypes = [ctypes.c_float]
    lib.oracle_radix_key.restype = ctypes.c_uint32
    lib.oracle_first_digit_hist.argtypes = [p, i64, p, i32, p]
    lib.oracle_first_digit_hist.restype = None
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_quantize_key.argtypes = [p, p, p]
    lib.oracle_quantize_key.restype = None
    lib.oracle_patch_new_keys.argtypes = [p, p, p, i32, p, i64, i32, p, p, i32, i64]
    lib.oracle_patch_new_keys.restype = i32
    lib.oracle_merge_topk.argtypes = [p, p, p, i32, i32, i32, i32, p]
    lib.oracle_merge_topk.restype = i32
    lib.oracle_top1.argtypes = [p, i64, i32, i64, p, p]
    lib.oracle_top1.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i32
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _kv(prob):
    if prob.kv_dtype == "e4m3":
        return KV_E4M3, _c(prob.k_cache, np.uint8), _c(prob.k_scale, np.float32)
    if prob.kv_dtype == "bf16":
        return KV_BF16, _c(prob.k_cache, np.uint16), None
    raise ValueError(prob.kv_dtype)


class Oracle:
    """numpy front end over one compiled copy of oracle.c."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        self.lib = _bind(lib_path)

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def e4m3_to_double(self, codes) -> np.ndarray:
        codes = np.asarray(codes, dtype=np.uint8)
        f = self.lib.oracle_e4m3_to_double
        return np.array([f(int(c)) for c in codes.ravel()], dtype=np.float64).reshape(codes.shape)

    def bf16_to_double(self, bits) -> np.ndarray:
        bits = np.asarray(bits, dtype=np.uint16)
        f = self.lib.oracle_bf16_to_double
        return np.array([f(int(b)) for b in bits.ravel()], dtype=np.float64).reshape(bits.shape)

    def score(self, prob, ld: int | None = None) -> np.ndarray:
        """Double-precision scores [R][ld]; positions from a row's bound on are NaN."""
        kv, kc, ks = _kv(prob)
        q = _c(prob.q, np.uint16)
        w = _c(prob.w, np.float32)
        pt = _c(prob.page_table, np.int32)
        rr = _c(prob.row_req, np.int32)
        rb = _c(prob.row_bound, np.int32)
        R = rb.shape[0]
        ld = int(ld if ld is not None else max(1, int(rb.max(initial=0))))
        out = np.full((R, ld), np.nan, dtype=np.float64)
        rc = self.lib.oracle_score(_ptr(q), _ptr(w), _ptr(kc), kv, _ptr(ks), _ptr(pt), pt.shape[1],
                                   _ptr(rr), _ptr(rb), R, kc.shape[0], _ptr(out), ld)
        if rc != 0:
            raise ValueError("oracle_score: argument out of range")
        return out

    def score_points(self, prob, rows, pos) -> np.ndarray:
        """Double-precision scores at the given (row, position) points."""
        kv, kc, ks = _kv(prob)
        q = _c(prob.q, np.uint16)
        w = _c(prob.w, np.float32)
        pt = _c(prob.page_table, np.int32)
        rr = _c(prob.row_req, np.int32)
        rb = _c(prob.row_bound, np.int32)
        rows = _c(rows, np.int32)
        pos = _c(pos, np.int64)
        out = np.empty(rows.shape[0], dtype=np.float64)
        rc = self.lib.oracle_score_points(_ptr(q), _ptr(w), _ptr(kc), kv, _ptr(ks), _ptr(pt),
                                          pt.shape[1], _ptr(rr), _ptr(rb), kc.shape[0], _ptr(rows),
                                          _ptr(pos), rows.shape[0], _ptr(out))
        if rc != 0:
            raise ValueError("oracle_score_points: point out of range")
        return out

    def topk(self, scores_f32, row_bound, K: int) -> np.ndarray:
        """Exact top-K positions [R][K] (score desc, position asc, -1 padded)."""
        s = _c(scores_f32, np.float32)
        rb = _c(row_bound, np.int32)
        R = rb.shape[0]
        out = np.empty((R, K), dtype=np.int32)
        rc = self.lib.oracle_topk(_ptr(s), s.shape[1], _ptr(rb), R, K, _ptr(out))
        if rc != 0:
            raise ValueError("oracle_topk: NaN score within a bound")
        return out

    def merge_topk(self, part_idx, part_score, offsets, K: int) -> np.ndarray:
        """Exact top-K [R][K] of the union of S parts ([S][R][Kin] positions, -1 for
        none, and scores), part s's positions shifted by offsets[s]."""
        pi = _c(part_idx, np.int32)
        ps = _c(part_score, np.float32)
        off = _c(offsets, np.int32)
        S, R, Kin = pi.shape
        out = np.empty((R, K), dtype=np.int32)
        rc = self.lib.oracle_merge_topk(_ptr(pi), _ptr(ps), _ptr(off), S, R, Kin, K, _ptr(out))
        if rc != 0:
            raise ValueError("oracle_merge_topk: NaN score")
        return out

    def radix_key(self, x) -> np.ndarray:
        x = np.asarray(x, dtype=np.float32)
        f = self.lib.oracle_radix_key
        return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint32).reshape(x.shape)

    def e4m3_encode(self, x) -> np.ndarray:
        x = np.asarray(x, dtype=np.float32).ravel()
        return np.array([self.lib.oracle_e4m3_encode(float(v)) for v in x], dtype=np.uint8)

    def quantize_key(self, key_bf16_bits):
        """(E4M3 codes [128], fp32 scale) of one key given as bf16 bit patterns."""
        k = _c(key_bf16_bits, np.uint16)
        codes = np.empty(128, dtype=np.uint8)
        sc = np.empty(1, dtype=np.float32)
        self.lib.oracle_quantize_key(_ptr(k), _ptr(codes), _ptr(sc))
        return codes, np.float32(sc[0])

    def patch_new_keys(self, prob, k_new_bits):
        """A copy of prob with every row's new key written at its position
        row_bound - 1 (rows with bound 0 write nothing): E4M3 codes and scale, or
        the bf16 values for a bf16 cache (oracle_patch_new_keys)."""
        import copy
        out = copy.copy(prob)
        kv, kc, ks = _kv(prob)
        out.k_cache = kc.copy()
        out.k_scale = None if ks is None else ks.copy()
        kn = _c(k_new_bits, np.uint16)
        rr = _c(prob.row_req, np.int32)
        rb = _c(prob.row_bound, np.int32)
        pt = _c(prob.page_table, np.int32)
        rc = self.lib.oracle_patch_new_keys(_ptr(kn), _ptr(rr), _ptr(rb), rb.shape[0], _ptr(pt), pt.shape[1],
                                            pt.shape[0], _ptr(out.k_cache), _ptr(out.k_scale), kv,
                                            out.k_cache.shape[0])
        if rc != 0:
            raise ValueError("oracle_patch_new_keys: request, bound or page id out of range")
        return out

    def top1(self, logits_f32):
        """(index, value) of each row's largest logit: ties to the lowest index,
        NaN read as -1e30."""
        x = _c(logits_f32, np.float32)
        R, V = x.shape
        idx = np.empty(R, dtype=np.int32)
        val = np.empty(R, dtype=np.float32)
        self.lib.oracle_top1(_ptr(x), V, R, V, _ptr(idx), _ptr(val))
        return idx, val

    def first_digit_hist(self, scores_f32, row_bound) -> np.ndarray:
        s = _c(scores_f32, np.float32)
        rb = _c(row_bound, np.int32)
        R = rb.shape[0]
        out = np.zeros((R, 64), dtype=np.uint32)
        self.lib.oracle_first_digit_hist(_ptr(s), s.shape[1], _ptr(rb), R, _ptr(out))
        return out


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile a (possibly edited) copy of oracle.c; used by the tests that check
    the pins reject planted mistakes."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", src, "-o", out_path,
                    "-lm"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
        return _lib


def num_threads() -> int:
    return default().num_threads()


def e4m3_to_double(codes):
    return default().e4m3_to_double(codes)


def bf16_to_double(bits):
    return default().bf16_to_double(bits)


def score(prob, ld=None):
    return default().score(prob, ld)


def score_points(prob, rows, pos):
    return default().score_points(prob, rows, pos)


def topk(scores_f32, row_bound, K):
    return default().topk(scores_f32, row_bound, K)


def radix_key(x):
    return default().radix_key(x)


def top1(logits_f32):
    return default().top1(logits_f32)


def first_digit_hist(scores_f32, row_bound):
    return default().first_digit_hist(scores_f32, row_bound)
