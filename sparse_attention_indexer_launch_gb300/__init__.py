"""Python binding of libidx.so, the GB300 decode indexer (C ABI in include/idx.h).

Argument marshalling only: every step of the indexer runs in the library's
CUDA kernels.  torch supplies device memory and streams.  If the library has
not been built, importing this package raises; there is no other code path.

    idx_score   scores of every visible key of every row (+ first-digit histogram)
    idx_topk    exact top-K positions of given scores
    idx_launch  both, fused on one stream
    idx_launch_host  idx_launch on host inputs, copies included
    idx_launch_scored, idx_merge_topk  the key-sharded indexer (shard.py splits
                     a problem and exchanges the shards' lists)
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libidx.so")

IDX_OK, IDX_EINVAL, IDX_EUNSUPPORTED, IDX_ECUDA, IDX_ETIMEOUT, IDX_EDEVICE = range(6)
IDX_KV_E4M3, IDX_KV_BF16 = 0, 1
IDX_HEADS, IDX_DIM, IDX_PAGE, IDX_MAX_K = 64, 128, 64, 2048
IDX_DEBUG_WAIT_LIMIT_NS, IDX_DEBUG_STALL_SCORE_MMA = 1, 2

EXPORTS = ["idx_workspace_size", "idx_score", "idx_topk", "idx_launch", "idx_host_arena_size",
           "idx_launch_host", "idx_last_device_status", "idx_status_string", "idx_version",
           "idx_debug_set", "idx_profile_events", "idx_top1_state_size", "idx_top1", "idx_topk_noalloc",
           "idx_patch_new_keys", "idx_launch_scored", "idx_merge_topk", "idx_launch_new_keys"]


class IdxError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class Problem(ctypes.Structure):
    """Mirror of idx_problem."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("w", ctypes.c_void_p), ("k_cache", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p), ("page_table", ctypes.c_void_p), ("row_req", ctypes.c_void_p),
        ("row_bound", ctypes.c_void_p), ("R", ctypes.c_int32), ("Q", ctypes.c_int32),
        ("P", ctypes.c_int64), ("pt_stride", ctypes.c_int32), ("max_bound", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32), ("rows_hint", ctypes.c_int32),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libidx.so is not built ({LIB_PATH}); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(Problem)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.idx_workspace_size.argtypes = [P, i32]
    lib.idx_workspace_size.restype = sz
    lib.idx_score.argtypes = [P, vp, i64, vp, vp, sz, vp]
    lib.idx_score.restype = ctypes.c_int
    lib.idx_topk.argtypes = [vp, i64, vp, i32, i32, i32, vp, vp, vp, sz, vp]
    lib.idx_topk.restype = ctypes.c_int
    lib.idx_launch.argtypes = [P, i32, vp, vp, sz, vp]
    lib.idx_launch.restype = ctypes.c_int
    lib.idx_host_arena_size.argtypes = [P, i32]
    lib.idx_host_arena_size.restype = sz
    lib.idx_launch_host.argtypes = [P, i32, vp, vp, sz, vp]
    lib.idx_launch_host.restype = ctypes.c_int
    lib.idx_last_device_status.argtypes = [vp, vp]
    lib.idx_last_device_status.restype = ctypes.c_int
    lib.idx_status_string.argtypes = [ctypes.c_int]
    lib.idx_status_string.restype = ctypes.c_char_p
    lib.idx_version.argtypes = []
    lib.idx_version.restype = i32
    lib.idx_debug_set.argtypes = [i32, i64]
    lib.idx_debug_set.restype = i64
    lib.idx_profile_events.argtypes = [vp, vp]
    lib.idx_profile_events.restype = None
    lib.idx_patch_new_keys.argtypes = [P, vp, vp]
    lib.idx_patch_new_keys.restype = ctypes.c_int
    lib.idx_top1_state_size.argtypes = [i32]
    lib.idx_top1_state_size.restype = sz
    lib.idx_top1.argtypes = [vp, i64, i32, i64, vp, vp, vp, i64, i32, vp, vp, sz, vp]
    lib.idx_top1.restype = ctypes.c_int
    lib.idx_topk_noalloc.argtypes = [vp, i64, vp, i32, i32, i32, vp, vp]
    lib.idx_topk_noalloc.restype = ctypes.c_int
    lib.idx_launch_scored.argtypes = [P, i32, vp, vp, vp, sz, vp]
    lib.idx_launch_scored.restype = ctypes.c_int
    lib.idx_merge_topk.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32), i32, i32, i32, i32, vp, vp, vp]
    lib.idx_merge_topk.restype = ctypes.c_int
    lib.idx_launch_new_keys.argtypes = [P, vp, i32, vp, vp, sz, vp]
    lib.idx_launch_new_keys.restype = ctypes.c_int
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.idx_status_string(status).decode()


def _check(status: int, what: str):
    if status != IDX_OK:
        raise IdxError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_problem(q, w, k_cache, k_scale, page_table, row_req, row_bound, max_bound: int,
                 kv_dtype: int, P: int | None = None, rows_hint: int = 0) -> Problem:
    """idx_problem from tensors (device tensors for the device calls, host tensors
    for idx_launch_host).  Shapes: q [R][64][128] bf16, w [R][64] fp32, k_cache
    [P][64][128] uint8 (E4M3 bytes) or bf16, k_scale [P][64] fp32 or None,
    page_table [Q][stride] int32, row_req and row_bound [R] int32.  rows_hint: the
    most rows any request has (0: unknown)."""
    R = int(row_bound.shape[0])
    return Problem(q=_ptr(q), w=_ptr(w), k_cache=_ptr(k_cache), k_scale=_ptr(k_scale),
                   page_table=_ptr(page_table), row_req=_ptr(row_req), row_bound=_ptr(row_bound),
                   R=R, Q=int(page_table.shape[0]), P=int(P if P is not None else k_cache.shape[0]),
                   pt_stride=int(page_table.shape[1]), max_bound=int(max_bound), kv_dtype=int(kv_dtype),
                   rows_hint=int(rows_hint))


def workspace_size(problem: Problem, K: int) -> int:
    return int(lib.idx_workspace_size(ctypes.byref(problem), int(K)))


def host_arena_size(problem: Problem, K: int) -> int:
    return int(lib.idx_host_arena_size(ctypes.byref(problem), int(K)))


def idx_score(problem: Problem, scores, ld: int, hist, ws, stream=None):
    _check(lib.idx_score(ctypes.byref(problem), _ptr(scores), int(ld), _ptr(hist), _ptr(ws),
                         ws.numel() * ws.element_size(), _stream(stream)), "idx_score")


def idx_topk(scores, ld: int, row_bound, R: int, max_bound: int, K: int, hist, out_idx, ws,
             stream=None):
    _check(lib.idx_topk(_ptr(scores), int(ld), _ptr(row_bound), int(R), int(max_bound), int(K),
                        _ptr(hist), _ptr(out_idx), _ptr(ws), ws.numel() * ws.element_size(),
                        _stream(stream)), "idx_topk")


def idx_patch_new_keys(problem: Problem, k_new, stream=None):
    """Writes each row's new key (bf16 [R][128] device tensor) into the problem's
    cache at position row_bound - 1 (see idx.h)."""
    _check(lib.idx_patch_new_keys(ctypes.byref(problem), _ptr(k_new), _stream(stream)), "idx_patch_new_keys")


def top1_state_size(R: int) -> int:
    return int(lib.idx_top1_state_size(int(R)))


def idx_top1(logits, out_idx, state, out_val=None, tokens=None, token_col: int = 0, positions=None,
             V: int | None = None, stream=None):
    """Top-1 of each row of a [R][ld] fp32 tensor (see idx.h); `state` is a zeroed
    uint8 device tensor of top1_state_size(R) bytes, left zero by every call."""
    R, ld = int(logits.shape[0]), int(logits.stride(0))
    V = int(V if V is not None else logits.shape[1])
    tokens_ld = int(tokens.stride(0)) if tokens is not None else 0
    _check(lib.idx_top1(_ptr(logits), ld, R, V, _ptr(out_idx), _ptr(out_val), _ptr(tokens), tokens_ld,
                        int(token_col), _ptr(positions), _ptr(state), state.numel() * state.element_size(),
                        _stream(stream)), "idx_top1")


def idx_topk_noalloc(scores, ld: int, row_bound, R: int, max_bound: int, K: int, out_idx, stream=None):
    _check(lib.idx_topk_noalloc(_ptr(scores), int(ld), _ptr(row_bound), int(R), int(max_bound), int(K),
                                _ptr(out_idx), _stream(stream)), "idx_topk_noalloc")


def idx_launch(problem: Problem, K: int, out_idx, ws, stream=None):
    _check(lib.idx_launch(ctypes.byref(problem), int(K), _ptr(out_idx), _ptr(ws),
                          ws.numel() * ws.element_size(), _stream(stream)), "idx_launch")


def idx_launch_new_keys(problem: Problem, k_new, K: int, out_idx, ws, stream=None):
    """idx_launch with every row's new key (bf16 [R][128] device tensor) written
    into the problem's cache first, inside the launch (see idx.h)."""
    _check(lib.idx_launch_new_keys(ctypes.byref(problem), _ptr(k_new), int(K), _ptr(out_idx), _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)), "idx_launch_new_keys")


def idx_launch_scored(problem: Problem, K: int, out_idx, out_score, ws, stream=None):
    _check(lib.idx_launch_scored(ctypes.byref(problem), int(K), _ptr(out_idx), _ptr(out_score), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream)), "idx_launch_scored")


def idx_merge_topk(part_idx, part_score, offsets, K: int, out_idx, out_score=None, stream=None):
    """part_idx / part_score: [S][R][Kin] device tensors (int32 / fp32); offsets: S
    host integers; out_idx [R][K] (and out_score [R][K]) device tensors."""
    S, R, Kin = (int(x) for x in part_idx.shape)
    off = (ctypes.c_int32 * S)(*[int(o) for o in offsets])
    _check(lib.idx_merge_topk(_ptr(part_idx), _ptr(part_score), off, S, R, Kin, int(K), _ptr(out_idx),
                              _ptr(out_score), _stream(stream)), "idx_merge_topk")


def idx_launch_host(host_problem: Problem, K: int, host_out, arena, stream=None):
    _check(lib.idx_launch_host(ctypes.byref(host_problem), int(K), _ptr(host_out), _ptr(arena),
                               arena.numel() * arena.element_size(), _stream(stream)),
           "idx_launch_host")


def last_device_status(ws, stream=None) -> int:
    return int(lib.idx_last_device_status(_ptr(ws), _stream(stream)))


def profile_next_score(start_event, stop_event):
    """Time the next scoring kernel with two torch.cuda.Event(enable_timing=True)."""
    lib.idx_profile_events(ctypes.c_void_p(start_event.cuda_event), ctypes.c_void_p(stop_event.cuda_event))


def version() -> int:
    return int(lib.idx_version())


def debug_set(what: int, value: int) -> int:
    return int(lib.idx_debug_set(int(what), int(value)))


def alloc_bytes(nbytes: int, device="cuda"):
    """A uint8 device buffer whose base is 1024-byte aligned (the caching allocator's
    blocks are 512-aligned, so one spare KB is taken and the view offset)."""
    import torch
    raw = torch.empty(int(nbytes) + 1024, dtype=torch.uint8, device=device)
    off = (-raw.data_ptr()) % 1024
    return raw[off:off + int(nbytes)]


class DeviceProblem:
    """A workloads.Problem uploaded to the GPU (plain tensor copies), with its
    idx_problem and a workspace."""

    def __init__(self, prob, device="cuda", K: int | None = None, max_bound: int | None = None,
                 rows_hint: int | None = None):
        """rows_hint: idx_problem.rows_hint; None counts the rows of each request
        in the host problem's row map."""
        import numpy as np
        import torch
        self.host = prob
        self.K = int(K if K is not None else prob.K)
        dev = torch.device(device)
        self.q = torch.from_numpy(prob.q.view(np.int16)).to(dev).view(torch.bfloat16)
        self.w = torch.from_numpy(prob.w).to(dev)
        if prob.kv_dtype == "e4m3":
            self.k_cache = torch.from_numpy(prob.k_cache).to(dev)
            self.k_scale = torch.from_numpy(prob.k_scale).to(dev)
            self.kv = IDX_KV_E4M3
        else:
            self.k_cache = torch.from_numpy(prob.k_cache.view(np.int16)).to(dev).view(torch.bfloat16)
            self.k_scale = None
            self.kv = IDX_KV_BF16
        self.page_table = torch.from_numpy(prob.page_table).to(dev)
        self.row_req = torch.from_numpy(prob.row_req).to(dev)
        self.row_bound = torch.from_numpy(prob.row_bound).to(dev)
        self.max_bound = int(max_bound if max_bound is not None else max(prob.max_bound, 0))
        if rows_hint is None:
            req = np.asarray(prob.row_req)
            rows_hint = int(np.bincount(req[req >= 0]).max()) if (req >= 0).any() else 0
        self.problem = make_problem(self.q, self.w, self.k_cache, self.k_scale, self.page_table,
                                    self.row_req, self.row_bound, self.max_bound, self.kv, P=prob.P,
                                    rows_hint=rows_hint)
        self.ws = alloc_bytes(workspace_size(self.problem, self.K), dev)
        self.R = prob.R

    def score(self, ld: int | None = None, with_hist: bool = True, stream=None):
        import torch
        ld = int(ld if ld is not None else max(self.max_bound, 1))
        scores = torch.full((self.R, ld), float("nan"), dtype=torch.float32, device=self.q.device)
        # uint32 counts held in an int32 tensor (counts stay below 2^31)
        hist = torch.zeros((self.R, 64), dtype=torch.int32, device=self.q.device) if with_hist else None
        idx_score(self.problem, scores, ld, hist, self.ws, stream)
        return scores, hist

    def topk(self, scores, hist=None, K: int | None = None, stream=None):
        import torch
        K = int(K if K is not None else self.K)
        out = torch.empty((self.R, K), dtype=torch.int32, device=self.q.device)
        idx_topk(scores, scores.shape[1], self.row_bound, self.R, self.max_bound, K, hist, out,
                 self.ws, stream)
        return out

    def launch(self, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty((self.R, self.K), dtype=torch.int32, device=self.q.device)
        idx_launch(self.problem, self.K, out, self.ws, stream)
        return out

    def launch_scored(self, out=None, out_score=None, stream=None):
        import torch
        if out is None:
            out = torch.empty((self.R, self.K), dtype=torch.int32, device=self.q.device)
        if out_score is None:
            out_score = torch.empty((self.R, self.K), dtype=torch.float32, device=self.q.device)
        idx_launch_scored(self.problem, self.K, out, out_score, self.ws, stream)
        return out, out_score

    def status(self, stream=None) -> int:
        return last_device_status(self.ws, stream)
