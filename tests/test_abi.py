"""The C ABI library on the CPU: it loads, exports every declared entry point, and
rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def idxlib():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_indexer_launch_gb300 as lib
    return lib


def declared_functions():
    text = open(os.path.join(ROOT, "include", "idx.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(idx_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["idx_score", "idx_topk", "idx_launch", "idx_workspace_size", "idx_last_device_status",
              "idx_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(idxlib):
    raw = ctypes.CDLL(idxlib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared in idx.h but not exported"
    assert sorted(idxlib.EXPORTS) == declared_functions()


def test_status_strings_and_version(idxlib):
    assert idxlib.status_string(idxlib.IDX_OK) == "ok"
    assert "timeout" in idxlib.status_string(idxlib.IDX_ETIMEOUT) or "time" in idxlib.status_string(idxlib.IDX_ETIMEOUT)
    assert idxlib.version() >= 100


def _fake_problem(idxlib, **kw):
    # Non-null, 16-byte aligned fake addresses: never dereferenced by host-side checks.
    base = dict(q=0x10000, w=0x20000, k_cache=0x30000, k_scale=0x40000, page_table=0x50000,
                row_req=0x60000, row_bound=0x70000, R=4, Q=1, P=64, pt_stride=64, max_bound=4096,
                kv_dtype=idxlib.IDX_KV_E4M3)
    base.update(kw)
    return idxlib.Problem(**base)


def test_workspace_size_and_validation(idxlib):
    p = _fake_problem(idxlib)
    n = idxlib.workspace_size(p, 2048)
    assert n > 4 * 4096 * 4          # holds at least the score scratch
    assert idxlib.workspace_size(p, 2049) == 0
    assert idxlib.workspace_size(p, 0) == 0
    bad = [dict(q=None), dict(R=0), dict(max_bound=64 * 64 + 1), dict(kv_dtype=7), dict(k_scale=None),
           dict(kv_dtype=idxlib.IDX_KV_BF16), dict(q=0x10008), dict(P=0), dict(pt_stride=0), dict(rows_hint=-1)]
    for kw in bad:
        assert idxlib.workspace_size(_fake_problem(idxlib, **kw), 2048) == 0, kw
    ok_bf16 = _fake_problem(idxlib, kv_dtype=idxlib.IDX_KV_BF16, k_scale=None)
    assert idxlib.workspace_size(ok_bf16, 2048) > 0


def test_entry_points_reject_bad_arguments_without_a_gpu(idxlib):
    L = idxlib.lib
    p = _fake_problem(idxlib, q=None)
    vp = ctypes.c_void_p
    assert L.idx_score(ctypes.byref(p), vp(0x1000), 4096, None, vp(0x4000), 1 << 30, None) == idxlib.IDX_EINVAL
    assert L.idx_launch(ctypes.byref(p), 2048, vp(0x1000), vp(0x4000), 1 << 30, None) == idxlib.IDX_EINVAL
    good = _fake_problem(idxlib)
    assert L.idx_score(ctypes.byref(good), vp(0x1000), 100, None, vp(0x4000), 1 << 30, None) == idxlib.IDX_EINVAL  # ld < max_bound
    assert L.idx_launch(ctypes.byref(good), 0, vp(0x1000), vp(0x4000), 1 << 30, None) == idxlib.IDX_EINVAL
    assert L.idx_launch(ctypes.byref(good), 2048, vp(0x1000), vp(0x4000), 16, None) == idxlib.IDX_EINVAL  # small ws
    assert L.idx_topk(vp(0x1000), 10, vp(0x2000), 0, 10, 5, None, vp(0x3000), vp(0x4000), 1 << 30, None) == idxlib.IDX_EINVAL
    assert L.idx_topk(vp(0x1000), 10, vp(0x2000), 1, 10, 4096, None, vp(0x3000), vp(0x4000), 1 << 30, None) == idxlib.IDX_EINVAL
    assert L.idx_topk(None, 10, vp(0x2000), 1, 10, 5, None, vp(0x3000), vp(0x4000), 1 << 30, None) == idxlib.IDX_EINVAL
    assert L.idx_last_device_status(None, None) == idxlib.IDX_EINVAL


def test_debug_hooks_roundtrip(idxlib):
    prev = idxlib.debug_set(idxlib.IDX_DEBUG_WAIT_LIMIT_NS, 12345)
    assert idxlib.debug_set(idxlib.IDX_DEBUG_WAIT_LIMIT_NS, prev) == 12345
    assert idxlib.debug_set(idxlib.IDX_DEBUG_STALL_SCORE_MMA, 0) == 0


def test_top1_rejects_bad_arguments_without_a_gpu(idxlib):
    lib = idxlib.lib
    st = 0x10000
    assert lib.idx_top1_state_size(8) == 8 * 16 and lib.idx_top1_state_size(0) == 0
    # null logits, V < 1, ld < V, small state, misaligned state, bad token column
    assert lib.idx_top1(None, 10, 2, 10, 0x20000, None, None, 0, 0, None, st, 64, None) == idxlib.IDX_EINVAL
    assert lib.idx_top1(0x30000, 10, 2, 0, 0x20000, None, None, 0, 0, None, st, 64, None) == idxlib.IDX_EINVAL
    assert lib.idx_top1(0x30000, 5, 2, 10, 0x20000, None, None, 0, 0, None, st, 64, None) == idxlib.IDX_EINVAL
    assert lib.idx_top1(0x30000, 10, 2, 10, 0x20000, None, None, 0, 0, None, st, 16, None) == idxlib.IDX_EINVAL
    assert lib.idx_top1(0x30000, 10, 2, 10, 0x20000, None, None, 0, 0, None, st + 4, 64, None) == idxlib.IDX_EINVAL
    assert lib.idx_top1(0x30000, 10, 2, 10, 0x20000, None, 0x40000, 4, 4, None, st, 64, None) == idxlib.IDX_EINVAL
    assert lib.idx_top1(0x30000, 1 << 32, 2, 1 << 32, 0x20000, None, None, 0, 0, None, st, 64, None) \
        == idxlib.IDX_EUNSUPPORTED


def test_patch_rejects_bad_arguments_without_a_gpu(idxlib):
    import ctypes as C
    lib = idxlib.lib
    prob = _fake_problem(idxlib)
    assert lib.idx_patch_new_keys(C.byref(prob), None, None) == idxlib.IDX_EINVAL
    assert lib.idx_patch_new_keys(C.byref(prob), 0x80008, None) == idxlib.IDX_EINVAL    # not 16-byte aligned
    bad = _fake_problem(idxlib, R=0)
    assert lib.idx_patch_new_keys(C.byref(bad), 0x80000, None) == idxlib.IDX_EINVAL


def test_binding_refuses_to_import_without_the_library(tmp_path):
    """The binding has no fallback: a copy of the package with no built library
    raises ImportError on import, naming the missing file."""
    import shutil
    import subprocess
    import sys
    pkg = tmp_path / "sparse_attention_indexer_launch_gb300"
    pkg.mkdir()
    shutil.copy(os.path.join(ROOT, "sparse_attention_indexer_launch_gb300", "__init__.py"), pkg / "__init__.py")
    proc = subprocess.run([sys.executable, "-c", "import sparse_attention_indexer_launch_gb300"],
                          cwd=str(tmp_path), env={**os.environ, "PYTHONPATH": str(tmp_path)},
                          capture_output=True, text=True, timeout=120)
    assert proc.returncode != 0
    assert "ImportError" in proc.stderr and "libidx.so is not built" in proc.stderr
