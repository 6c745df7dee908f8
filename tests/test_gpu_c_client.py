"""The C ABI from plain C: tests/c_client/idx_client.c, compiled here with gcc
against include/idx.h, libidx.so and the CUDA runtime only, runs
idx_launch_host on a problem read from raw files.  Its result must equal the
Python binding's idx_launch bit for bit and the oracle's selection on the GPU's
own scores, for an E4M3 and a bf16 cache; the client also checks that bad
arguments are refused before any launch."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import workloads
from tests import gpu_util

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    import sparse_attention_indexer_launch_gb300 as lib
    return lib


def _cuda_root():
    nvcc = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(nvcc)) if nvcc else "/usr/local/cuda"


@pytest.fixture(scope="module")
def client(lib, tmp_path_factory):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.fail("gcc not found")
    out = str(tmp_path_factory.mktemp("c_client") / "idx_client")
    libdir = os.path.dirname(lib.LIB_PATH)
    cuda = _cuda_root()
    cmd = [gcc, "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c_client", "idx_client.c"),
           "-L", libdir, "-lidx", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-o", out]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    assert proc.returncode == 0, proc.stderr
    return out


def _write_problem(prob, d, kv):
    d.mkdir(parents=True, exist_ok=True)
    rows_per_req = np.bincount(prob.row_req).max()
    with open(d / "meta.txt", "w") as f:
        f.write(f"{prob.R} {prob.page_table.shape[0]} {prob.P} {prob.page_table.shape[1]} {prob.max_bound} "
                f"{0 if kv == 'e4m3' else 1} {prob.K} {0 if rows_per_req > 2 else rows_per_req}\n")
    np.ascontiguousarray(prob.q).tofile(d / "q.bin")
    np.ascontiguousarray(prob.w).tofile(d / "w.bin")
    np.ascontiguousarray(prob.k_cache).tofile(d / "k_cache.bin")
    if kv == "e4m3":
        np.ascontiguousarray(prob.k_scale).tofile(d / "k_scale.bin")
    np.ascontiguousarray(prob.page_table).tofile(d / "page_table.bin")
    np.ascontiguousarray(prob.row_req).tofile(d / "row_req.bin")
    np.ascontiguousarray(prob.row_bound).tofile(d / "row_bound.bin")


CASES = [
    ("e4m3", [6000, 2500, 700], [4, 2, 1]),
    ("bf16", [4100, 1900], [2, 3]),
    ("e4m3", [9000], [1]),        # a lone row: the library picks the batched scan itself
]


@pytest.mark.parametrize("kv,lengths,rows", CASES, ids=["e4m3_mixed", "bf16_mixed", "e4m3_lone_row"])
def test_c_client_matches_the_binding_and_the_oracle(lib, orc, client, tmp_path, kv, lengths, rows):
    prob = workloads.build(f"c_{kv}", lengths, rows, kv, seed=sum(lengths) % 997)
    _write_problem(prob, tmp_path, kv)
    proc = subprocess.run([client, str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert proc.returncode == 0, proc.stdout + proc.stderr
    got = np.fromfile(tmp_path / "out.bin", dtype=np.int32).reshape(prob.R, prob.K)
    dp = lib.DeviceProblem(prob)
    assert np.array_equal(got, dp.launch().cpu().numpy()), "C client differs from the binding's idx_launch"
    scores, _ = dp.score()
    gpu_util.check_selection(orc, got, scores.cpu().numpy(), prob.row_bound, prob.K)
