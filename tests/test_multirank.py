"""The multi-rank host logic of bench.py, run as two gloo ranks on the CPU.

One rank per GPU scores its own batch of requests (the indexer shards by
request with no exchange); the timings are reduced by a maximum over ranks and
rank 0 alone prints.  No GPU is touched here."""
import json
import os
import socket
import sys

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        prob = bench.rank_problem(0, rank)
        # per-rank "timings": rank r reports (1 + r, 10 - r, 3 r)
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.0 * rank], "cpu")
        total = bench.total_key_rows(prob.key_rows, world)
        np.save(os.path.join(out_dir, f"q{rank}.npy"), prob.q)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"max": got, "total": total, "key_rows": prob.key_rows,
                       "shape": list(prob.q.shape), "bounds": prob.row_bound.tolist()}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_by_request_and_reduce_by_max(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    r = [json.load(open(tmp_path / f"r{i}.json")) for i in range(world)]
    # every rank sees the same maxima
    assert r[0]["max"] == r[1]["max"] == [2.0, 10.0, 3.0]
    # same shapes and bounds, independent values
    assert r[0]["shape"] == r[1]["shape"] and r[0]["bounds"] == r[1]["bounds"]
    q0, q1 = np.load(tmp_path / "q0.npy"), np.load(tmp_path / "q1.npy")
    assert not np.array_equal(q0, q1)
    # whole-job units are the per-rank units times the world size
    assert r[0]["total"] == r[1]["total"] == 2 * r[0]["key_rows"]


def test_rank_zero_alone_prints(capsys):
    import bench
    bench.emit({"metric": "m", "value": 1.0}, 0)
    bench.emit(None, 1)
    bench.emit({"metric": "m", "value": 2.0}, 1)
    lines = capsys.readouterr().out.strip().splitlines()
    assert len(lines) == 1 and json.loads(lines[0])["value"] == 1.0


def test_rank_zero_runs_the_named_workload():
    import bench
    import workloads
    a, b = bench.rank_problem(0, 0), workloads.make_config(0)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.k_cache, b.k_cache)
    assert np.array_equal(a.page_table, b.page_table)
