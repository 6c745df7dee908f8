"""The key-sharded indexer's exchange as two gloo ranks on the CPU.

Each rank takes its shard of a request's pages (shard.split), ranks the keys it
holds with the oracle (standing in for idx_launch_scored on its GPU), and the
ranks all-gather their (position, score) lists with shard.exchange.  The
owner's merge of the gathered lists (the oracle's merge, standing in for
idx_merge_topk) must equal the oracle's selection of the unsharded problem.
No GPU is touched here."""
import os
import socket
import sys

import numpy as np
import torch
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
    import oracle
    import workloads
    from sparse_attention_indexer_launch_gb300 import shard
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        orc = oracle.default()
        prob = workloads.build("dcp", [5000, 1300, 300], [3, 2, 1], "e4m3", seed=71, dup_frac=0.05)
        K = 512
        sp, off = shard.split(prob, world)[rank]
        s = orc.score(sp).astype(np.float32)
        idx = orc.topk(s, sp.row_bound, K)
        sc = np.full(idx.shape, -np.inf, np.float32)
        for r in range(idx.shape[0]):
            ok = idx[r] >= 0
            sc[r, ok] = s[r, idx[r, ok]]
        all_idx, all_sc = shard.exchange(torch.from_numpy(idx), torch.from_numpy(sc))
        if rank == 0:   # the owner merges
            offs = shard.offsets(int(prob.page_table.shape[1]), world)
            assert off == offs[rank]
            got = orc.merge_topk(all_idx.numpy(), all_sc.numpy(), np.array(offs, np.int32), K)
            want = orc.topk(orc.score(prob).astype(np.float32), prob.row_bound, K)
            np.save(os.path.join(out_dir, "got.npy"), got)
            np.save(os.path.join(out_dir, "want.npy"), want)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_shard_exchange_and_owner_merge(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got, want = np.load(tmp_path / "got.npy"), np.load(tmp_path / "want.npy")
    assert np.array_equal(got, want)
