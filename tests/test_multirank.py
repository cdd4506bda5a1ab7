"""N > 1 host logic on CPU: two gloo ranks (no GPU).

Checks block sharding (every block exactly once), max-over-ranks timing, the count
gather, and that the data-parallel skip consensus is identical on every rank even when
only one rank saw nonfinite values.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

from rank_gradient_compression_gb300 import dist as pd


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, W = 7, 3
        mine = pd.shard_blocks(B, rank, world)
        t = pd.max_over_ranks(1.5 + rank)
        local = torch.tensor([[b * 10 + w for w in range(W)] for b in mine], dtype=torch.int64)
        full = pd.gather_block_counts(local, B, W, mine)
        # DP consensus: block 2 has 5 nonfinite entries on rank 0 only; threshold 5
        counts = torch.zeros(B, dtype=torch.int64)
        if rank == 0:
            counts[2] = 5
        counts[4] = 2  # 2 per rank -> 4 total, below 5
        skip = pd.consensus_skip(counts, torch.full((B,), 5, dtype=torch.int64))
        out[rank] = (mine, t, full.tolist(), skip.tolist())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    blocks = res[0][0] + res[1][0]
    assert sorted(blocks) == list(range(7)) and not set(res[0][0]) & set(res[1][0])
    assert res[0][1] == res[1][1] == 2.5
    want = [[b * 10 + w for w in range(3)] for b in range(7)]
    assert res[0][2] == res[1][2] == want
    assert res[0][3] == res[1][3]
    assert res[0][3][2] is True and res[0][3][4] is False


@pytest.mark.parametrize("B,N", [(1, 1), (64, 8), (5, 3), (2, 4)])
def test_shard_blocks_partition(B, N):
    parts = [pd.shard_blocks(B, k, N) for k in range(N)]
    flat = [b for p in parts for b in p]
    assert flat == list(range(B))
    sizes = [len(p) for p in parts]
    assert max(sizes) - min(sizes) <= 1
