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


# ------------------------------------------------------------------ exchange protocol
class _OracleEngine:
    """The three exchange calls of the library, written with the oracle's steps on the CPU
    (fp64), so that the data-parallel protocol of ``dist.allreduce_step`` can be checked
    on gloo ranks without a GPU. It holds this rank's workers of every block."""

    def __init__(self, shapes, B, W, r, frac, err_fmt):
        import numpy as np
        self.np, self.shapes, self.B, self.W, self.r = np, shapes, B, W, r
        self.frac, self.fmt = frac, err_fmt
        self.xp = torch.zeros(B * sum(m for m, _ in shapes) * r, dtype=torch.float64)
        self.xq = torch.zeros(B * sum(n for _, n in shapes) * r, dtype=torch.float64)
        self.xc = torch.zeros(B, dtype=torch.int64)

    def exchange_p(self):
        return self.xp

    def exchange_q(self):
        return self.xq

    def exchange_counts(self):
        return self.xc

    def _views(self, flat, rows):
        out, off = [], 0
        for b in range(self.B):
            row = []
            for j, sh in enumerate(self.shapes):
                k = sh[rows] * self.r
                row.append(flat[off:off + k].view(sh[rows], self.r))
                off += k
            out.append(row)
        return out

    def step_p(self, grads, errs, q, scales, ghat, scales_device=None):
        from oracle import powersgd as o
        self.ms = [[[None] * self.W for _ in self.shapes] for _ in range(self.B)]
        xp = self._views(self.xp, 0)
        for b in range(self.B):
            cnt = 0
            for j in range(len(self.shapes)):
                acc = 0.0
                for w in range(self.W):
                    g, mask = o.unscale_and_mask(grads[b][j][w], scales[b])
                    cnt += int(mask.sum())
                    self.ms[b][j][w] = o.accumulate_error(g, errs[b][j][w], self.fmt)
                    acc = acc + self.ms[b][j][w] @ q[b][j]
                xp[b][j][:] = torch.from_numpy(acc)
            self.xc[b] = cnt

    def step_q(self, grads, errs, q, scales, ghat, block_counts, total_workers, scales_device=None):
        from oracle import powersgd as o
        numel = sum(m * n for m, n in self.shapes)
        thr = o.skip_threshold(self.frac, total_workers, numel)
        self.skip = [int(block_counts[b]) >= thr for b in range(self.B)]
        xp, xq = self._views(self.xp, 0), self._views(self.xq, 1)
        self.p_hat = [[None] * len(self.shapes) for _ in range(self.B)]
        for b in range(self.B):
            if self.skip[b]:
                continue
            for j in range(len(self.shapes)):
                p_hat = o.orthonormalize(xp[b][j].numpy() / total_workers)
                self.p_hat[b][j] = p_hat
                xq[b][j][:] = torch.from_numpy(sum(m.T @ p_hat for m in self.ms[b][j]))

    def step_e(self, grads, errs, q, scales, ghat, total_workers, scales_device=None):
        from oracle import powersgd as o
        from oracle.numerics import round_to_format
        xq = self._views(self.xq, 1)
        for b in range(self.B):
            for j in range(len(self.shapes)):
                if self.skip[b]:
                    ghat[b][j][:] = 0.0
                    continue
                q[b][j][:] = round_to_format(xq[b][j].numpy() / total_workers, "f32")
                ghat[b][j][:] = self.p_hat[b][j] @ q[b][j].T
                for w in range(self.W):
                    errs[b][j][w][:] = o.error_update(self.ms[b][j][w], ghat[b][j], self.fmt)[0]


def _exchange_inputs(B, W_total, shapes, r, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    grads = [[[rng.normal(0, 2.0 ** -2, (m, n)) for _ in range(W_total)] for (m, n) in shapes]
             for _ in range(B)]
    errs = [[[np.zeros((m, n)) for _ in range(W_total)] for (m, n) in shapes] for _ in range(B)]
    q = [[rng.normal(0, 1, (n, r)) for (_, n) in shapes] for _ in range(B)]
    # block 1: 6 nonfinite entries on the last worker only (rank 1); the threshold over all
    # workers is 5, and rank 1 alone (half the entries) would see a threshold of 3
    grads[1][0][W_total - 1][0, :6] = np.inf
    # block 2: 2 nonfinite entries on worker 0 and 2 on the last worker: 4 < 5 in total
    grads[2][1][0][1, :2] = np.nan
    grads[2][1][W_total - 1][2, :2] = -np.inf
    return grads, errs, q


_EX_SHAPES, _EX_B, _EX_W, _EX_R = [(24, 16), (16, 32)], 3, 2, 3
_EX_FRAC = 5.0 / (2 * _EX_W * (24 * 16 + 16 * 32))  # threshold 5 over all 4 workers


def _exchange_worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        W = _EX_W
        grads, errs, q = _exchange_inputs(_EX_B, W * world, _EX_SHAPES, _EX_R, 7)
        mine = slice(rank * W, (rank + 1) * W)
        g = [[grads[b][j][mine] for j in range(len(_EX_SHAPES))] for b in range(_EX_B)]
        e = [[errs[b][j][mine] for j in range(len(_EX_SHAPES))] for b in range(_EX_B)]
        ghat = [[None for _ in _EX_SHAPES] for _ in range(_EX_B)]
        for b in range(_EX_B):
            for j, (m, n) in enumerate(_EX_SHAPES):
                ghat[b][j] = __import__("numpy").zeros((m, n))
        eng = _OracleEngine(_EX_SHAPES, _EX_B, W, _EX_R, _EX_FRAC, "f16")
        w_total = pd.total_workers(W)
        pd.allreduce_step(eng, g, e, q, [1.0] * _EX_B, ghat, w_total)
        out[rank] = (w_total, eng.skip, [[x.tolist() for x in row] for row in ghat],
                     [[x.tolist() for x in row] for row in q],
                     [[[x.tolist() for x in col] for col in row] for row in e])
    finally:
        dist.destroy_process_group()


def test_allreduce_step_matches_one_process_over_all_workers():
    """Two gloo ranks with two workers each run the exchange protocol; the result equals
    the oracle's block step over all four workers in one process (fp64, up to the order
    of the worker sums), and both ranks take the same skip decisions, including a block
    whose nonfinite entries sit on one rank only."""
    import numpy as np
    from oracle import powersgd as o
    world = 2
    port = _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_exchange_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 4
    assert res[0][1] == res[1][1] == [False, True, False]
    grads, errs, q = _exchange_inputs(_EX_B, _EX_W * world, _EX_SHAPES, _EX_R, 7)
    for b in range(_EX_B):
        st = o.BlockState(e=[list(errs[b][j]) for j in range(len(_EX_SHAPES))],
                          q=[q[b][j].copy() for j in range(len(_EX_SHAPES))])
        want = o.block_step(grads[b], st, 1.0, "f16", skip_fraction=_EX_FRAC)
        assert want.skip == res[0][1][b]
        for rank in range(world):
            for j in range(len(_EX_SHAPES)):
                gh = np.array(res[rank][2][b][j])
                assert np.linalg.norm(gh - want.g_hat[j]) <= 1e-12 * max(1.0, np.linalg.norm(want.g_hat[j]))
                assert np.allclose(np.array(res[rank][3][b][j]), st.q[j], rtol=1e-6, atol=1e-12)
                for w in range(_EX_W):
                    got_e = np.array(res[rank][4][b][j][w])
                    want_e = st.e[j][rank * _EX_W + w]
                    # E is f16-rounded on both sides: the fp64 sums differ in order only,
                    # so an entry may round the other way at most once in a long while
                    assert np.mean(got_e != want_e) < 1e-3


_UNEVEN = (1, 2, 3)  # workers held by each of three ranks


def _uneven_worker(rank, world, port, out):
    import numpy as np
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        W_all = sum(_UNEVEN)
        grads, errs, q = _exchange_inputs(_EX_B, W_all, _EX_SHAPES, _EX_R, 11)
        lo = sum(_UNEVEN[:rank])
        mine = slice(lo, lo + _UNEVEN[rank])
        g = [[grads[b][j][mine] for j in range(len(_EX_SHAPES))] for b in range(_EX_B)]
        e = [[errs[b][j][mine] for j in range(len(_EX_SHAPES))] for b in range(_EX_B)]
        ghat = [[np.zeros((m, n)) for (m, n) in _EX_SHAPES] for _ in range(_EX_B)]
        frac = 5.0 / (W_all * (24 * 16 + 16 * 32))  # threshold 5 over all six workers
        eng = _OracleEngine(_EX_SHAPES, _EX_B, _UNEVEN[rank], _EX_R, frac, "f16")
        w_total = pd.total_workers(_UNEVEN[rank])
        pd.allreduce_step(eng, g, e, q, [1.0] * _EX_B, ghat, w_total)
        out[rank] = (w_total, eng.skip, [[x.tolist() for x in row] for row in ghat])
    finally:
        dist.destroy_process_group()


def test_allreduce_step_with_uneven_workers_per_rank():
    """Three gloo ranks holding 1, 2 and 3 workers: the total worker count is summed, the
    factors divided by it, and every rank ends with the oracle's G-hat over all six workers
    and the same skip decisions (block 1's nonfinite entries sit on the last worker only)."""
    import numpy as np
    from oracle import powersgd as o
    world = len(_UNEVEN)
    port = _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_uneven_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    W_all = sum(_UNEVEN)
    assert all(res[k][0] == W_all for k in range(world))
    grads, errs, q = _exchange_inputs(_EX_B, W_all, _EX_SHAPES, _EX_R, 11)
    frac = 5.0 / (W_all * (24 * 16 + 16 * 32))
    for b in range(_EX_B):
        st = o.BlockState(e=[list(errs[b][j]) for j in range(len(_EX_SHAPES))],
                          q=[q[b][j].copy() for j in range(len(_EX_SHAPES))])
        want = o.block_step(grads[b], st, 1.0, "f16", skip_fraction=frac)
        for k in range(world):
            assert res[k][1][b] == want.skip
            for j in range(len(_EX_SHAPES)):
                gh = np.array(res[k][2][b][j])
                assert np.linalg.norm(gh - want.g_hat[j]) <= 1e-12 * max(1.0, np.linalg.norm(want.g_hat[j]))
    assert res[0][1] == [False, True, False]
