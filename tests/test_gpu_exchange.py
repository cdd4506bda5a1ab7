"""The data-parallel exchange calls (psgd_step_p / psgd_step_q / psgd_step_e) on one GPU.

One rank: the three calls, with the exchange buffers passed through unchanged, give
psgd_step's result bit for bit (every engine: fp16 and bf16 on the tensor cores, fp32 on
the FFMA engine). Two ranks: two handles on the same GPU, each holding half of the
workers, with the buffers summed by torch between the calls in place of the all-reduce.
Nothing waits across handles: the calls run one after the other on one stream. Both
ranks then hold the same G-hat, Q and skip flags, and these match the fp64 oracle over
all workers. A block whose nonfinite entries sit on one rank only is skipped on both.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import GpuRun, TOL, f64, rel_err

pytestmark = pytest.mark.gpu


def _psgd():
    from rank_gradient_compression_gb300 import psgd
    return psgd


def _exchange_step(g: GpuRun, w_total=None):
    ps = g.ps
    w_total = ps.W if w_total is None else w_total
    ps.step_p(g.grads, g.errs, g.q, g.scales, g.ghat)
    ps.step_q(g.grads, g.errs, g.q, g.scales, g.ghat, ps.exchange_counts(), w_total)
    ps.step_e(g.grads, g.errs, g.q, g.scales, g.ghat, w_total)


@pytest.mark.parametrize("dtype,rank", [("f16", 16), ("f16", 112), ("bf16", 16), ("f32", 8)])
def test_one_rank_equals_the_whole_step_bit_for_bit(dtype, rank):
    psgd = _psgd()
    shapes = ((256, 192), (130, 136))
    if dtype == "f16":
        wl = synth.with_shapes(synth.stress(steps=3, workers=4, rank=rank, blocks=2, bad_step=1), shapes)
    else:
        wl = synth.with_shapes(synth.resblock_shard(steps=3, workers=4, rank=rank, dtype=dtype), shapes)
    a = GpuRun(wl)
    b = GpuRun(wl, flags=psgd.PSGD_FLAG_EXCHANGE)
    for t in range(wl.steps):
        a.load_inputs(t)
        b.load_inputs(t)
        a.step()
        _exchange_step(b)
        torch.cuda.synchronize()
        assert torch.equal(a.ps.counts, b.ps.counts)
        assert torch.equal(a.ps.skip, b.ps.skip)
        assert torch.equal(b.ps.exchange_counts(), a.ps.counts.view(wl.blocks, wl.workers).sum(1))
        for bb in range(wl.blocks):
            for j in range(len(shapes)):
                assert torch.equal(a.ghat[bb][j], b.ghat[bb][j]), (t, bb, j)
                assert torch.equal(a.q[bb][j], b.q[bb][j]), (t, bb, j)
                for w in range(wl.workers):
                    assert torch.equal(a.errs[bb][j][w], b.errs[bb][j][w]), (t, bb, j, w)
    if dtype == "f16":
        assert bool(a.ps.skip[1]) is False  # the bad step (1) was followed by a clean one


def _rank_engine(wl, workers, flags):
    from rank_gradient_compression_gb300.psgd import PowerSGD
    return PowerSGD(wl.shapes, wl.blocks, workers, wl.rank, wl.grad_dtype,
                    skip_fraction=wl.skip_fraction, flags=flags)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_two_ranks_match_the_oracle_over_all_workers(dtype):
    psgd = _psgd()
    shapes = ((384, 256), (200, 136))
    R, Wr = 2, 2
    wl = synth.with_shapes(synth.resblock_shard(steps=2, workers=R * Wr, rank=16, dtype=dtype,
                                                blocks=2), shapes, skip_fraction=0.5)
    dev = torch.device("cuda")
    tdt = synth.TORCH_DTYPE[dtype]
    ranks = [_rank_engine(wl, Wr, psgd.PSGD_FLAG_EXCHANGE) for _ in range(R)]
    B, J = wl.blocks, len(shapes)
    state = {b: oracle.BlockState(e=[[np.zeros(s) for _ in range(wl.workers)] for s in shapes],
                                  q=[synth.q0(wl, b, j).double().numpy() for j in range(J)])
             for b in range(B)}
    for t in range(wl.steps):
        # Every step starts both sides from the oracle's state (E, Q), as the single-rank
        # parity tests do. Block 1 at step 1 is nonfinite on every worker of rank 0 only:
        # with T = 1/2 of all workers' entries that skips it, where rank 1 alone would not.
        raw = [[[synth.grad(wl, t, b, j, w).double().numpy() for w in range(wl.workers)]
                for j in range(J)] for b in range(B)]
        if t == 1:
            for j in range(J):
                for w in range(Wr):
                    raw[1][j][w][:] = np.inf
        per_rank = []
        for k, ps in enumerate(ranks):
            mine = range(k * Wr, (k + 1) * Wr)
            grads = [[[torch.from_numpy(raw[b][j][w]).to(tdt).to(dev) for w in mine] for j in range(J)]
                     for b in range(B)]
            errs = [[[torch.from_numpy(state[b].e[j][w]).to(tdt).to(dev) for w in mine] for j in range(J)]
                    for b in range(B)]
            q = [[torch.from_numpy(state[b].q[j]).float().to(dev) for j in range(J)] for b in range(B)]
            ghat = [[torch.empty(s, dtype=torch.float32, device=dev) for s in shapes] for _ in range(B)]
            per_rank.append((grads, errs, q, ghat))
        scales = [wl.scale(b) for b in range(B)]
        w_total = R * Wr
        for ps, (g, e, q, gh) in zip(ranks, per_rank):
            ps.step_p(g, e, q, scales, gh)
        xp = sum(ps.exchange_p() for ps in ranks)
        xc = sum(ps.exchange_counts() for ps in ranks)
        for ps, (g, e, q, gh) in zip(ranks, per_rank):
            ps.exchange_p().copy_(xp)
            ps.exchange_counts().copy_(xc)
            ps.step_q(g, e, q, scales, gh, ps.exchange_counts(), w_total)
        xq = sum(ps.exchange_q() for ps in ranks)
        for ps, (g, e, q, gh) in zip(ranks, per_rank):
            ps.exchange_q().copy_(xq)
            ps.step_e(g, e, q, scales, gh, w_total)
        torch.cuda.synchronize()

        want = {b: oracle.block_step(raw[b], state[b], wl.scale(b), dtype, skip_fraction=wl.skip_fraction)
                for b in range(B)}
        assert [bool(x) for x in ranks[0].skip.cpu()] == [want[b].skip for b in range(B)]
        assert torch.equal(ranks[0].skip, ranks[1].skip)
        if t == 1:
            assert want[1].skip
        for b in range(B):
            for j in range(J):
                g0, g1 = per_rank[0][3][b][j], per_rank[1][3][b][j]
                assert torch.equal(g0, g1), "the ranks' G-hat differ"
                assert torch.equal(per_rank[0][2][b][j], per_rank[1][2][b][j]), "the ranks' Q differ"
                if want[b].skip:
                    assert torch.all(g0 == 0)
                    continue
                assert rel_err(f64(g0), want[b].g_hat[j]) <= TOL, (t, b, j)
                for k in range(R):
                    for i, w in enumerate(range(k * Wr, (k + 1) * Wr)):
                        m_gpu = f64(ranks[k].debug_m(b, j, i, tdt))
                        assert np.array_equal(m_gpu, want[b].m[j][w])
                        pre = m_gpu - f64(g0)
                        e_gpu = f64(per_rank[k][1][b][j][i])
                        assert np.array_equal(e_gpu, oracle.round_to_format(pre, dtype))
                        assert rel_err(pre, want[b].e_pre[j][w]) <= TOL, (t, b, j, w)
