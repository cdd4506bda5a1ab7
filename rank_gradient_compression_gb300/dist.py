"""Host-side multi-rank logic around the single-GPU step (torch.distributed).

Two ways to spread the step over ranks.

Block sharding: a resblock's skip decision, error buffers and Q depend only on its own
gradients, so N ranks (one per GPU) can shard the blocks and run the step with no data
exchange. The only collectives are host-side bookkeeping: the slowest rank's time, and
gathering the per-block counts for reporting.

Data parallel: every rank holds other workers' gradients of the SAME blocks. The step
then stops at its two exchange points (the worker sums of P and of Q) for an all-reduce
of the low-rank factors (``allreduce_step``), and all ranks must take the same skip
decision ("AIGC 基本功|混合精度与数值稳定性", §6.2): the integer counts are summed over
ranks before the comparison (``consensus_skip`` on the host; on the device the count
sum travels with P and the library compares it).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard_blocks(num_blocks: int, rank: int, world: int) -> list[int]:
    """Contiguous, balanced block ranges: rank k gets blocks [k*B/N, (k+1)*B/N)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    lo = rank * num_blocks // world
    hi = (rank + 1) * num_blocks // world
    return list(range(lo, hi))


def max_over_ranks(x: float, device=None) -> float:
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def gather_block_counts(local_counts: torch.Tensor, num_blocks: int, workers: int, rank_blocks) -> torch.Tensor:
    """Assemble the [num_blocks, workers] nonfinite counts of all ranks (int64, CPU).

    ``local_counts`` is this rank's [len(rank_blocks), workers] counts.
    """
    full = torch.zeros((num_blocks, workers), dtype=torch.int64, device=local_counts.device)
    full[list(rank_blocks)] = local_counts.to(torch.int64)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(full, op=dist.ReduceOp.SUM)
    return full.cpu()


def consensus_skip(local_counts: torch.Tensor, threshold: torch.Tensor) -> torch.Tensor:
    """Data-parallel skip rule: sum each block's nonfinite count over all ranks, then
    compare with the block's integer threshold. Every rank gets the same [B] result."""
    total = local_counts.to(torch.int64).clone()
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(total, op=dist.ReduceOp.SUM)
    return total >= threshold.to(torch.int64)


def total_workers(workers: int, group=None, device=None) -> int:
    """Sum of the simulated workers over the ranks of ``group`` (each rank may hold a
    different number)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return int(workers)
    t = torch.tensor([int(workers)], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return int(t.item())


def allreduce_step(engine, grads, errs, q, scales, ghat, w_total: int, group=None, scales_device=None):
    """One data-parallel PowerSGD step over the ranks of ``group``.

    ``engine`` is a ``psgd.PowerSGD`` made with PSGD_FLAG_EXCHANGE (or any object with
    the same step_p / step_q / step_e / exchange_* methods). The two factors are summed
    over the ranks between the three calls, one grouped all-reduce each, with the
    block counts travelling with P ("Zero-Shot Text-to-Image Generation - 中文验证版",
    §方法适配 and §证据: the low-rank factors are all-reduced, grouped; "AIGC 基本功|
    混合精度与数值稳定性", §6.2: every rank skips alike). ``w_total`` is
    ``total_workers(engine.W, group)``, computed once. The collectives run on the
    current stream's order, as the engine's kernels do.
    """
    multi = dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1
    engine.step_p(grads, errs, q, scales, ghat, scales_device=scales_device)
    counts = engine.exchange_counts()
    if multi:
        dist.all_reduce(engine.exchange_p(), op=dist.ReduceOp.SUM, group=group)
        dist.all_reduce(counts, op=dist.ReduceOp.SUM, group=group)
    engine.step_q(grads, errs, q, scales, ghat, counts, w_total, scales_device=scales_device)
    if multi:
        dist.all_reduce(engine.exchange_q(), op=dist.ReduceOp.SUM, group=group)
    engine.step_e(grads, errs, q, scales, ghat, w_total, scales_device=scales_device)
