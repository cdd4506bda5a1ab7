"""Host-side multi-rank logic around the single-GPU step (torch.distributed).

Blocks are independent: a resblock's skip decision, error buffers and Q depend only on
its own gradients. So N ranks (one per GPU) shard the blocks and run the step with no
data exchange. The only collectives are host-side bookkeeping: the slowest rank's time,
and gathering the per-block counts for reporting.

``consensus_skip`` is the data-parallel form of the skip rule. There, every rank holds a
different worker's gradient of the SAME block, and all ranks must take the same
decision ("AIGC 基本功|混合精度与数值稳定性", §6.2). Summing the integer counts over ranks
before the comparison makes the decision identical everywhere.
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
