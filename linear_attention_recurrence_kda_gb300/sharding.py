"""Host-side logic of running the KDA path on several GPUs, one process per GPU.

Sequences and heads never interact in the recurrence (each (sequence, head) pair carries its own
state; "Kimi K3: the paper and proofs side by side", section 2.1.1, Equation 1), so the path shards
with no collective on the data path: every rank runs the kernels on its own sequences.  The only
cross-rank traffic is timing (the slowest rank's step time) and, for callers that want the whole
batch back on one rank, a gather of results.

This module is plain torch.distributed on whatever backend the caller initialised (NCCL on GPUs,
gloo in the CPU tests); it never launches a kernel.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import torch
import torch.distributed as dist


def split_sequences(lengths: Sequence[int], world: int) -> List[Tuple[int, int]]:
    """Contiguous ranges [lo, hi) of sequence indices, one per rank, balancing tokens.

    Rank r takes sequences lo_r .. hi_r - 1; the ranges cover every sequence exactly once, in order,
    and a rank may get none (hi == lo) when there are fewer sequences than ranks.  The boundary
    between ranks r - 1 and r is placed at the first sequence whose token prefix reaches r / world of
    the total, which keeps each rank's share within one sequence of the ideal.
    """
    if world < 1:
        raise ValueError("world must be >= 1")
    n = len(lengths)
    total = sum(int(x) for x in lengths)
    if any(int(x) < 0 for x in lengths):
        raise ValueError("sequence lengths must be >= 0")
    bounds = [0]
    prefix = 0
    i = 0
    for r in range(1, world):
        target = total * r / world
        while i < n and prefix + int(lengths[i]) / 2 <= target:
            prefix += int(lengths[i])
            i += 1
        bounds.append(max(i, bounds[-1]))
    bounds.append(n)
    return [(bounds[r], bounds[r + 1]) for r in range(world)]


def local_batch(cu_seqlens: Sequence[int], lo: int, hi: int) -> Tuple[int, int, List[int]]:
    """Token range [t_lo, t_hi) of sequences lo .. hi - 1 and their cu_seqlens rebased to zero."""
    cu = [int(x) for x in cu_seqlens]
    if not (0 <= lo <= hi <= len(cu) - 1):
        raise ValueError("sequence range out of bounds")
    t_lo, t_hi = cu[lo], cu[hi]
    return t_lo, t_hi, [c - t_lo for c in cu[lo:hi + 1]]


def max_over_ranks(x: float, device=None) -> float:
    """The largest x over all ranks (a step time: the job is as slow as its slowest rank)."""
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, device=None) -> float:
    """Sum of x over all ranks (units processed by the whole job)."""
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def gather_rows(local: torch.Tensor, dst: int = 0) -> torch.Tensor | None:
    """Concatenate every rank's tensor along dim 0 on rank ``dst`` (rows may differ per rank).

    Returns the concatenation on ``dst`` and None elsewhere.  Used to assemble a sharded batch's
    outputs (token-major) or final states (sequence-major) for checking.
    """
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return local
    world = dist.get_world_size()
    n = torch.tensor([local.shape[0]], dtype=torch.int64, device=local.device)
    sizes = [torch.zeros_like(n) for _ in range(world)]
    dist.all_gather(sizes, n)
    rows = [int(s.item()) for s in sizes]
    top = max(rows)
    pad = torch.zeros((top,) + tuple(local.shape[1:]), dtype=local.dtype, device=local.device)
    pad[: local.shape[0]] = local
    bufs = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(bufs, pad)
    if dist.get_rank() != dst:
        return None
    return torch.cat([b[:r] for b, r in zip(bufs, rows)], dim=0)
