"""Context-parallel prefill (KCP): sequences split by tokens across ranks, one exchange per call.

"Kimi K3" reading notes, section 7 ("Scaling to 1M Tokens: NoPE and KDA Context Parallelism"): a
range of tokens acts on the recurrent state as an affine map S -> M S + S~, so every rank summarises
its own range, the fixed-size summaries are all-gathered once, and a prefix scan of the gathered maps
gives every rank the state its range starts from; each rank then runs its range from that state
("Kimi K3: architecture, derivations and a pinned-source audit", section 4.5: the maps compose
associatively, which is what makes the scan exact).

Layout: N sequences of equal length T, each split into ``world`` contiguous token ranges; rank r
holds range r of every sequence, packed like kda_forward's equal-length input ([N * T_r, H, d], the
tokens of sequence n at rows n * T_r ... (n + 1) * T_r - 1).  Every rank holds the same initial
state (or none).  The exchange is one all-gather of 4 d_k (d_k + d_v) bytes per sequence and head
from every rank (128 KiB at d_k = d_v = 128); remote summaries arrive in local memory and are read
from there.  Rank world - 1 ends with the sequences' final state.

The arithmetic runs in the library's kernels (``CudaKernels``: kda_forward_summary, kda_state_scan
and kda_forward through the C ABI); this module only moves tensors between ranks with
torch.distributed on whatever backend the caller initialised.
"""
from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist

from . import binding as B


class CudaKernels:
    """The three per-rank steps, on the GPU through the C ABI."""

    @staticmethod
    def summary(q, k, v, z, A, beta, num_seqs):
        return B.kda_forward_summary(q, k, v, z, A, beta, num_seqs=num_seqs)

    @staticmethod
    def scan(transitions, states_from_zero, initial_state, count):
        return B.kda_state_scan(transitions, states_from_zero, initial_state=initial_state, count=count)

    @staticmethod
    def forward(q, k, v, z, A, beta, initial_state, num_seqs):
        return B.kda_forward(q, k, v, z, A, beta, initial_state=initial_state)


def exchange_summaries(M: torch.Tensor, St: torch.Tensor, group=None):
    """All-gather every rank's (M, S~) as one fixed-size message; returns ([R, ...M], [R, ...S~])."""
    world = dist.get_world_size(group)
    flat = torch.cat([M.reshape(-1), St.reshape(-1)])
    parts = [torch.empty_like(flat) for _ in range(world)]
    dist.all_gather(parts, flat, group=group)
    nm = M.numel()
    Ms = torch.stack([p[:nm].view(M.shape) for p in parts])
    Ss = torch.stack([p[nm:].view(St.shape) for p in parts])
    return Ms, Ss


def kcp_forward(q, k, v, z, A, beta, initial_state: Optional[torch.Tensor] = None, num_seqs: int = 1, group=None,
                kernels=CudaKernels):
    """This rank's outputs of a sequence-sharded prefill and the state after its range (the
    sequences' final state on the last rank).  Shapes: q, k, z [N * T_r, H, d_k]; v [N * T_r, H, d_v];
    A [H]; beta [N * T_r, H]; initial_state [N, H, d_k, d_v] or None."""
    rank = dist.get_rank(group)
    M, St = kernels.summary(q, k, v, z, A, beta, num_seqs)
    Ms, Ss = exchange_summaries(M, St, group=group)
    S_in = kernels.scan(Ms, Ss, initial_state, rank)
    return kernels.forward(q, k, v, z, A, beta, S_in, num_seqs)
