"""Seeded synthetic inputs for KDA prefill and decode.

This module only draws random tensors; it holds none of the recurrence's arithmetic, and it is
the one module that both the CUDA path's tests and the oracle's tests take inputs from.

Recipe (all draws from one CPU ``torch.Generator`` seeded per workload, in this order):
  lengths (varlen only), q, k, v, z  ~ N(0, 1)           [T, H, d]
  A^h                               ~ N(0, 0.5^2)        [H]         (0.5 read as the std)
  beta                              = sigmoid(N(0, 1))   [T, H]
  S0                                ~ N(0, 0.02^2)       [N, H, d, d] (absent: zero state)
q and k are then divided by sqrt(sum x^2 + 1e-6) over each (token, head) vector -- the
regularised L2 normalisation of the layer's input preparation ("Kimi K3: the paper and proofs
side by side", section 2.1.1, Equations 2-4) -- in fp32, before any cast.  q, k, v and z are then
rounded to the I/O dtype (round-to-nearest-even); A, beta and S0 stay fp32.

The five named workloads follow the shapes of the pages' long-context prefill and streaming
decode use (1M-token context; fixed-size per-head state).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

L2_EPS = 1e-6
A_STD = 0.5
S0_STD = 0.02


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    num_heads: int
    d: int
    io_dtype: torch.dtype
    lengths: Optional[tuple] = None          # fixed lengths; None -> drawn (varlen)
    varlen_range: Optional[tuple] = None     # (lo, hi) inclusive, number of sequences
    num_varlen: int = 0
    random_s0: bool = True
    decode_steps: int = 0                    # decode tokens per sequence after the prefill


WORKLOADS = {
    0: Workload("prefill B=1 H=2 T=64 d=32 fp32", 0, 2, 32, torch.float32, lengths=(64,), random_s0=False),
    1: Workload("prefill B=1 H=16 T=4096 d=128 bf16", 1, 16, 128, torch.bfloat16, lengths=(4096,)),
    2: Workload("varlen prefill 8 seqs U[1024,16384] H=32 d=128 bf16", 2, 32, 128, torch.bfloat16,
                varlen_range=(1024, 16384), num_varlen=8),
    3: Workload("prefill B=1 H=8 T=1048576 d=128 bf16", 3, 8, 128, torch.bfloat16, lengths=(1 << 20,)),
    4: Workload("decode 256 seqs H=32 d=128: 512-token prefill then 64 decode steps", 4, 32, 128,
                torch.bfloat16, lengths=(512,) * 256, decode_steps=64),
}


def _l2n(x: torch.Tensor) -> torch.Tensor:
    return x / torch.sqrt((x * x).sum(dim=-1, keepdim=True) + L2_EPS)


def draw_tokens(gen: torch.Generator, shape_k, shape_v, io_dtype):
    """q, k, v, z for token-major [..., H, d] shapes; q, k L2-normalised, cast to io_dtype."""
    q = torch.randn(*shape_k, generator=gen)
    k = torch.randn(*shape_k, generator=gen)
    v = torch.randn(*shape_v, generator=gen)
    z = torch.randn(*shape_k, generator=gen)
    q = _l2n(q)
    k = _l2n(k)
    return tuple(t.to(io_dtype).contiguous() for t in (q, k, v, z))


def make_inputs(wl: int | Workload, lengths=None, num_heads=None, d=None, io_dtype=None, seed=None,
                random_s0=None, d_k=None, d_v=None):
    """Inputs for a workload (or an override of its shape).  Returns a dict of CPU tensors:

    q, k, z [T, H, d_k]; v [T, H, d_v]; A [H] fp32; beta [T, H] fp32; S0 [N, H, d_k, d_v] fp32 or
    None; cu_seqlens [N+1] int32; lengths (list); and, for decode workloads, ``dec`` with per-step
    q, k, z [steps, N, H, d_k], v [steps, N, H, d_v] and beta [steps, N, H].
    ``d`` overrides both d_k and d_v; ``d_k`` / ``d_v`` override one.
    """
    w = WORKLOADS[wl] if isinstance(wl, int) else wl
    H = num_heads or w.num_heads
    dk = d_k or d or w.d
    dv = d_v or d or w.d
    dt = io_dtype or w.io_dtype
    sd = w.seed if seed is None else seed
    rs0 = w.random_s0 if random_s0 is None else random_s0
    gen = torch.Generator().manual_seed(sd)
    if lengths is None:
        if w.varlen_range is not None:
            lo, hi = w.varlen_range
            lengths = torch.randint(lo, hi + 1, (w.num_varlen,), generator=gen).tolist()
        else:
            lengths = list(w.lengths)
    lengths = [int(x) for x in lengths]
    N = len(lengths)
    T = sum(lengths)
    q, k, v, z = draw_tokens(gen, (T, H, dk), (T, H, dv), dt)
    A = (torch.randn(H, generator=gen) * A_STD).float()
    beta = torch.sigmoid(torch.randn(T, H, generator=gen)).float().contiguous()
    S0 = (torch.randn(N, H, dk, dv, generator=gen) * S0_STD).float().contiguous() if rs0 else None
    cu = torch.zeros(N + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    out = dict(q=q, k=k, v=v, z=z, A=A, beta=beta, S0=S0, cu_seqlens=cu, lengths=lengths,
               num_heads=H, d_k=dk, d_v=dv, io_dtype=dt)
    if w.decode_steps:
        s = w.decode_steps
        dq, dk_, dv_, dz = draw_tokens(gen, (s, N, H, dk), (s, N, H, dv), dt)
        db = torch.sigmoid(torch.randn(s, N, H, generator=gen)).float().contiguous()
        out["dec"] = dict(q=dq, k=dk_, v=dv_, z=dz, beta=db, steps=s)
    return out
