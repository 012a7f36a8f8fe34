"""Small, self-contained invocations of each kernel for profiler captures.

    python -m linear_attention_recurrence_kda_gb300.profile_cases prefill-tc [--tokens T] [--heads H] [--reps R]
    python -m linear_attention_recurrence_kda_gb300.profile_cases decode [--seqs N] [--heads H] [--reps R]
    python -m linear_attention_recurrence_kda_gb300.profile_cases replay [--seqs N] [--heads H] [--window L] [--reps R]
    python -m linear_attention_recurrence_kda_gb300.profile_cases layer [--tokens T] [--heads H] [--reps R]
    python -m linear_attention_recurrence_kda_gb300.profile_cases prefill-simt [...]

Each case generates seeded inputs on the device (same recipe as the benchmark), runs one warm-up
call and then `reps` calls through the C ABI, and synchronises.  Sizes default to captures that
hold at most a few GB on the device and finish in seconds under a profiler.
"""
from __future__ import annotations

import argparse

import torch

from . import binding as B
from . import inputs as I


def _tokens(gen, shape, d, dtype, dev):
    q = torch.randn(*shape, d, generator=gen, device=dev)
    k = torch.randn(*shape, d, generator=gen, device=dev)
    v = torch.randn(*shape, d, generator=gen, device=dev)
    z = torch.randn(*shape, d, generator=gen, device=dev)
    n = lambda x: x / torch.sqrt((x * x).sum(-1, keepdim=True) + I.L2_EPS)
    return [t.to(dtype).contiguous() for t in (n(q), n(k), v, z)]


def prefill(tokens: int, heads: int, reps: int, dtype, d: int = 128, seqs: int = 1):
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(1)
    T = tokens * seqs
    q, k, v, z = _tokens(g, (T, heads), d, dtype, dev)
    A = (torch.randn(heads, generator=g, device=dev) * I.A_STD).float()
    beta = torch.sigmoid(torch.randn(T, heads, generator=g, device=dev)).float()
    s0 = (torch.randn(seqs, heads, d, d, generator=g, device=dev) * I.S0_STD).float()
    out = torch.empty(T, heads, d, dtype=dtype, device=dev)
    fin = torch.empty_like(s0)
    for _ in range(reps + 1):
        B.kda_forward(q, k, v, z, A, beta, initial_state=s0, out=out, final_state=fin)
    torch.cuda.synchronize()


def decode(seqs: int, heads: int, reps: int, d: int = 128):
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(4)
    q, k, v, z = _tokens(g, (seqs, heads), d, torch.bfloat16, dev)
    A = (torch.randn(heads, generator=g, device=dev) * I.A_STD).float()
    beta = torch.sigmoid(torch.randn(seqs, heads, generator=g, device=dev)).float()
    state = (torch.randn(seqs, heads, d, d, generator=g, device=dev) * 0.1).float()
    out = torch.empty(seqs, heads, d, dtype=torch.bfloat16, device=dev)
    for _ in range(reps + 1):
        B.kda_decode_step(q, k, v, z, A, beta, state, out=out)
    torch.cuda.synchronize()


def replay(seqs: int, heads: int, window: int, reps: int, d: int = 128):
    """Each rep: verify a window of drafted tokens from the snapshot (outputs only), then commit the
    accepted prefixes in place (state only)."""
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(5)
    q, k, v, z = _tokens(g, (seqs * window, heads), d, torch.bfloat16, dev)
    A = (torch.randn(heads, generator=g, device=dev) * I.A_STD).float()
    beta = torch.sigmoid(torch.randn(seqs * window, heads, generator=g, device=dev)).float()
    state = (torch.randn(seqs, heads, d, d, generator=g, device=dev) * 0.1).float()
    accepted = torch.randint(0, window + 1, (seqs,), generator=g, device=dev, dtype=torch.int32)
    out = torch.empty(seqs * window, heads, d, dtype=torch.bfloat16, device=dev)
    for _ in range(reps + 1):
        B.kda_decode_replay(q, k, v, z, A, beta, state, out=out, want_state=False)
        B.kda_decode_replay(q, k, v, z, A, beta, state, accepted=accepted, state_out=state, want_out=False)
    torch.cuda.synchronize()


def layer(tokens: int, heads: int, reps: int, d: int = 128, conv_width: int = 4):
    """Each rep: the prologue over the three projections, then the epilogue."""
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(6)
    x = [torch.randn(tokens, heads, d, generator=g, device=dev).to(torch.bfloat16) for _ in range(3)]
    w = [(torch.randn(heads, d, conv_width, generator=g, device=dev) * 0.5).float() for _ in range(3)]
    o = torch.randn(tokens, heads, d, generator=g, device=dev).to(torch.bfloat16)
    gate = torch.randn(tokens, heads, d, generator=g, device=dev).to(torch.bfloat16)
    wt = torch.randn(d, generator=g, device=dev).float()
    for _ in range(reps + 1):
        B.kda_prologue(*x, *w)
        B.kda_epilogue(o, gate, wt)
    torch.cuda.synchronize()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["prefill-tc", "prefill-simt", "decode", "replay", "layer"])
    ap.add_argument("--tokens", type=int, default=4096)
    ap.add_argument("--heads", type=int, default=16)
    ap.add_argument("--seqs", type=int, default=1)
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--window", type=int, default=7)
    a = ap.parse_args()
    if a.case == "prefill-tc":
        prefill(a.tokens, a.heads, a.reps, torch.bfloat16, seqs=a.seqs)
    elif a.case == "prefill-simt":
        prefill(a.tokens, a.heads, a.reps, torch.float32, seqs=a.seqs)
    elif a.case == "layer":
        layer(a.tokens, a.heads, a.reps)
    elif a.case == "replay":
        replay(a.seqs if a.seqs > 1 else 256, a.heads if a.heads != 16 else 32, a.window, a.reps)
    else:
        decode(a.seqs if a.seqs > 1 else 128, a.heads if a.heads != 16 else 32, a.reps)


if __name__ == "__main__":
    main()
