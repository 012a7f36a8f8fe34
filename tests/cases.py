"""Seeded device-side prefill invocations shared by GPU tests (inputs drawn on the device with the
workloads' distributions, as the benchmark draws them)."""
import torch

from linear_attention_recurrence_kda_gb300 import binding as B
from linear_attention_recurrence_kda_gb300 import inputs as I


def device_tokens(gen, shape, d, dtype, dev):
    """q, k (regularised-L2-normalised), v, z ~ N(0, 1), in ``dtype``, shaped ``shape + (d,)``."""
    q = torch.randn(*shape, d, generator=gen, device=dev)
    k = torch.randn(*shape, d, generator=gen, device=dev)
    v = torch.randn(*shape, d, generator=gen, device=dev)
    z = torch.randn(*shape, d, generator=gen, device=dev)
    n = lambda x: x / torch.sqrt((x * x).sum(-1, keepdim=True) + I.L2_EPS)
    return [t.to(dtype).contiguous() for t in (n(q), n(k), v, z)]


def prefill(tokens: int, heads: int, reps: int, dtype, d: int = 128, seqs: int = 1):
    """``reps + 1`` kda_forward calls on ``seqs`` equal sequences of ``tokens`` tokens."""
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(1)
    T = tokens * seqs
    q, k, v, z = device_tokens(g, (T, heads), d, dtype, dev)
    A = (torch.randn(heads, generator=g, device=dev) * I.A_STD).float()
    beta = torch.sigmoid(torch.randn(T, heads, generator=g, device=dev)).float()
    s0 = (torch.randn(seqs, heads, d, d, generator=g, device=dev) * I.S0_STD).float()
    out = torch.empty(T, heads, d, dtype=dtype, device=dev)
    fin = torch.empty_like(s0)
    for _ in range(reps + 1):
        B.kda_forward(q, k, v, z, A, beta, initial_state=s0, out=out, final_state=fin)
    torch.cuda.synchronize()
