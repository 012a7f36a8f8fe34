"""Parity helpers: run the CUDA path through the C ABI and the oracle on the same inputs, and
measure the error the way the tolerances are stated.

Tolerances (per tensor, outputs and final states separately):
  fp32 inputs : max|gpu - ref| / max|ref|  <= 1e-4
  bf16 inputs : max|gpu - ref| / RMS(ref)  <= 2e-2   (fp32 state and accumulation)
"""
import numpy as np
import torch

import oracle
from linear_attention_recurrence_kda_gb300 import binding as B

TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def err_max_rel(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max() if ref.size else 1.0
    return float(np.abs(gpu - ref).max() / max(den, 1e-30)) if ref.size else 0.0


def err_rms_rel(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if not ref.size:
        return 0.0
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.abs(gpu - ref).max() / max(rms, 1e-30))


def check(gpu, ref, io_dtype, what=""):
    """Assert the stated tolerance for the I/O dtype; returns the error."""
    if io_dtype == torch.float32:
        e = err_max_rel(gpu, ref)
        assert e <= TOL_F32, f"{what}: max-rel error {e:.3e} > {TOL_F32}"
    else:
        e = err_rms_rel(gpu, ref)
        assert e <= TOL_BF16, f"{what}: max/RMS error {e:.3e} > {TOL_BF16}"
    assert np.isfinite(np.asarray(gpu, dtype=np.float64)).all(), f"{what}: non-finite values"
    return e


def to_dev(inp, dev="cuda"):
    d = {}
    for key in ("q", "k", "v", "z", "A", "beta", "S0", "cu_seqlens"):
        t = inp.get(key)
        d[key] = None if t is None else t.to(dev)
    return d


def gpu_forward(inp, dev="cuda", use_cu=True, **kw):
    d = to_dev(inp, dev)
    cu = d["cu_seqlens"] if use_cu else None
    out, sf = B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"],
                            cu_seqlens=cu, max_seqlen=max(inp["lengths"]) if inp["lengths"] else 0, **kw)
    torch.cuda.synchronize()
    return out, sf


def oracle_forward(inp, heads=None, tokens=None, **kw):
    """Oracle on the same inputs; optionally restricted to some heads and a token prefix of a
    single sequence."""
    q, k, v, z, A, beta, S0 = (inp[x] for x in ("q", "k", "v", "z", "A", "beta", "S0"))
    cu = inp["cu_seqlens"]
    if heads is not None:
        hs = list(heads)
        q, k, v, z, beta = (t[:, hs] for t in (q, k, v, z, beta))
        A = A[hs]
        S0 = None if S0 is None else S0[:, hs]
    if tokens is not None:
        q, k, v, z, beta = (t[:tokens] for t in (q, k, v, z, beta))
        cu = torch.tensor([0, tokens], dtype=torch.int32)
    return oracle.forward(q, k, v, z, A, beta, S0=S0, cu_seqlens=cu, **kw)
