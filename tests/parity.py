"""Parity helpers: run the CUDA path through the C ABI and the oracle on the same inputs, and
measure the error the way the tolerances are stated.

Tolerances (per tensor, outputs and final states separately):
  fp32 inputs : max|gpu - ref| / max|ref|  <= 1e-4
  bf16 inputs : max|gpu - ref| / RMS(ref)  <= 2e-2   (fp32 state and accumulation)

A bf16 *output* cannot be closer to the exact value than its own rounding: half a bf16 ulp of the
reference value (2^-9 relative) is not counted as error for tensors stored in bf16.  Without that
allowance the format alone fails the bound whenever max|o| / RMS(o) exceeds ~5 (a 33-token
sequence from a zero state has max/RMS = 9.5, and rounding the exact result to bf16 gives
3.5e-2).  fp32 tensors (the states, and outputs of the fp32 path) get no allowance.
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


def bf16_half_ulp(x):
    """Half the spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def err_rms_rel(gpu, ref, stored_bf16=False):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if not ref.size:
        return 0.0
    rms = np.sqrt(np.mean(ref * ref))
    d = np.abs(gpu - ref)
    if stored_bf16:
        d = np.maximum(d - bf16_half_ulp(ref), 0.0)
    return float(d.max() / max(rms, 1e-30))


def check(gpu, ref, io_dtype, what=""):
    """Assert the stated tolerance for the I/O dtype; returns the error.  ``gpu`` is a torch
    tensor (its storage dtype decides the bf16 rounding allowance) or an array of fp32 values."""
    stored_bf16 = torch.is_tensor(gpu) and gpu.dtype == torch.bfloat16
    if torch.is_tensor(gpu):
        gpu = gpu.detach().double().cpu().numpy()
    if io_dtype == torch.float32:
        e = err_max_rel(gpu, ref)
        assert e <= TOL_F32, f"{what}: max-rel error {e:.3e} > {TOL_F32}"
    else:
        e = err_rms_rel(gpu, ref, stored_bf16)
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
