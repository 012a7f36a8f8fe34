"""Stage parity helpers: the fp32 path's per-chunk intermediates in the forward workspace, and the
same quantities from the fp64 chunk-form restatement.

Workspace layout of the fp32 path (``include/kda.h``: the check word, then per token-head fp32
scratch): 256 bytes of check word; G [T][H][d_k] (in-chunk inclusive cumulative log-decay);
W [T][H][d_k] = T diag(beta) (K * Gamma); U~ [T][H][d_v] = T diag(beta) V; each region starting on
a 256-byte boundary."""
import numpy as np

from chunk_form import chunk_forward


def _up(x, a=256):
    return (x + a - 1) // a * a


def fp32_stage_layout(T, H, dk, dv):
    th = T * H
    g_off = 256
    w_off = _up(g_off + th * dk * 4)
    ut_off = _up(w_off + th * dk * 4)
    total = _up(ut_off + th * dv * 4)
    return g_off, w_off, ut_off, total


def fp32_stage_views(ws, T, H, dk, dv):
    """(G, W, U~) as float64 numpy arrays from a uint8 workspace tensor (any device)."""
    import torch
    g_off, w_off, ut_off, _ = fp32_stage_layout(T, H, dk, dv)
    b = ws.detach().cpu()

    def region(off, d):
        return b[off:off + T * H * d * 4].view(torch.float32).reshape(T, H, d).double().numpy()

    return region(g_off, dk), region(w_off, dk), region(ut_off, dv)


def chunk_reference_stages(q, k, v, g, beta, S0, cu, C=16):
    """Per-token (G, W, U~) of the chunk form, chunks restarting at every sequence start."""
    T, H, dk = np.asarray(k).shape
    dv = np.asarray(v).shape[2]
    G = np.zeros((T, H, dk))
    W = np.zeros((T, H, dk))
    Ut = np.zeros((T, H, dv))
    _, _, inter = chunk_forward(q, k, v, g, beta, S0=S0, cu_seqlens=cu, C=C, keep=True)
    cu = np.asarray(cu, dtype=np.int64)
    for (n, h, ci), st in inter.items():
        t0 = int(cu[n]) + C * ci
        rows = slice(t0, t0 + st["G"].shape[0])
        G[rows, h] = st["G"]
        W[rows, h] = st["W"]
        Ut[rows, h] = st["Ut"]
    return G, W, Ut
