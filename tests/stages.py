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


# ---------------------------------------------------------------- split tensor-core plan (bf16, d = 128)
#
# Workspace of the bf16 d = 128 path: 256 bytes of check word, then the operand blocks
# [T_tot // 32 + N + 1 slots][H][53,760 B] (32-token step s of sequence n in slot cu[n] // 32 + n + s),
# then, for segmented plans, S_in and S~ as fp32 [N][H][max_seg][128][128] and the transitions M as
# [N][H][max_seg] x 64 KiB, each region starting on a 256-byte boundary.
#
# One block (one 32-token step of one head, tokens counted from the step's first token, decays
# referred to that token):
#   [W ; Q Gamma]  bf16 [64 rows][128 channels], 128-byte swizzle: element (r, k) at
#                  (k // 64) * 64 * 128 + (r // 8) * 1024 + (r % 8) * 128 + (((k % 64) // 8) ^ (r % 8)) * 16
#                  + (k % 8) * 2; rows 0..31 are W, rows 32..63 Q Gamma
#   [P ; K~^T]     bf16 hi at byte 16,384 and lo at 26,624, [160 rows][32 tokens] without swizzle:
#                  element (row, i) at (row // 8) * 512 + (i // 8) * 128 + (row % 8) * 16 + (i % 8) * 2;
#                  rows 0..31 are P (token r, token i), rows 32..159 K~^T (channel c, token i)
#   U~             fp32 [32][128] at byte 36,864
#   Gamma_C        fp32 [128] at byte 53,248
BLOCK_BYTES = 53760
BLK_WQ, BLK_PK, BLK_PK_LO, BLK_UT, BLK_GC = 0, 16384, 10240, 36864, 53248
D_TC = 128


def _bf16_bits_to_f64(u16):
    return (np.asarray(u16, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _sw128_index(rows):
    r = np.arange(rows)[:, None]
    k = np.arange(D_TC)[None, :]
    kk = k % 64
    return (k // 64) * rows * 128 + (r // 8) * 1024 + (r % 8) * 128 + (((kk // 8) ^ (r % 8)) * 16) + (kk % 8) * 2


def _pk_index(rows, cols=32):
    r = np.arange(rows)[:, None]
    i = np.arange(cols)[None, :]
    return (r // 8) * 512 + (i // 8) * 128 + (r % 8) * 16 + (i % 8) * 2


def decode_block(blk):
    """One operand block (numpy uint8 [53760]) -> dict of float64 arrays: W [32,128],
    QG [32,128], P [32,32] (hi + lo), KtT [128,32] (hi + lo), Ut [32,128], GC [128]."""
    blk = np.asarray(blk, dtype=np.uint8)
    u16 = lambda off, idx: blk[off + idx].astype(np.uint16) | (blk[off + idx + 1].astype(np.uint16) << 8)
    wq = _bf16_bits_to_f64(u16(BLK_WQ, _sw128_index(64)))
    pki = _pk_index(160)
    pk = _bf16_bits_to_f64(u16(BLK_PK, pki)) + _bf16_bits_to_f64(u16(BLK_PK + BLK_PK_LO, pki))
    ut = blk[BLK_UT:BLK_UT + 32 * D_TC * 4].view(np.float32).reshape(32, D_TC).astype(np.float64)
    gc = blk[BLK_GC:BLK_GC + D_TC * 4].view(np.float32).astype(np.float64)
    return dict(W=wq[:32], QG=wq[32:], P=pk[:32], KtT=pk[32:], Ut=ut, GC=gc)


def split_layout(T, N, H, max_seg=1):
    """Byte offsets (blocks, seg_in, seg_st, seg_mt, total) of the split plan's workspace."""
    blocks = 256
    bb = _up((T // 32 + N + 1) * H * BLOCK_BYTES)
    seg = N * H * max_seg * D_TC * D_TC * 4 if max_seg > 1 else 0
    seg_in = blocks + bb
    seg_st = _up(seg_in + seg)
    seg_mt = _up(seg_st + seg)
    return blocks, seg_in, seg_st, seg_mt, _up(seg_mt + seg)


def split_block(ws_np, cu, H, n, h, s):
    """The bytes of the block of step s of sequence n, head h, from a host copy of the workspace."""
    slot = int(cu[n]) // 32 + n + s
    off = 256 + (slot * H + h) * BLOCK_BYTES
    return ws_np[off:off + BLOCK_BYTES]


def pair_reference(q, k, v, g, beta, t0, t1, h):
    """The block's quantities for tokens [t0, t1) (at most 32) of head h in fp64: the 32-token chunk
    form with decays referred to token t0 (absent tokens as zero rows / columns)."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    c = t1 - t0
    Kc, Qc, Vc, b = k[t0:t1, h], q[t0:t1, h], v[t0:t1, h], beta[t0:t1, h]
    G = np.cumsum(g[t0:t1, h], axis=0)
    KG, QG, KI = Kc * np.exp(G), Qc * np.exp(G), Kc * np.exp(-G)
    D = np.exp(G[:, None, :] - G[None, :, :])
    KK = np.einsum("rc,ric,ic->ri", Kc, D, Kc)
    QK = np.einsum("rc,ric,ic->ri", Qc, D, Kc)
    A = np.tril(b[:, None] * KK, -1)
    Tinv = np.linalg.inv(np.eye(c) + A)
    ref = dict(W=np.zeros((32, D_TC)), QG=np.zeros((32, D_TC)), P=np.zeros((32, 32)), KtT=np.zeros((D_TC, 32)),
               Ut=np.zeros((32, D_TC)), GC=np.exp(G[-1]))
    ref["W"][:c] = Tinv @ (b[:, None] * KG)
    ref["Ut"][:c] = Tinv @ (b[:, None] * Vc)
    ref["QG"][:c] = QG
    ref["P"][:c, :c] = np.tril(QK)
    ref["KtT"][:, :c] = (Kc * np.exp(G[-1][None, :] - G)).T
    del KI
    return ref
