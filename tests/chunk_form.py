"""Chunk-form restatement of the KDA recurrence in fp64 -- test-only.

This is the derivation the GPU path uses, written out plainly so that its intermediates
(in-chunk cumulative log-decay, the strictly-lower Gram A, T = (I+A)^-1, the WY/UT-transformed
W and U~, the corrected U, and the per-chunk states) can be compared stage by stage.  It is
checked against the token-by-token oracle to ~1e-12 in ``test_chunk_form.py``; it shares no code
with the CUDA library.

Derivation (one sequence, one head, chunk of C tokens entering with state S0).
Write u_r = beta_r (v_r - (Diag(alpha_r) S_{r-1})^T k_r), so Equation 1 is
S_r = Diag(alpha_r) S_{r-1} + k_r u_r^T.  With G_r = sum_{s<=r} g_s (inclusive, per key channel)
and Gamma_r = exp(G_r):

    S_r = Diag(Gamma_r) S0 + sum_{i<=r} Diag(Gamma_r / Gamma_i) k_i u_i^T
    u_r + beta_r sum_{i<r} <k_r*Gamma_r, k_i/Gamma_i> u_i = beta_r (v_r - S0^T (k_r*Gamma_r))

so with A_{r,i} = beta_r <k_r*Gamma_r, k_i/Gamma_i> (i < r) and T = (I + A)^-1:

    U  = U~ - W S0,         U~ = T diag(beta) V,     W = T diag(beta) (K*Gamma)
    O  = (Q*Gamma) S0 + tril_incl((Q*Gamma)(K/Gamma)^T) U
    S_C = Diag(Gamma_C) S0 + (K * Gamma_C/Gamma)^T U

The chunk-wise form is an exact regrouping ("Kimi K3: architecture, derivations and a
pinned-source audit", section 4.5: compositions of the affine state maps are associative).
Pairwise decays exp(G_r - G_i) are formed directly here (no reciprocal rescaling).
"""
import numpy as np


def chunk_forward(q, k, v, g, beta, S0=None, cu_seqlens=None, C=16, keep=False):
    """q, k, g: [T,H,dk]; v: [T,H,dv]; beta: [T,H]; g = log-decay (<= 0).

    Returns (out [T,H,dv], S_final [N,H,dk,dv]) and, when ``keep``, a dict of intermediates
    keyed by (n, h, chunk index) with G, A, Tinv, W, Ut, U, S_in.
    """
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    T, H, dk = k.shape
    dv = v.shape[2]
    cu = np.array([0, T]) if cu_seqlens is None else np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    out = np.zeros((T, H, dv))
    Sf = np.zeros((N, H, dk, dv))
    inter = {}
    for n in range(N):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[n, h], dtype=np.float64)
            for ci, t0 in enumerate(range(cu[n], cu[n + 1], C)):
                t1 = min(t0 + C, cu[n + 1])
                Kc, Qc, Vc = k[t0:t1, h], q[t0:t1, h], v[t0:t1, h]
                b = beta[t0:t1, h]
                G = np.cumsum(g[t0:t1, h], axis=0)                  # [c, dk]
                D = np.exp(G[:, None, :] - G[None, :, :])            # D[r,i,:] = Gamma_r/Gamma_i
                KK = np.einsum("rc,ric,ic->ri", Kc, D, Kc)
                QK = np.einsum("rc,ric,ic->ri", Qc, D, Kc)
                c = t1 - t0
                A = np.tril(b[:, None] * KK, -1)
                Tinv = np.linalg.inv(np.eye(c) + A)
                W = Tinv @ (b[:, None] * (Kc * np.exp(G)))
                Ut = Tinv @ (b[:, None] * Vc)
                U = Ut - W @ S
                O = (Qc * np.exp(G)) @ S + np.tril(QK) @ U
                if keep:
                    inter[(n, h, ci)] = dict(G=G, A=A, Tinv=Tinv, W=W, Ut=Ut, U=U, S_in=S.copy())
                S = np.exp(G[-1])[:, None] * S + (Kc * np.exp(G[-1][None, :] - G)).T @ U
                out[t0:t1, h] = O
            Sf[n, h] = S
    if keep:
        return out, Sf, inter
    return out, Sf


def window_verify(q, k, v, g, beta, S0, dtype=np.float64):
    """Outputs of a window of L tokens read from the state S0 as ONE chunk, in the form the verify
    half of the speculative-decode replay uses: Gamma and 1/Gamma formed separately (reciprocal
    rescaling), [W0; Y0] = [K*Gamma; Q*Gamma] S0, A = beta (K*Gamma)(K/Gamma)^T strictly lower,
    P = (Q*Gamma)(K/Gamma)^T lower inclusive, U = (I + A)^-1 diag(beta) (V - W0), O = Y0 + P U.

    One sequence and head: q, k, g [L, dk]; v [L, dv]; beta [L]; S0 [dk, dv].  ``dtype`` sets the
    arithmetic (float32 mirrors the kernel's range: with L <= 8 and g >= -5, Gamma >= e^-40)."""
    q, k, v, g, beta, S0 = (np.asarray(x, dtype=dtype) for x in (q, k, v, g, beta, S0))
    L = k.shape[0]
    G = np.cumsum(g, axis=0, dtype=dtype)
    KG, QG, KI = k * np.exp(G), q * np.exp(G), k * np.exp(-G)
    A = np.tril(beta[:, None] * (KG @ KI.T), -1)
    P = np.tril(QG @ KI.T)
    Tp = np.linalg.inv(np.eye(L, dtype=dtype) + A) * beta[None, :]
    U = Tp @ (v - KG @ S0)
    return QG @ S0 + P @ U
