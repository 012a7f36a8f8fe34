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


def chunk_backward(q, k, v, g, beta, dO, dS_final, S0=None, cu_seqlens=None, C=16):
    """Reverse-mode gradients of ``chunk_forward`` taken chunk by chunk (fp64): the chunk-wise
    backward a tensor-core kernel would implement, restated plainly.  Returns
    (dq, dk, dv, dg, dbeta, dS0) for L = sum(dO * out) + sum(dS_final * S_final); ``g`` is the
    log-decay (the gate's own chain rule is left to the caller).

    Per chunk entering with state S (forward as in ``chunk_forward``, G inclusive cumsum of g,
    KG = K e^G, QG = Q e^G, KI = K e^-G, Kt = K e^(G_C - G), A = tril_strict(diag(b) KG KI^T),
    T = (I + A)^-1, W = T diag(b) KG, Ut = T diag(b) V, U = Ut - W S, P = tril(QG KI^T),
    O = QG S + P U, S' = e^G_C S + Kt^T U), going back from dO and dS':
        dS = e^G_C dS' + QG^T dO - W^T dU;   dU = Kt dS' + P^T dO
        dKt = U dS'^T;  dQG = dO S^T + tril(dP) KI;  dP = tril(dO U^T);  dW = -dU S^T
        dT = dU (diag(b) V)^T + dW (diag(b) KG)^T;  dA = -tril_strict(T^T dT T^T)
        dV = diag(b) T^T dU;  dKG = diag(b) T^T dW + diag(b) dA KI
        dKI = dA^T diag(b) KG + tril(dP)^T QG
        dbeta = rowsum(T^T dU * V) + rowsum(T^T dW * KG) + rowsum(dA * KG KI^T)
    and the gradients reach G through the scaled rows themselves (never through 1/Gamma^2):
        dG = dKG * KG + dQG * QG - dKI * KI - dKt * Kt,  dG_C += sum_t dKt * Kt + e^G_C rowsum(dS' * S)
    then dg = reversed cumulative sum of dG over the chunk."""
    q, k, v, g, beta, dO, dS_final = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta, dO, dS_final))
    T, H, dk = k.shape
    dv = v.shape[2]
    cu = np.array([0, T]) if cu_seqlens is None else np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    dq, dkk, dvv, dg = (np.zeros_like(x) for x in (q, k, v, g))
    dbeta = np.zeros_like(beta)
    dS0 = np.zeros((N, H, dk, dv))
    for n in range(N):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[n, h], dtype=np.float64)
            chunks = []
            for t0 in range(cu[n], cu[n + 1], C):  # forward, keeping each chunk's entering state
                t1 = min(t0 + C, cu[n + 1])
                Kc, Qc, Vc, b = k[t0:t1, h], q[t0:t1, h], v[t0:t1, h], beta[t0:t1, h]
                G = np.cumsum(g[t0:t1, h], axis=0)
                KG, QG, KI = Kc * np.exp(G), Qc * np.exp(G), Kc * np.exp(-G)
                Kt = Kc * np.exp(G[-1][None, :] - G)
                c = t1 - t0
                M = KG @ KI.T
                A = np.tril(b[:, None] * M, -1)
                Tn = np.linalg.inv(np.eye(c) + A)
                W = Tn @ (b[:, None] * KG)
                U = Tn @ (b[:, None] * Vc) - W @ S
                P = np.tril(QG @ KI.T)
                chunks.append((t0, t1, S, G, KG, QG, KI, Kt, M, Tn, W, U, P))
                S = np.exp(G[-1])[:, None] * S + Kt.T @ U
            dS = dS_final[n, h].copy()
            for (t0, t1, S, G, KG, QG, KI, Kt, M, Tn, W, U, P) in reversed(chunks):
                Vc, b, dOc = v[t0:t1, h], beta[t0:t1, h], dO[t0:t1, h]
                eGC = np.exp(G[-1])
                dSn = dS
                dKt = U @ dSn.T
                dU = Kt @ dSn + P.T @ dOc
                dP = np.tril(dOc @ U.T)
                dQG = dOc @ S.T + dP @ KI
                dW = -dU @ S.T
                dS = eGC[:, None] * dSn + QG.T @ dOc - W.T @ dU
                dTn = dU @ (b[:, None] * Vc).T + dW @ (b[:, None] * KG).T
                dA = -np.tril(Tn.T @ dTn @ Tn.T, -1)
                TdU, TdW = Tn.T @ dU, Tn.T @ dW
                dvv[t0:t1, h] = b[:, None] * TdU
                dKG = b[:, None] * TdW + b[:, None] * (dA @ KI)
                dKI = (b[:, None] * dA).T @ KG + dP.T @ QG
                dbeta[t0:t1, h] = (TdU * Vc).sum(1) + (TdW * KG).sum(1) + (dA * M).sum(1)
                dkk[t0:t1, h] = dKG * np.exp(G) + dKI * np.exp(-G) + dKt * np.exp(G[-1][None, :] - G)
                dq[t0:t1, h] = dQG * np.exp(G)
                dG = dKG * KG + dQG * QG - dKI * KI - dKt * Kt
                dG[-1] += (dKt * Kt).sum(0) + eGC * (dSn * S).sum(1)
                dg[t0:t1, h] = np.cumsum(dG[::-1], axis=0)[::-1]
            dS0[n, h] = dS
    return dq, dkk, dvv, dg, dbeta, dS0
