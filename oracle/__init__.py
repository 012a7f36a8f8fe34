"""fp64 CPU oracle for the Kimi Delta Attention (KDA) recurrence -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import this package.  The product path (the CUDA library and its Python
binding) never calls it, and the two share no code.

The arithmetic lives in ``kda_oracle.c`` (plain C, double precision, OpenMP over independent
(sequence, head, value-column block) units).  This module only marshals arrays:

* every input is converted to a C-contiguous float64 array (bf16 and fp32 values are upcast
  exactly), and
* results come back as float64 numpy arrays.

What is computed (see the C file for the step-by-step statement):

* ``gate``        -- Equation 5 of "Kimi K3: the paper and proofs side by side" (section 2.1.1):
                     g = g_min * sigmoid(exp(A_h) z), alpha = exp(g).
* ``recurrence``  -- Equation 1 with alpha given directly, token by token:
                     S_t = (I - b k k^T) Diag(alpha) S_{t-1} + b k v^T, o_t = S_t^T q_t.
* ``forward``     -- Equation 1 driven by the Equation 5 gate (what ``kda_forward`` computes).
* ``decode_step`` -- one token per sequence (what ``kda_decode_step`` computes).
* ``replay``      -- speculative-decode state replay: a window of drafted tokens per sequence read
                     from a snapshot that is left untouched, with the state kept after the
                     accepted prefix only (what ``kda_decode_replay`` computes).
* ``prologue``    -- short convolution, Swish and (q, k) regularised L2 normalisation of the
                     projections (what ``kda_prologue`` computes), numpy in float64.
* ``epilogue``    -- head-wise RMSNorm and sigmoid output gate (what ``kda_epilogue`` computes).
* ``backward``    -- reverse-mode gradients of ``forward`` (numpy, float64; what ``kda_backward``
                     computes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``libkda_oracle.so`` beside it (gcc, OpenMP, no FMA contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-fopenmp", "-ffp-contract=off",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.kda_oracle_gate.restype = None
            lib.kda_oracle_gate.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _dp, _dp,
                                            ctypes.c_double, _dp, _dp]
            run_args = [ctypes.c_int32, _i64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                        _dp, _dp, _dp]
            lib.kda_oracle_recurrence.restype = ctypes.c_int
            lib.kda_oracle_recurrence.argtypes = run_args + [_dp, _dp, _dp, _dp, _dp,
                                                             ctypes.c_int32, ctypes.c_int32]
            lib.kda_oracle_forward.restype = ctypes.c_int
            lib.kda_oracle_forward.argtypes = run_args + [_dp, _dp, ctypes.c_double, _dp, _dp, _dp, _dp,
                                                          ctypes.c_int32, ctypes.c_int32]
            lib.kda_oracle_decode_step.restype = ctypes.c_int
            lib.kda_oracle_decode_step.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                   ctypes.c_int32, _dp, _dp, _dp, _dp, _dp,
                                                   ctypes.c_double, _dp, _dp, _dp, _dp, ctypes.c_int32]
            lib.kda_oracle_max_threads.restype = ctypes.c_int
            lib.kda_oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact upcast of a numpy array or a CPU/GPU torch tensor to C-contiguous float64."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        import torch
        x = x.detach().to(device="cpu", dtype=torch.float64).contiguous().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _cu(cu_seqlens, T: int) -> np.ndarray:
    if cu_seqlens is None:
        return np.array([0, T], dtype=np.int64)
    if hasattr(cu_seqlens, "detach"):
        cu_seqlens = cu_seqlens.detach().cpu().numpy()
    return np.ascontiguousarray(cu_seqlens, dtype=np.int64)


def max_threads() -> int:
    """OpenMP threads the oracle uses by default."""
    return int(_load().kda_oracle_max_threads())


def gate(z, A, g_min: float = -5.0):
    """Equation 5 over z [T, H, d_k] with A [H]; returns (g, alpha) as float64 arrays."""
    z = _f64(z)
    A = _f64(A)
    T, H, dk = z.shape
    g = np.empty_like(z)
    al = np.empty_like(z)
    _load().kda_oracle_gate(T, H, dk, _ptr(z), _ptr(A), float(g_min), _ptr(g), _ptr(al))
    return g, al


def _auto_col_block(col_block: int, units: int, dv: int, threads: int) -> int:
    """Value columns per parallel unit: all of them unless there are fewer (sequence, head) units
    than threads, in which case columns are split (they evolve independently)."""
    if col_block > 0:
        return col_block
    nt = threads if threads > 0 else max_threads()
    if units >= nt:
        return dv
    blocks = min(dv, -(-nt // max(units, 1)))
    return max(1, -(-dv // blocks))


def _check(rc: int):
    if rc == -1:
        raise ValueError("oracle: invalid arguments")
    if rc != 0:
        raise MemoryError("oracle: allocation failed")


def recurrence(q, k, v, alpha, beta, S0=None, cu_seqlens=None, col_block: int = 0, threads: int = 0,
               want_out: bool = True):
    """Equation 1 with retentions ``alpha`` [T, H, d_k] given directly.

    q, k: [T, H, d_k]; v: [T, H, d_v]; beta: [T, H]; S0: [N, H, d_k, d_v] or None (zeros);
    cu_seqlens: [N+1] offsets or None (one sequence).  Returns (out [T,H,d_v], S_final [N,H,d_k,d_v]).
    """
    q, k, v, alpha, beta, S0 = map(_f64, (q, k, v, alpha, beta, S0))
    T, H, dk = k.shape
    dv = v.shape[2]
    cu = _cu(cu_seqlens, T)
    N = cu.shape[0] - 1
    out = np.zeros((T, H, dv), dtype=np.float64) if want_out else None
    Sf = np.zeros((N, H, dk, dv), dtype=np.float64)
    col_block = _auto_col_block(col_block, N * H, dv, threads)
    rc = _load().kda_oracle_recurrence(N, cu.ctypes.data_as(_i64p), H, dk, dv, _ptr(q), _ptr(k),
                                       _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0), _ptr(out),
                                       _ptr(Sf), int(col_block), int(threads))
    _check(rc)
    return out, Sf


def forward(q, k, v, z, A, beta, S0=None, cu_seqlens=None, g_min: float = -5.0, col_block: int = 0,
            threads: int = 0, want_out: bool = True):
    """Equation 1 driven by the Equation 5 gate: the result ``kda_forward`` must reproduce.

    Shapes as in :func:`recurrence`, with z [T, H, d_k] and A [H] in place of alpha.
    """
    q, k, v, z, A, beta, S0 = map(_f64, (q, k, v, z, A, beta, S0))
    T, H, dk = k.shape
    dv = v.shape[2]
    cu = _cu(cu_seqlens, T)
    N = cu.shape[0] - 1
    out = np.zeros((T, H, dv), dtype=np.float64) if want_out else None
    Sf = np.zeros((N, H, dk, dv), dtype=np.float64)
    col_block = _auto_col_block(col_block, N * H, dv, threads)
    rc = _load().kda_oracle_forward(N, cu.ctypes.data_as(_i64p), H, dk, dv, _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(z), _ptr(A), float(g_min), _ptr(beta), _ptr(S0), _ptr(out),
                                    _ptr(Sf), int(col_block), int(threads))
    _check(rc)
    return out, Sf


def decode_step(q, k, v, z, A, beta, S, g_min: float = -5.0, threads: int = 0):
    """One token for each of N sequences: q, k, z [N, H, d_k]; v [N, H, d_v]; beta [N, H];
    S [N, H, d_k, d_v].  Returns (out [N, H, d_v], S_new)."""
    q, k, v, z, A, beta, S = map(_f64, (q, k, v, z, A, beta, S))
    N, H, dk = k.shape
    dv = v.shape[2]
    out = np.zeros((N, H, dv), dtype=np.float64)
    S_new = np.empty_like(S)
    rc = _load().kda_oracle_decode_step(N, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A),
                                        float(g_min), _ptr(beta), _ptr(S), _ptr(S_new), _ptr(out),
                                        int(threads))
    _check(rc)
    return out, S_new


def replay(q, k, v, z, A, beta, S, accepted=None, g_min: float = -5.0, threads: int = 0):
    """Speculative-decode state replay ("Kimi K3: architecture, derivations and a pinned-source
    audit", section 10.3 "KDA state replay for speculative decoding", and the replay checks of its
    "CPU laboratory"): a speculating server keeps, for each of L drafted tokens per sequence, only
    that token's inputs (far less memory than a copy of the state); the verifier reads every
    drafted token from the saved state, and once it is known how many drafts survive, the state
    is moved forward over those alone.  The saved state is never modified.

    q, k, z: [N*L, H, d_k] with token t of sequence n at row n*L + t; v: [N*L, H, d_v];
    beta: [N*L, H]; A: [H]; S: the snapshot [N, H, d_k, d_v]; accepted: N counts in [0, L], or
    None for all L.

    Returns (out, S_acc): out [N*L, H, d_v] holds o_t for every drafted token, read from the
    recurrence started at the snapshot and run over the whole window (Equation 1, o_t = S_t^T q_t);
    S_acc [N, H, d_k, d_v] is the state after the first accepted[n] tokens of sequence n (the
    snapshot itself where that count is 0).  Both come from :func:`forward`: the window as N
    sequences of L tokens, and the accepted prefixes gathered as N sequences of accepted[n] tokens.
    """
    q, k, v, z, A, beta, S = map(_f64, (q, k, v, z, A, beta, S))
    N = S.shape[0]
    T = k.shape[0]
    if N < 1 or T % N:
        raise ValueError("oracle.replay: the token count must be a multiple of the sequence count")
    L = T // N
    acc = np.full(N, L, dtype=np.int64) if accepted is None else np.asarray(accepted, dtype=np.int64).reshape(N)
    if (acc < 0).any() or (acc > L).any():
        raise ValueError("oracle.replay: accepted counts must lie in [0, L]")
    out, _ = forward(q, k, v, z, A, beta, S0=S, cu_seqlens=np.arange(N + 1, dtype=np.int64) * L, g_min=g_min,
                     threads=threads)
    rows = np.concatenate([n * L + np.arange(acc[n], dtype=np.int64) for n in range(N)])
    cu_acc = np.concatenate([[0], np.cumsum(acc)]).astype(np.int64)
    _, S_acc = forward(q[rows], k[rows], v[rows], z[rows], A, beta[rows], S0=S, cu_seqlens=cu_acc, g_min=g_min,
                       threads=threads, want_out=False)
    return out, S_acc


def _sigmoid(x):
    """Logistic function in the overflow-free form for both signs."""
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def _sigmoid_slope(x):
    """Slope of the logistic function, sigmoid(x) (1 - sigmoid(x)), as e^{-|x|} / (1 + e^{-|x|})^2: the
    same function, written so that no 1 - sigmoid(x) is formed (that difference cancels to zero in
    float64 once |x| passes about 37, where the gate saturates)."""
    e = np.exp(-np.abs(x))
    return e / ((1.0 + e) * (1.0 + e))


def _seq_index(T: int, cu) -> np.ndarray:
    """Sequence start of every token (tokens of empty sequences do not exist)."""
    cu = _cu(cu, T)
    start = np.zeros(T, dtype=np.int64)
    for n in range(len(cu) - 1):
        start[cu[n]:cu[n + 1]] = cu[n]
    return start


def prologue(x, w, cu_seqlens=None, normalise: bool = True, eps: float = 1e-6):
    """The per-head preparation of q, k (``normalise``) or v from their projections ("Kimi K3: the
    paper and proofs side by side", section 2.1.1, "Preparing the queries, keys, values, and decay";
    "Kimi K3: architecture, derivations and a pinned-source audit", section 4.3):

        y_t = sum_{i < K} w[h, c, i] x_{t-i}     causal depthwise short convolution, x = 0 before
                                                 the sequence start
        y_t = y_t * sigmoid(y_t)                 Swish
        y_t = y_t / sqrt(sum_c y_t^2 + eps)      regularised L2 normalisation (q and k only)

    x: [T, H, d]; w: [H, d, K] (w[..., 0] weighs the current token); cu_seqlens: [N+1] or None.
    Returns float64 [T, H, d]."""
    x = _f64(x)
    w = _f64(w)
    T, H, d = x.shape
    K = w.shape[2]
    start = _seq_index(T, cu_seqlens)
    y = np.zeros_like(x)
    for i in range(K):
        src = np.arange(T) - i
        ok = src >= start
        xs = np.where(ok[:, None, None], x[np.maximum(src, 0)], 0.0)
        y += xs * w[None, :, :, i]
    y = y * _sigmoid(y)
    if normalise:
        y = y / np.sqrt((y * y).sum(-1, keepdims=True) + eps)
    return y


def epilogue(o, gate, weight, eps: float):
    """Head-wise RMSNorm of the recurrence output followed by the sigmoid output gate ("Kimi K3:
    architecture, derivations and a pinned-source audit", section 4.3; the gate of Equation 6 in
    "Kimi K3: the paper and proofs side by side", section 2.1.1):

        y = o / sqrt(mean_c o^2 + eps) * weight * sigmoid(gate)

    o, gate: [T, H, d_v]; weight: [d_v] (shared by the heads).  Returns float64 [T, H, d_v]."""
    o = _f64(o)
    gate = _f64(gate)
    weight = _f64(weight)
    rms = np.sqrt((o * o).mean(-1, keepdims=True) + eps)
    return o / rms * weight * _sigmoid(gate)


def backward(q, k, v, z, A, beta, dO, dS_final, S0=None, cu_seqlens=None, g_min: float = -5.0):
    """Reverse-mode gradients of ``forward``: for the scalar
    L = sum(dO * out) + sum(dS_final * S_final), returns (dq, dk, dv, dz, dA, dbeta, dS0) with the
    shapes of q, k, v, z, A, beta and S0 (zeros when S0 is None).

    The chain rule is taken through each token's steps in reverse order ("Kimi K3: the paper and
    proofs side by side", section 2.1.1, Equation 1 with the gate of Equation 5), per sequence and
    head, with the states of the forward pass kept:
        x = e^{A_h} z,  g = g_min sigmoid(x),  alpha = e^g
        Sbar = Diag(alpha) S_{t-1},  r = Sbar^T k,  u = beta (v - r),  S_t = Sbar + k u^T,
        o_t = S_t^T q.
    Going back from dS (the gradient reaching S_t):
        dq = S_t dO_t;  dS += q dO_t^T;  dk = dS u;  du = dS^T k;  dv = beta du;
        dbeta = du . (v - r);  dr = -beta du;  dSbar = dS + k dr^T;  dk += Sbar dr;
        dalpha_c = sum_j dSbar[c, j] S_{t-1}[c, j];  dS_{t-1} = Diag(alpha) dSbar;
        dx = dalpha alpha g_min sigmoid'(x);  dz = dx e^{A_h};  dA_h += sum dx x
    (sigmoid'(x) = sigmoid(x) (1 - sigmoid(x)), evaluated without cancellation).
    Plain numpy in float64, for test sizes."""
    q, k, v, z, A, beta, dO, dS_final, S0 = map(_f64, (q, k, v, z, A, beta, dO, dS_final, S0))
    T, H, dk_ = k.shape
    dv_ = v.shape[2]
    cu = _cu(cu_seqlens, T)
    N = cu.shape[0] - 1
    grads = [np.zeros_like(a) for a in (q, k, v, z)]
    dq, dkk, dvv, dz = grads
    dA = np.zeros(H)
    dbeta = np.zeros_like(beta)
    dS0 = np.zeros((N, H, dk_, dv_))
    for n in range(N):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in range(H):
            eA = np.exp(A[h])
            S = np.zeros((dk_, dv_)) if S0 is None else S0[n, h].copy()
            saved = []
            for t in range(t0, t1):
                x = eA * z[t, h]
                sig = _sigmoid(x)
                al = np.exp(g_min * sig)
                Sbar = al[:, None] * S
                r = Sbar.T @ k[t, h]
                u = beta[t, h] * (v[t, h] - r)
                saved.append((S, Sbar, x, sig, al, r, u))
                S = Sbar + np.outer(k[t, h], u)
            dS = dS_final[n, h].copy()
            for t in range(t1 - 1, t0 - 1, -1):
                S_prev, Sbar, x, sig, al, r, u = saved[t - t0]
                S_t = Sbar + np.outer(k[t, h], u)
                dq[t, h] = S_t @ dO[t, h]
                dS = dS + np.outer(q[t, h], dO[t, h])
                dk_t = dS @ u
                du = dS.T @ k[t, h]
                dvv[t, h] = beta[t, h] * du
                dbeta[t, h] = du @ (v[t, h] - r)
                dr = -beta[t, h] * du
                dSbar = dS + np.outer(k[t, h], dr)
                dkk[t, h] = dk_t + Sbar @ dr
                dal = (dSbar * S_prev).sum(axis=1)
                dS = al[:, None] * dSbar
                dx = dal * al * g_min * _sigmoid_slope(x)
                dz[t, h] = dx * eA
                dA[h] += (dx * x).sum()
            dS0[n, h] = dS
    return dq, dkk, dvv, dz, dA, dbeta, dS0
