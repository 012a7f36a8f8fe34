"""The chunk-form restatement used for stage parity agrees with the token-by-token oracle."""
import numpy as np
import pytest

import oracle
from chunk_form import chunk_forward


@pytest.mark.parametrize("lens,C", [([64], 16), ([37], 16), ([5, 0, 33, 16, 1], 16), ([50], 8), ([29], 64)])
def test_chunk_form_matches_token_oracle(lens, C):
    rng = np.random.default_rng(sum(lens) + C)
    T, H, dk, dv = sum(lens), 2, 8, 6
    q = rng.normal(size=(T, H, dk))
    k = rng.normal(size=(T, H, dk))
    k /= np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
    v = rng.normal(size=(T, H, dv))
    z = rng.normal(size=(T, H, dk))
    A = rng.normal(size=H) * 0.5
    b = 1 / (1 + np.exp(-rng.normal(size=(T, H))))
    S0 = rng.normal(size=(len(lens), H, dk, dv)) * 0.02
    cu = np.concatenate([[0], np.cumsum(lens)])
    g, _ = oracle.gate(z, A)
    o_ref, s_ref = oracle.forward(q, k, v, z, A, b, S0=S0, cu_seqlens=cu)
    o, s = chunk_forward(q, k, v, g, b, S0=S0, cu_seqlens=cu, C=C)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12 * max(1.0, np.abs(o_ref).max()))
    np.testing.assert_allclose(s, s_ref, rtol=0, atol=1e-12 * max(1.0, np.abs(s_ref).max()))


def test_chunk_form_extreme_decay_stays_finite():
    """With every log-decay at the floor g_min=-5, a 16-token chunk spans exp(-80); the
    pairwise-decay form stays finite and matches the oracle."""
    rng = np.random.default_rng(7)
    T, H, dk, dv = 48, 1, 4, 3
    q, k, v = rng.normal(size=(T, H, dk)), rng.normal(size=(T, H, dk)), rng.normal(size=(T, H, dv))
    z = np.full((T, H, dk), 60.0)
    A = np.zeros(H)
    b = np.full((T, H), 0.5)
    g, _ = oracle.gate(z, A)
    assert np.all(g == -5.0)
    o_ref, s_ref = oracle.forward(q, k, v, z, A, b)
    o, s = chunk_forward(q, k, v, g, b)
    assert np.isfinite(o).all()
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(s, s_ref, atol=1e-12)


@pytest.mark.parametrize("L,floor", [(1, False), (5, False), (8, False), (8, True)])
def test_window_verify_form_matches_token_oracle(L, floor):
    """The one-chunk window form of the replay's verify (reciprocal rescaling) equals the token
    oracle in fp64, and stays within fp32 rounding of it in fp32 even with every decay at the
    floor (the window then spans e^-40)."""
    from chunk_form import window_verify
    rng = np.random.default_rng(100 + L + floor)
    H, dk, dv = 1, 16, 8
    q = rng.normal(size=(L, H, dk))
    k = rng.normal(size=(L, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.normal(size=(L, H, dv))
    z = np.full((L, H, dk), 60.0) if floor else rng.normal(size=(L, H, dk))
    A = np.zeros(H) if floor else rng.normal(size=H) * 0.5
    b = 1 / (1 + np.exp(-rng.normal(size=(L, H))))
    S0 = rng.normal(size=(1, H, dk, dv))
    g, _ = oracle.gate(z, A)
    o_ref, _ = oracle.forward(q, k, v, z, A, b, S0=S0)
    scale = max(1.0, np.abs(o_ref).max())
    o64 = window_verify(q[:, 0], k[:, 0], v[:, 0], g[:, 0], b[:, 0], S0[0, 0])
    np.testing.assert_allclose(o64, o_ref[:, 0], rtol=0, atol=1e-12 * scale)
    o32 = window_verify(q[:, 0], k[:, 0], v[:, 0], g[:, 0], b[:, 0], S0[0, 0], dtype=np.float32)
    assert np.isfinite(o32).all()
    np.testing.assert_allclose(o32, o_ref[:, 0], rtol=0, atol=2e-5 * scale)


@pytest.mark.parametrize("lens,C", [([40], 16), ([5, 0, 33, 17], 16), ([29], 8)])
def test_chunk_backward_matches_token_oracle(lens, C):
    """The chunk-wise backward (gradients reaching the log-decay through the scaled rows) equals
    the token-level reverse-mode oracle; the gate's chain rule links dg to dz and dA."""
    from chunk_form import chunk_backward
    rng = np.random.default_rng(300 + sum(lens) + C)
    T, H, dk, dv = sum(lens), 2, 6, 5
    q = rng.normal(size=(T, H, dk))
    k = rng.normal(size=(T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(T, H, dv))
    z = rng.normal(size=(T, H, dk))
    A = rng.normal(size=H) * 0.5
    b = rng.uniform(0.1, 0.9, size=(T, H))
    S0 = rng.normal(size=(len(lens), H, dk, dv)) * 0.3
    cu = np.concatenate([[0], np.cumsum(lens)])
    dO = rng.normal(size=(T, H, dv))
    dSf = rng.normal(size=(len(lens), H, dk, dv))
    g, _ = oracle.gate(z, A)
    ref = oracle.backward(q, k, v, z, A, b, dO, dSf, S0=S0, cu_seqlens=cu)
    dq, dk_, dv_, dg, db, dS0 = chunk_backward(q, k, v, g, b, dO, dSf, S0=S0, cu_seqlens=cu, C=C)
    tol = dict(rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(dq, ref[0], **tol)
    np.testing.assert_allclose(dk_, ref[1], **tol)
    np.testing.assert_allclose(dv_, ref[2], **tol)
    np.testing.assert_allclose(db, ref[5], **tol)
    np.testing.assert_allclose(dS0, ref[6], **tol)
    # dz = dg * g_min sigmoid'(x) e^A with x = e^A z; dA = sum dg * g_min sigmoid'(x) x
    x = np.exp(A)[None, :, None] * z
    s = 1 / (1 + np.exp(-x))
    dx = dg * -5.0 * s * (1 - s)
    np.testing.assert_allclose(dx * np.exp(A)[None, :, None], ref[3], **tol)
    np.testing.assert_allclose((dx * x).sum(axis=(0, 2)), ref[4], **tol)
