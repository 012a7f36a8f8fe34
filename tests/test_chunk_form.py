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
