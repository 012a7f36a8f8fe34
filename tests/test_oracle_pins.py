"""Pins for the fp64 oracle: values the pages print, closed forms, special cases, brute force
and invariants.  None of these re-types the oracle's loop; each would fail for a plausible
mistake in it (a dropped term, the erase and decay swapped, a wrong index, a transposed state,
reading before the update, a wrong gate sign or scale)."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _one(x):
    return np.asarray(x, dtype=np.float64)


def _run(q, k, v, alpha, beta, S0=None, cu=None, **kw):
    """Oracle with [T,H,*] inputs built from per-token lists (H=1 unless already 3-D)."""
    return oracle.recurrence(q, k, v, alpha, beta, S0=S0, cu_seqlens=cu, **kw)


# ---------------------------------------------------------------- values printed on the pages

def test_golden_scalar_delta_update():
    g = _golden("scalar_delta_update.json")
    for case in g["cases"]:
        out, Sf = _run(_one([[g["q"]]]), _one([[g["k"]]]), _one([[[g["v"]]]]), _one([[[g["alpha"]]]]),
                       _one([[case["beta"]]]), S0=_one([[[[g["S0"]]]]]))
        assert abs(Sf[0, 0, 0, 0] - case["S1"]) < 1e-12
        # the query reads the updated state
        assert abs(out[0, 0, 0] - case["S1"]) < 1e-12
        if "decayed" in case:
            assert abs(g["alpha"] * g["S0"] - case["decayed"]) < 1e-12
            assert abs(g["v"] - case["decayed"] - case["error"]) < 1e-12


def test_golden_scalar_token_order():
    g = _golden("scalar_token_order.json")
    finals = []
    for case in g["cases"]:
        T = len(case["values"])
        q = np.ones((T, 1, 1))
        k = np.ones((T, 1, 1))
        v = np.asarray(case["values"], dtype=np.float64).reshape(T, 1, 1)
        al = np.full((T, 1, 1), g["alpha"])
        b = np.full((T, 1), g["beta"])
        _, Sf = _run(q, k, v, al, b, S0=np.full((1, 1, 1, 1), g["S0"]))
        assert abs(Sf[0, 0, 0, 0] - case["S_T"]) < 1e-12
        finals.append(Sf[0, 0, 0, 0])
    # tokens cannot be permuted
    assert abs(finals[0] - finals[1]) > 1.0


def test_golden_lean_step_2x1():
    g = _golden("lean_step_2x1.json")
    out, Sf = _run(_one([[g["q"]]]), _one([[g["k"]]]), _one([[g["v"]]]), _one([[g["alpha"]]]),
                   _one([[g["beta"]]]), S0=_one([[g["S0"]]]))
    assert out[0, 0, 0] == g["out0"]


def test_golden_worked_2x2():
    g = _golden("worked_2x2.json")
    out, Sf = _run(_one([[g["q"]]]), _one([[g["k"]]]), _one([[g["v"]]]), _one([[g["alpha"]]]),
                   _one([[g["beta"]]]), S0=_one([[g["S0"]]]))
    np.testing.assert_allclose(Sf[0, 0], g["S1"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(out[0, 0], g["out"], rtol=0, atol=1e-12)
    # the intermediate quantities printed on the page are consistent with the final state
    decayed = np.asarray(g["alpha"])[:, None] * np.asarray(g["S0"])
    np.testing.assert_allclose(decayed, g["decayed"], atol=1e-12)
    np.testing.assert_allclose(np.asarray(g["k"]) @ decayed, g["old_value"], atol=1e-12)
    np.testing.assert_allclose(np.asarray(g["v"]) - np.asarray(g["old_value"]), g["correction"], atol=1e-12)


def test_golden_gate_slider():
    g = _golden("gate_slider.json")
    for A in (-3.0, -0.5, 0.0, 0.7, 2.0):
        gg, al = oracle.gate(np.full((1, 1, 1), g["z"]), np.array([A]), g_min=g["g_min"])
        assert gg[0, 0, 0] == g["g"]
        assert round(al[0, 0, 0], 4) == g["alpha_4dp"]
        assert abs(al[0, 0, 0] - math.exp(-2.5)) < 1e-15


# ---------------------------------------------------------------- the gate (Equation 5)

def test_gate_bounds_monotone_and_scale():
    z = np.linspace(-30, 30, 601).reshape(-1, 1, 1)
    for A in (-1.0, 0.0, 1.0):
        g, al = oracle.gate(z, np.array([A]))
        g = g.ravel()
        al = al.ravel()
        assert np.all(g <= 0.0) and np.all(g >= -5.0)
        assert np.all(al <= 1.0) and np.all(al >= math.exp(-5.0))
        # moving the logit right forgets faster (smaller retention); strictly so until the
        # sigmoid saturates in double precision
        assert np.all(np.diff(g) <= 0)
        inner = np.abs(z.ravel()[1:]) < 10
        assert np.all(np.diff(g)[inner] < 0)
        # strict interior for moderate logits, as in paper_retention_bounds
        mid = np.abs(z.ravel()) < 5
        assert np.all(al[mid] < 1.0) and np.all(al[mid] > math.exp(-5.0))
        # e^A scales the logit: g(z; A) = g(z e^A; 0)
        g0, _ = oracle.gate(z * math.exp(A), np.array([0.0]))
        np.testing.assert_allclose(g, g0.ravel(), rtol=1e-14, atol=1e-14)
    # the limits are g_min (z -> +inf) and 0 (z -> -inf); the midpoint is g_min / 2
    g, _ = oracle.gate(np.array([[[60.0]], [[-60.0]], [[0.0]]]), np.array([0.0]), g_min=-7.0)
    assert abs(g[0, 0, 0] + 7.0) < 1e-12 and abs(g[1, 0, 0]) < 1e-12 and g[2, 0, 0] == -3.5


def test_gate_tile_cumulative_log_decay_bound():
    rng = np.random.default_rng(1)
    z = rng.normal(size=(16 * 64, 2, 32)) * 4.0
    A = rng.normal(size=2)
    g, _ = oracle.gate(z, A)
    G = g.reshape(64, 16, 2, 32).sum(axis=1)
    assert np.all(G <= 0.0) and np.all(G >= -80.0)


def test_gate_driven_forward_equals_recurrence_with_gate_alpha():
    rng = np.random.default_rng(2)
    T, H, dk, dv = 21, 2, 5, 3
    q, k = rng.normal(size=(T, H, dk)), rng.normal(size=(T, H, dk))
    v, z = rng.normal(size=(T, H, dv)), rng.normal(size=(T, H, dk))
    A, b = rng.normal(size=H), rng.uniform(size=(T, H))
    S0 = rng.normal(size=(1, H, dk, dv))
    _, al = oracle.gate(z, A)
    o1, s1 = oracle.forward(q, k, v, z, A, b, S0=S0)
    o2, s2 = oracle.recurrence(q, k, v, al, b, S0=S0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(s1, s2)


# ---------------------------------------------------------------- closed forms / special cases

def _rand(rng, T, H, dk, dv, unit_keys=True):
    k = rng.normal(size=(T, H, dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q = rng.normal(size=(T, H, dk))
    v = rng.normal(size=(T, H, dv))
    al = rng.uniform(0.2, 0.99, size=(T, H, dk))
    b = rng.uniform(0.05, 0.95, size=(T, H))
    S0 = rng.normal(size=(1, H, dk, dv))
    return q, k, v, al, b, S0


def test_beta_zero_is_pure_decay():
    rng = np.random.default_rng(3)
    T, H, dk, dv = 13, 2, 6, 4
    q, k, v, al, _, S0 = _rand(rng, T, H, dk, dv)
    out, Sf = oracle.recurrence(q, k, v, al, np.zeros((T, H)), S0=S0)
    Gam = np.cumprod(al, axis=0)  # [T, H, dk]
    for t in range(T):
        for h in range(H):
            St = Gam[t, h][:, None] * S0[0, h]
            np.testing.assert_allclose(out[t, h], St.T @ q[t, h], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Sf[0], Gam[-1][:, :, None] * S0[0], rtol=1e-12, atol=1e-12)


def test_alpha_one_beta_one_orthonormal_keys_read_back_value():
    rng = np.random.default_rng(4)
    T, dk, dv = 7, 9, 5
    # distinct standard-basis keys from a zero state: bit-exact
    idx = rng.permutation(dk)[:T]
    k = np.zeros((T, 1, dk))
    k[np.arange(T), 0, idx] = 1.0
    v = rng.normal(size=(T, 1, dv))
    out, _ = oracle.recurrence(k, k, v, np.ones((T, 1, dk)), np.ones((T, 1)))
    np.testing.assert_array_equal(out, v)
    # general orthonormal keys (rows of a random orthogonal matrix) and a random state
    Qm, _ = np.linalg.qr(rng.normal(size=(dk, dk)))
    k = Qm[:T].reshape(T, 1, dk)
    S0 = rng.normal(size=(1, 1, dk, dv))
    out, _ = oracle.recurrence(k, k, v, np.ones((T, 1, dk)), np.ones((T, 1)), S0=S0)
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-12)


def test_alpha_one_beta_zero_constant_state():
    rng = np.random.default_rng(5)
    T, H, dk, dv = 9, 3, 4, 6
    q, k, v, _, _, S0 = _rand(rng, T, H, dk, dv)
    out, Sf = oracle.recurrence(q, k, v, np.ones((T, H, dk)), np.zeros((T, H)), S0=S0)
    np.testing.assert_array_equal(Sf, S0)
    np.testing.assert_allclose(out, np.einsum("thc,hcj->thj", q, S0[0]), rtol=1e-13, atol=1e-13)


def test_scalar_case_is_the_textbook_delta_rule():
    rng = np.random.default_rng(6)
    T = 40
    q, k, v = rng.normal(size=T), rng.normal(size=T), rng.normal(size=T)
    al, b = rng.uniform(0.1, 1.0, size=T), rng.uniform(size=T)
    s = 0.3
    ref_o = []
    for t in range(T):
        pred = k[t] * al[t] * s
        s = al[t] * s + b[t] * k[t] * (v[t] - pred)
        ref_o.append(q[t] * s)
    out, Sf = oracle.recurrence(q.reshape(T, 1, 1), k.reshape(T, 1, 1), v.reshape(T, 1, 1),
                                al.reshape(T, 1, 1), b.reshape(T, 1), S0=np.full((1, 1, 1, 1), 0.3))
    np.testing.assert_allclose(out.ravel(), ref_o, rtol=1e-13, atol=1e-13)
    assert abs(Sf.item() - s) < 1e-13


# ---------------------------------------------------------------- brute force (dense affine maps)

def _affine(k, v, a, b):
    dk = k.shape[0]
    M = (np.eye(dk) - b * np.outer(k, k)) @ np.diag(a)
    return M, b * np.outer(k, v)


def _compose(later, earlier):
    M2, U2 = later
    M1, U1 = earlier
    return M2 @ M1, M2 @ U1 + U2


@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_bruteforce_affine_maps(T):
    rng = np.random.default_rng(10 + T)
    H, dk, dv = 2, 4, 3
    q, k, v, al, b, S0 = _rand(rng, T, H, dk, dv, unit_keys=False)
    b = rng.uniform(0, 1.5, size=(T, H))  # the algebra holds for any beta
    out, Sf = oracle.recurrence(q, k, v, al, b, S0=S0)
    for h in range(H):
        agg = (np.eye(dk), np.zeros((dk, dv)))
        for t in range(T):
            agg = _compose(_affine(k[t, h], v[t, h], al[t, h], b[t, h]), agg)
            St = agg[0] @ S0[0, h] + agg[1]
            np.testing.assert_allclose(out[t, h], St.T @ q[t, h], rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(Sf[0, h], agg[0] @ S0[0, h] + agg[1], rtol=1e-11, atol=1e-11)
        # S_T = M_{T:1} S_0 + sum_i M_{T:i+1} U_i, summed explicitly
        acc = np.zeros((dk, dv))
        for i in range(T):
            Mi = np.eye(dk)
            for s in range(i + 1, T):
                Mi = _affine(k[s, h], v[s, h], al[s, h], b[s, h])[0] @ Mi
            acc += Mi @ _affine(k[i, h], v[i, h], al[i, h], b[i, h])[1]
        Mall = np.eye(dk)
        for s in range(T):
            Mall = _affine(k[s, h], v[s, h], al[s, h], b[s, h])[0] @ Mall
        np.testing.assert_allclose(Sf[0, h], Mall @ S0[0, h] + acc, rtol=1e-11, atol=1e-11)
    if T >= 3:
        maps = [_affine(k[t, 0], v[t, 0], al[t, 0], b[t, 0]) for t in range(3)]
        left = _compose(maps[2], _compose(maps[1], maps[0]))
        right = _compose(_compose(maps[2], maps[1]), maps[0])
        for x, y in zip(left, right):
            np.testing.assert_allclose(x, y, atol=1e-12)


def test_mutations_are_detected():
    """Plausible mistakes in an oracle (swapped erase/decay, reading before the update,
    a dropped erase, a transposed read) disagree with it on a single random token."""
    rng = np.random.default_rng(20)
    dk = dv = 4
    q, k, v, al, b, S0 = _rand(rng, 1, 1, dk, dv)
    out, Sf = oracle.recurrence(q, k, v, al, b, S0=S0)
    S, kk, vv, a, bb, qq = S0[0, 0], k[0, 0], v[0, 0], al[0, 0], b[0, 0], q[0, 0]
    wrong_order = np.diag(a) @ (np.eye(dk) - bb * np.outer(kk, kk)) @ S + bb * np.outer(kk, vv)
    no_erase = np.diag(a) @ S + bb * np.outer(kk, vv)
    assert np.max(np.abs(wrong_order - Sf[0, 0])) > 1e-3
    assert np.max(np.abs(no_erase - Sf[0, 0])) > 1e-3
    assert np.max(np.abs(S.T @ qq - out[0, 0])) > 1e-3  # read before the update
    # retention applied to value columns instead of key rows
    cols = S * a[None, :]
    transposed = cols + bb * np.outer(kk, vv - kk @ cols)
    assert np.max(np.abs(transposed - Sf[0, 0])) > 1e-3


# ---------------------------------------------------------------- invariants

def test_chunk_split_invariance():
    rng = np.random.default_rng(30)
    T, H, dk, dv = 37, 2, 5, 4
    q, k, v, al, b, S0 = _rand(rng, T, H, dk, dv)
    out, Sf = oracle.recurrence(q, k, v, al, b, S0=S0)
    for cut in (1, 16, 18, 36):
        o1, s1 = oracle.recurrence(q[:cut], k[:cut], v[:cut], al[:cut], b[:cut], S0=S0)
        o2, s2 = oracle.recurrence(q[cut:], k[cut:], v[cut:], al[cut:], b[cut:], S0=s1)
        np.testing.assert_array_equal(np.concatenate([o1, o2]), out)
        np.testing.assert_array_equal(s2, Sf)


def test_head_and_column_independence():
    rng = np.random.default_rng(31)
    T, H, dk, dv = 19, 3, 6, 5
    q, k, v, al, b, S0 = _rand(rng, T, H, dk, dv)
    out, Sf = oracle.recurrence(q, k, v, al, b, S0=S0)
    for h in range(H):
        o, s = oracle.recurrence(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], al[:, h:h + 1],
                                 b[:, h:h + 1], S0=S0[:, h:h + 1])
        np.testing.assert_array_equal(o[:, 0], out[:, h])
        np.testing.assert_array_equal(s[:, 0], Sf[:, h])
    for cb in (1, 2, 3):
        o, s = oracle.recurrence(q, k, v, al, b, S0=S0, col_block=cb)
        np.testing.assert_array_equal(o, out)
        np.testing.assert_array_equal(s, Sf)
    perm = rng.permutation(dv)
    o, s = oracle.recurrence(q, k, v[:, :, perm], al, b, S0=S0[..., perm])
    np.testing.assert_array_equal(o, out[:, :, perm])
    np.testing.assert_array_equal(s, Sf[..., perm])


def test_varlen_packing_equals_separate_runs_and_empty_sequence():
    rng = np.random.default_rng(32)
    lens = [5, 0, 17, 1, 16]
    T = sum(lens)
    H, dk, dv = 2, 4, 3
    q, k, v, al, b, _ = _rand(rng, T, H, dk, dv)
    S0 = rng.normal(size=(len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)])
    out, Sf = oracle.recurrence(q, k, v, al, b, S0=S0, cu_seqlens=cu)
    for n, L in enumerate(lens):
        sl = slice(cu[n], cu[n + 1])
        o, s = oracle.recurrence(q[sl], k[sl], v[sl], al[sl], b[sl], S0=S0[n:n + 1])
        np.testing.assert_array_equal(o, out[sl])
        np.testing.assert_array_equal(s[0], Sf[n])
        if L == 0:
            np.testing.assert_array_equal(Sf[n], S0[n])


def test_stability_bound():
    rng = np.random.default_rng(33)
    T, H, dk, dv = 200, 2, 8, 8
    q, k, v, al, b, S0 = _rand(rng, T, H, dk, dv)
    k *= rng.uniform(0.1, 1.0, size=(T, H, 1))  # ||k|| <= 1
    _, Sf = oracle.recurrence(q, k, v, np.ones_like(al), b, S0=S0)
    for h in range(H):
        bound = np.linalg.norm(S0[0, h]) + np.sum(b[:, h] * np.linalg.norm(k[:, h], axis=-1)
                                                   * np.linalg.norm(v[:, h], axis=-1))
        assert np.linalg.norm(Sf[0, h]) <= bound + 1e-9


def test_decode_step_is_one_token_of_the_recurrence():
    rng = np.random.default_rng(34)
    N, H, dk, dv, T = 3, 2, 6, 5, 9
    q, k, v, _, b, _ = _rand(rng, N * (T + 1), H, dk, dv)
    z = rng.normal(size=(N * (T + 1), H, dk))
    A = rng.normal(size=H) * 0.5
    S0 = rng.normal(size=(N, H, dk, dv))
    cu_full = np.arange(N + 1) * (T + 1)
    o_full, s_full = oracle.forward(q, k, v, z, A, b, S0=S0, cu_seqlens=cu_full)
    # prefill T tokens per sequence, then one decode step on the last token of each
    pre = np.concatenate([np.arange(n * (T + 1), n * (T + 1) + T) for n in range(N)])
    last = np.array([n * (T + 1) + T for n in range(N)])
    _, s_pre = oracle.forward(q[pre], k[pre], v[pre], z[pre], A, b[pre], S0=S0, cu_seqlens=np.arange(N + 1) * T)
    o_dec, s_dec = oracle.decode_step(q[last], k[last], v[last], z[last], A, b[last], s_pre)
    np.testing.assert_allclose(o_dec, o_full[last], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(s_dec, s_full, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- speculative-decode state replay

def _window(rng, N, L, H, dk, dv):
    q, k, v, _, b, _ = _rand(rng, N * L, H, dk, dv)
    z = rng.normal(size=(N * L, H, dk))
    A = rng.normal(size=H) * 0.5
    S = rng.normal(size=(N, H, dk, dv))
    return q, k, v, z, A, b, S


def test_replay_accepted_prefix_composes_and_leaves_the_snapshot():
    """The replay checks of the audit's CPU laboratory: a boundary after 3 tokens, 3 drafts of
    which 2 are accepted.  Replaying the 2 accepted drafts from the cached boundary state equals
    running all 5 tokens from the start; replaying all 3 drafts gives another state; the cached
    snapshot is unchanged by either replay."""
    rng = np.random.default_rng(41)
    H, dk, dv = 2, 5, 3
    q, k, v, z, A, b, S0 = _window(rng, 1, 6, H, dk, dv)
    _, s_boundary = oracle.forward(q[:3], k[:3], v[:3], z[:3], A, b[:3], S0=S0)
    snapshot = s_boundary.copy()
    d = slice(3, 6)
    _, s_all = oracle.replay(q[d], k[d], v[d], z[d], A, b[d], s_boundary)
    _, s_two = oracle.replay(q[d], k[d], v[d], z[d], A, b[d], s_boundary, accepted=[2])
    _, s_five = oracle.forward(q[:5], k[:5], v[:5], z[:5], A, b[:5], S0=S0)
    np.testing.assert_allclose(s_two, s_five, rtol=1e-12, atol=1e-12)
    assert not np.allclose(s_all, s_two)
    np.testing.assert_array_equal(s_boundary, snapshot)


def test_replay_matches_chained_decode_steps():
    """Brute force: each sequence advanced token by token with decode_step from the snapshot.
    Every drafted token's output matches the chain whatever was accepted, and the state matches
    the chain after exactly accepted[n] steps (0 and L included)."""
    rng = np.random.default_rng(42)
    N, L, H, dk, dv = 5, 4, 2, 6, 5
    q, k, v, z, A, b, S = _window(rng, N, L, H, dk, dv)
    accepted = np.array([0, 1, 2, 4, 3])
    out, s_acc = oracle.replay(q, k, v, z, A, b, S, accepted=accepted)
    cur = S.copy()
    states = [cur]
    for t in range(L):
        rows = np.arange(N) * L + t
        o_t, cur = oracle.decode_step(q[rows], k[rows], v[rows], z[rows], A, b[rows], cur)
        np.testing.assert_allclose(out[rows], o_t, rtol=1e-12, atol=1e-12)
        states.append(cur)
    for n in range(N):
        np.testing.assert_allclose(s_acc[n], states[accepted[n]][n], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(s_acc[0], S[0])  # nothing accepted: the snapshot itself


def test_replay_outputs_do_not_depend_on_acceptance():
    """The outputs verify the whole window from the snapshot; the accepted counts only choose
    which state is kept (computing outputs from the kept state would fail this)."""
    rng = np.random.default_rng(43)
    N, L, H, dk, dv = 3, 5, 1, 4, 4
    q, k, v, z, A, b, S = _window(rng, N, L, H, dk, dv)
    o_all, s_all = oracle.replay(q, k, v, z, A, b, S)
    o_some, s_some = oracle.replay(q, k, v, z, A, b, S, accepted=[1, 5, 0])
    np.testing.assert_array_equal(o_all, o_some)
    np.testing.assert_array_equal(s_all[1], s_some[1])
    _, s_fwd = oracle.forward(q, k, v, z, A, b, S0=S, cu_seqlens=np.arange(N + 1) * L)
    np.testing.assert_allclose(s_all, s_fwd, rtol=1e-13, atol=1e-13)
    with pytest.raises(ValueError):
        oracle.replay(q, k, v, z, A, b, S, accepted=[1, 6, 0])


# ---------------------------------------------------------------- layer prologue / epilogue

def test_prologue_regularised_l2_norm_facts():
    """What the pages state about the regularised L2 normalisation: a normalised vector is always
    shorter than one (approaching it for long inputs), and the zero vector maps to itself."""
    rng = np.random.default_rng(50)
    x = rng.normal(size=(20, 2, 8)) * np.logspace(-3, 2, 20)[:, None, None]
    w = np.zeros((2, 8, 1))
    w[..., 0] = 1.0
    y = oracle.prologue(x, w)
    n = np.linalg.norm(y, axis=-1)
    assert np.all(n < 1.0) and n.max() > 0.999  # large vectors approach one from below
    z = oracle.prologue(np.zeros((3, 1, 4)), w[:1, :4])
    np.testing.assert_array_equal(z, 0.0)


def test_prologue_swish_values_and_causal_shift():
    """Swish at printed points (0, +-1) through an identity tap; a one-token shift tap reads the
    previous token of the same sequence and zero at every sequence start."""
    x = np.array([0.0, 1.0, -1.0, 2.0, 3.0, -4.0]).reshape(6, 1, 1)
    ident = np.array([1.0, 0.0]).reshape(1, 1, 2)
    y = oracle.prologue(x, ident, normalise=False)[:, 0, 0]
    np.testing.assert_allclose(y[:3], [0.0, 0.7310585786300049, -0.2689414213699951], rtol=1e-14, atol=1e-15)
    shift = np.array([0.0, 1.0]).reshape(1, 1, 2)
    cu = np.array([0, 2, 2, 6])  # sequences of 2, 0 and 4 tokens
    ys = oracle.prologue(x, shift, cu_seqlens=cu, normalise=False)[:, 0, 0]
    swish = lambda a: a / (1 + np.exp(-a))
    np.testing.assert_allclose(ys, [0.0, swish(0.0), 0.0, swish(-1.0), swish(2.0), swish(3.0)], rtol=1e-14, atol=1e-15)


def test_prologue_taps_add_linearly_before_the_activation():
    """Two taps equal the sum of the one-tap convolutions before Swish (checked through the
    activation's inverse-free form: with normalise off, y = s * sigmoid(s) where s is the sum)."""
    rng = np.random.default_rng(51)
    x = rng.normal(size=(9, 1, 3))
    w = rng.normal(size=(1, 3, 3))
    y = oracle.prologue(x, w, normalise=False)
    s = w[None, :, :, 0] * x
    s[1:] += w[None, :, :, 1] * x[:-1]
    s[2:] += w[None, :, :, 2] * x[:-2]
    np.testing.assert_allclose(y, s / (1 + np.exp(-s)), rtol=1e-13, atol=1e-15)


def test_epilogue_closed_forms():
    """RMSNorm of a constant row is its sign (up to eps); a zero gate halves; the output does not
    depend on the scale of o (eps aside); the normalised row has unit RMS."""
    eps = 1e-6
    o = np.full((1, 1, 8), -3.0)
    y = oracle.epilogue(o, np.zeros((1, 1, 8)), np.ones(8), eps)
    np.testing.assert_allclose(y, -0.5 / np.sqrt(1 + eps / 9.0), rtol=1e-14)
    rng = np.random.default_rng(52)
    o = rng.normal(size=(5, 2, 16))
    g = rng.normal(size=(5, 2, 16))
    wt = rng.normal(size=16)
    np.testing.assert_allclose(oracle.epilogue(7.5 * o, g, wt, 0.0), oracle.epilogue(o, g, wt, 0.0), rtol=1e-13)
    y = oracle.epilogue(o, np.full_like(g, 40.0), np.ones(16), 0.0)
    np.testing.assert_allclose(np.sqrt((y * y).mean(-1)), 1.0, rtol=1e-12)


# ---------------------------------------------------------------- gradients (backward)

def _bw_case(rng, lens, H, dk, dv):
    T = sum(lens)
    q = rng.normal(size=(T, H, dk))
    k = rng.normal(size=(T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(T, H, dv))
    z = rng.normal(size=(T, H, dk))
    A = rng.normal(size=H) * 0.5
    b = rng.uniform(0.1, 0.9, size=(T, H))
    S0 = rng.normal(size=(len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)])
    dO = rng.normal(size=(T, H, dv))
    dSf = rng.normal(size=(len(lens), H, dk, dv))
    return q, k, v, z, A, b, S0, cu, dO, dSf


def test_backward_matches_central_differences():
    """Every gradient entry against a central difference of L = sum(dO * out) + sum(dS_f * S_f)
    through the forward oracle (two sequences of 3 and 2 tokens, two heads, d_k = 3, d_v = 2)."""
    rng = np.random.default_rng(60)
    q, k, v, z, A, b, S0, cu, dO, dSf = _bw_case(rng, [3, 2], 2, 3, 2)

    def loss(*args):
        o, sf = oracle.forward(*args[:6], S0=args[6], cu_seqlens=cu)
        return float((dO * o).sum() + (dSf * sf).sum())

    args = [q, k, v, z, A, b, S0]
    grads = oracle.backward(q, k, v, z, A, b, dO, dSf, S0=S0, cu_seqlens=cu)
    order = [0, 1, 2, 3, 4, 5, 6]  # q k v z A beta S0 <- dq dk dv dz dA dbeta dS0
    eps = 1e-6
    for ai, gi in zip(order, range(7)):
        base = args[ai]
        num = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[ai][idx] += eps
            minus[ai][idx] -= eps
            num[idx] = (loss(*plus) - loss(*minus)) / (2 * eps)
        np.testing.assert_allclose(grads[gi], num, rtol=1e-6, atol=1e-7)


def test_backward_one_step_sum_of_squares():
    """The gradient of sum(S_1^2) with respect to the old state after one token, in closed form:
    S_1 = (I - b k k^T) Diag(alpha) S_0 + b k v^T gives 2 Diag(alpha) (I - b k k^T) S_1."""
    rng = np.random.default_rng(61)
    q, k, v, z, A, b, S0, cu, _, _ = _bw_case(rng, [1], 1, 4, 3)
    _, S1 = oracle.forward(q, k, v, z, A, b, S0=S0)
    _, al = oracle.gate(z, A)
    kk = k[0, 0]
    P = np.eye(4) - b[0, 0] * np.outer(kk, kk)
    expect = 2 * np.diag(al[0, 0]) @ P @ S1[0, 0]
    grads = oracle.backward(q, k, v, z, A, b, np.zeros((1, 1, 3)), 2 * S1, S0=S0)
    np.testing.assert_allclose(grads[6][0, 0], expect, rtol=1e-12, atol=1e-13)


def test_backward_zero_upstream_gives_zero():
    rng = np.random.default_rng(62)
    q, k, v, z, A, b, S0, cu, dO, dSf = _bw_case(rng, [4, 0, 2], 2, 3, 3)
    grads = oracle.backward(q, k, v, z, A, b, np.zeros_like(dO), np.zeros_like(dSf), S0=S0, cu_seqlens=cu)
    for gr in grads:
        np.testing.assert_array_equal(gr, 0.0)


def test_sigmoid_slope_closed_form():
    """The gate's slope sigmoid(x) (1 - sigmoid(x)) equals 1 / (4 cosh^2(x / 2)) everywhere, including
    where the sigmoid saturates and 1 - sigmoid(x) cannot be formed in float64."""
    x = np.concatenate([np.linspace(-700.0, 700.0, 2801), [0.0, 1e-9, -36.9, 37.5, 45.0, -60.0]])
    np.testing.assert_allclose(oracle._sigmoid_slope(x), 0.25 / np.cosh(x / 2.0) ** 2, rtol=1e-13, atol=0)
    assert oracle._sigmoid_slope(np.array([45.0]))[0] > 0.0


def test_backward_dz_at_a_saturated_gate():
    """One token from a random state, L = sum(dS_f * S_1): with S_1 = (I - b k k^T) Diag(alpha) S_0 +
    b k v^T, dL/dalpha_c = sum_j [(I - b k k^T)^T dS_f]_{cj} S_0[c, j], and through Equation 5
    dz_c = dL/dalpha_c * alpha_c * g_min * e^{-x_c} / (1 + e^{-x_c})^2 * e^A with x = e^A z.  Here
    x reaches 45 (a gate at its floor), where a central difference cannot resolve the slope."""
    rng = np.random.default_rng(63)
    q, k, v, z, A, b, S0, cu, _, dSf = _bw_case(rng, [1], 1, 4, 3)
    z = np.array([[[30.0, 12.0, -25.0, 2.0]]])
    A = np.array([np.log(1.5)])
    _, al = oracle.gate(z, A)
    kk = k[0, 0]
    P = np.eye(4) - b[0, 0] * np.outer(kk, kk)
    dal = ((P.T @ dSf[0, 0]) * S0[0, 0]).sum(axis=1)
    x = 1.5 * z[0, 0]
    expect = dal * al[0, 0] * (-5.0) * np.exp(-np.abs(x)) / (1.0 + np.exp(-np.abs(x))) ** 2 * 1.5
    grads = oracle.backward(q, k, v, z, A, b, np.zeros((1, 1, 3)), dSf, S0=S0)
    np.testing.assert_allclose(grads[3][0, 0], expect, rtol=1e-10, atol=0)
    assert abs(grads[3][0, 0, 0]) > 0.0
