"""GPU parity of kda_backward (the gradients of kda_forward) against the fp64 oracle's reverse-mode
gradients (``oracle.backward``, itself pinned by central differences), element by element on the
same seeded inputs.

Tolerances: the tensors stored in the io dtype (dq, dk, dv, dz) and the fp32 ones (dbeta, dS0) use
the forward path's per-tensor metrics (fp32: max-rel 1e-4; bf16: max / RMS 2e-2 with half a bf16
ulp excused for bf16-stored tensors).  dA is a sum over every token and key channel of a head
(dA_h = sum dz * z), whose value can be much smaller than its terms, so its error is measured
against the size of those terms: |dA - dA_ref| <= tol * sum |dz_ref * z| per head, tol = 1e-4 for
fp32 inputs and 1e-3 for bf16 inputs (fp32 accumulation either way)."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrence_kda_gb300 import binding as B
from linear_attention_recurrence_kda_gb300 import inputs as I
from parity import check, to_dev

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dz", "dA", "dbeta", "dS0")


def _cotangents(inp, seed, with_dsf=True):
    g = torch.Generator().manual_seed(seed)
    T, H, _ = inp["k"].shape
    dv = inp["v"].shape[2]
    N = len(inp["lengths"])
    d_out = torch.randn(T, H, dv, generator=g).to(inp["k"].dtype)
    dsf = (torch.randn(N, H, inp["k"].shape[2], dv, generator=g) * 0.1).float() if with_dsf else None
    return d_out, dsf


def _run(inp, d_out, dsf, **kw):
    d = to_dev(inp)
    ml = max(inp["lengths"]) if inp["lengths"] else 0
    return B.kda_backward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d_out.cuda(),
                          None if dsf is None else dsf.cuda(), initial_state=d["S0"], cu_seqlens=d["cu_seqlens"],
                          max_seqlen=ml, **kw)


def _oracle(inp, d_out, dsf, heads=None, **kw):
    q, k, v, z, A, beta, S0 = (inp[x] for x in ("q", "k", "v", "z", "A", "beta", "S0"))
    N = len(inp["lengths"])
    if dsf is None:
        dsf = torch.zeros(N, k.shape[1], k.shape[2], v.shape[2])
    if heads is not None:
        q, k, v, z, beta, d_out = (t[:, heads] for t in (q, k, v, z, beta, d_out))
        A = A[heads]
        S0 = None if S0 is None else S0[:, heads]
        dsf = dsf[:, heads]
    return oracle.backward(q, k, v, z, A, beta, d_out, dsf, S0=S0, cu_seqlens=inp["cu_seqlens"], **kw)


def _check_all(got, ref, inp, io, what=""):
    errs = {}
    for name, g, r in zip(NAMES, got, ref):
        if g is None or name == "dA":
            continue
        errs[name] = check(g, r, io, f"{what} {name}")
    z = inp["z"].double().numpy()
    dA = got[4].double().cpu().numpy()
    scale = np.abs(ref[3] * z).sum(axis=(0, 2))
    tol = 1e-4 if io == torch.float32 else 1e-3
    err = np.abs(dA - ref[4])
    assert np.all(err <= tol * scale + 1e-30), f"{what} dA: {err} vs scale {scale}"
    errs["dA"] = float((err / np.maximum(scale, 1e-30)).max())
    return errs


SMALL = [
    ([5, 0, 40, 16, 1], 32, 32), ([33], 128, 128), ([17, 64], 64, 128), ([100, 3, 77], 128, 64),
    ([16], 32, 64), ([250], 128, 128), ([0], 32, 32),
]


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("lengths,dk,dv", SMALL)
@pytest.mark.parametrize("with_s0", [False, True], ids=["s0zero", "s0rand"])
def test_backward_small(io, lengths, dk, dv, with_s0):
    inp = I.make_inputs(1, lengths=lengths, num_heads=3, d_k=dk, d_v=dv, io_dtype=io,
                        seed=sum(lengths) + dk + 3 * dv, random_s0=with_s0)
    d_out, dsf = _cotangents(inp, seed=sum(lengths) + 1)
    got = _run(inp, d_out, dsf)
    torch.cuda.synchronize()
    ref = _oracle(inp, d_out, dsf)
    errs = _check_all(got, ref, inp, io, what=f"{lengths} d_k={dk} d_v={dv}")
    print({k: f"{v:.1e}" for k, v in errs.items()})


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("d", [32, 128])
def test_backward_decay_floor(io, d):
    """Every log-decay at g_min: a 16-token chunk spans e^-80, so K / Gamma reaches e^80 inside the
    chunk products (the sigmoid's slope, and with it dz, is ~0 there; dq, dk, dv, dbeta, dS0 are not)."""
    inp = I.make_inputs(1, lengths=[48, 17, 0, 33], num_heads=2, d=d, io_dtype=io, seed=61 + d)
    inp["z"] = torch.full_like(inp["z"], 60.0)
    d_out, dsf = _cotangents(inp, seed=62)
    got = _run(inp, d_out, dsf)
    torch.cuda.synchronize()
    _check_all(got, _oracle(inp, d_out, dsf), inp, io, what="decay floor")


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_backward_half_floor_and_no_final_gradient(io):
    """No decay on half the key channels, the floor on the other half; no gradient on the final
    state (d_final_state NULL) and no initial state."""
    inp = I.make_inputs(1, lengths=[70, 9], num_heads=2, d=64, io_dtype=io, seed=63, random_s0=False)
    z = inp["z"].float()
    z[..., :32] = -1e4
    z[..., 32:] = 60.0
    inp["z"] = z.to(io)
    d_out, _ = _cotangents(inp, seed=64)
    got = _run(inp, d_out, None)
    torch.cuda.synchronize()
    _check_all(got, _oracle(inp, d_out, None), inp, io, what="half floor")


def test_backward_sequence_gradients_only_from_the_final_state():
    """d_out = 0: every gradient comes through the final state (the chain through all chunks)."""
    inp = I.make_inputs(1, lengths=[90, 31], num_heads=2, d=128, io_dtype=torch.float32, seed=65)
    d_out, dsf = _cotangents(inp, seed=66)
    d_out = torch.zeros_like(d_out)
    got = _run(inp, d_out, dsf)
    torch.cuda.synchronize()
    _check_all(got, _oracle(inp, d_out, dsf), inp, torch.float32, what="final-state only")


def test_backward_deterministic_and_optional_outputs():
    inp = I.make_inputs(1, lengths=[100, 37], num_heads=2, d=128, seed=67)
    d_out, dsf = _cotangents(inp, seed=68)
    a = _run(inp, d_out, dsf)
    b = _run(inp, d_out, dsf, want_d_initial=False)
    torch.cuda.synchronize()
    assert b[6] is None
    for x, y in zip(a[:6], b[:6]):
        assert torch.equal(x, y)


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_backward_steepest_supported_floor(io):
    """g_min = -5.4, every log-decay at the floor: a chunk spans e^-86.4, close to the smallest
    normal fp32 number, and the gradients still match."""
    inp = I.make_inputs(1, lengths=[40, 33], num_heads=2, d=128, io_dtype=io, seed=72)
    inp["z"] = torch.full_like(inp["z"], 60.0)
    d_out, dsf = _cotangents(inp, seed=73)
    got = _run(inp, d_out, dsf, g_min=-5.4)
    torch.cuda.synchronize()
    _check_all(got, _oracle(inp, d_out, dsf, g_min=-5.4), inp, io, what="g_min -5.4")


def test_backward_steep_floor_is_unsupported():
    inp = I.make_inputs(1, lengths=[16], num_heads=1, d=32, seed=69)
    d_out, dsf = _cotangents(inp, seed=70)
    with pytest.raises(B.KdaError) as e:
        _run(inp, d_out, dsf, g_min=-6.0)
    assert e.value.status == B.KDA_ERR_UNSUPPORTED


def test_backward_many_short_sequences():
    """120 sequences of 0 to 40 tokens, bf16 d = 128: per-sequence chunk slots, states and dS0 at a
    large N."""
    g = torch.Generator().manual_seed(36)
    lengths = torch.randint(0, 41, (120,), generator=g).tolist()
    inp = I.make_inputs(1, lengths=lengths, num_heads=2, d=128, io_dtype=torch.bfloat16, seed=37, random_s0=True)
    d_out, dsf = _cotangents(inp, seed=38)
    got = _run(inp, d_out, dsf)
    torch.cuda.synchronize()
    ref = _oracle(inp, d_out, dsf)
    _check_all(got, ref, inp, torch.bfloat16, what="120 short sequences")


def test_backward_config1_sampled():
    """The 4096-token, 16-head, d = 128 bf16 workload: all heads on the GPU, the oracle's gradients
    on heads 0 and 9 (heads are independent)."""
    inp = I.make_inputs(1)
    d_out, dsf = _cotangents(inp, seed=71)
    got = _run(inp, d_out, dsf)
    torch.cuda.synchronize()
    heads = [0, 9]
    ref = _oracle(inp, d_out, dsf, heads=heads)
    z = inp["z"].double().numpy()[:, heads]
    names_tok = ("dq", "dk", "dv", "dz")
    for name, g, r in zip(names_tok, got[:4], ref[:4]):
        check(g[:, heads], r, torch.bfloat16, f"config 1 {name}")
    check(got[5][:, heads], ref[5], torch.bfloat16, "config 1 dbeta")
    check(got[6][:, heads], ref[6], torch.bfloat16, "config 1 dS0")
    dA = got[4].double().cpu().numpy()[heads]
    scale = np.abs(ref[3] * z).sum(axis=(0, 2))
    assert np.all(np.abs(dA - ref[4]) <= 1e-3 * scale)


def test_backward_config2_varlen_sampled():
    """The varlen workload (8 sequences of 1,024 .. 16,384 tokens, 32 heads, bf16): all gradients on the
    GPU; the oracle's gradients for the shortest sequence on heads 0 and 17 (sequences and heads are
    independent, so the sample is exact)."""
    inp = I.make_inputs(2)
    d_out, dsf = _cotangents(inp, seed=74)
    got = _run(inp, d_out, dsf)
    torch.cuda.synchronize()
    lengths = inp["lengths"]
    n = int(np.argmin(lengths))
    cu = inp["cu_seqlens"].numpy()
    t0, t1 = int(cu[n]), int(cu[n + 1])
    heads = [0, 17]
    sub = {x: inp[x][t0:t1][:, heads] for x in ("q", "k", "v", "z", "beta")}
    ref = oracle.backward(sub["q"], sub["k"], sub["v"], sub["z"], inp["A"][heads], sub["beta"],
                          d_out[t0:t1][:, heads], dsf[n:n + 1][:, heads], S0=inp["S0"][n:n + 1][:, heads])
    for name, g, r in zip(("dq", "dk", "dv", "dz"), got[:4], ref[:4]):
        check(g[t0:t1][:, heads], r, torch.bfloat16, f"config 2 {name}")
    check(got[5][t0:t1][:, heads], ref[5], torch.bfloat16, "config 2 dbeta")
    check(got[6][n:n + 1][:, heads], ref[6], torch.bfloat16, "config 2 dS0")
