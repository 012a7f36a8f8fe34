"""Stage parity on the GPU: intermediates of kda_forward read back from its workspace and compared with
the fp64 chunk-form restatement (``chunk_form.py``, itself matched to the token oracle) and with the
oracle's own runs over segments.

* split tensor-core plan (bf16, d = 128): every 32-token operand block -- W, Q Gamma, P, K~^T, U~ and
  Gamma_C of the pair, laid out for the state pass -- and the segment summaries (incoming states S_in,
  end states from zero S~, transitions M) of a segmented run;
* fp32 path: T = (I + A)^-1 and A, recovered from the stored U~ = T diag(beta) V (diag(beta) V has full
  row rank, so T = U~ pinv(diag(beta) V) exactly).
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrence_kda_gb300 import binding as B
from linear_attention_recurrence_kda_gb300 import inputs as I
from chunk_form import chunk_forward
from parity import check, err_max_rel, to_dev
from stages import (decode_block, fp32_stage_views, pair_reference, split_block, split_layout)

pytestmark = pytest.mark.gpu


def _np(inp):
    """The inputs as float64 numpy arrays (bf16 values upcast exactly)."""
    return {k: inp[k].double().numpy() for k in ("q", "k", "v", "z", "A", "beta", "S0") if inp.get(k) is not None}

# fp32-level arithmetic with hardware exp2 / reciprocal approximations in the decays: a layout, index
# or sign mistake moves these by O(1)
TOL_FP32_STAGE = 1e-3


def _bf16_rel_ok(got, ref, what, rel=2.0 ** -8):
    """bf16-stored operand: every element within its own rounding (plus fp32 noise) of the reference."""
    scale = np.abs(ref).max() if ref.size else 1.0
    bad = np.abs(got - ref) > rel * np.abs(ref) + 2.0 ** -14 * scale
    assert not bad.any(), f"{what}: {int(bad.sum())} elements outside bf16 rounding, max diff " \
                          f"{np.abs(got - ref).max():.3e} (max |ref| {scale:.3e})"


def _run_split(inp, monkeypatch, seg_chunks):
    monkeypatch.delenv("KDA_TC_PLAN", raising=False)
    monkeypatch.setenv("KDA_SEGMENT_CHUNKS", str(seg_chunks))
    lengths = inp["lengths"]
    T, N, H = sum(lengths), len(lengths), inp["q"].shape[1]
    prob = B.make_problem(N, T, max(lengths), H, 128, 128, torch.bfloat16)
    wsb = B.kda_forward_workspace_bytes(prob)
    plan = B.kda_forward_plan(prob, wsb)
    assert plan["split"]
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    d = to_dev(inp)
    B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"],
                  cu_seqlens=d["cu_seqlens"], max_seqlen=max(lengths), workspace=ws)
    torch.cuda.synchronize()
    assert B.kda_workspace_status(ws) == B.KDA_OK
    max_seg = plan["num_segments"]
    assert split_layout(T, N, H, max_seg)[4] == wsb  # the layout read below is the library's
    return ws.cpu().numpy(), plan


@pytest.mark.parametrize("floor", [False, True], ids=["random-decay", "decay-floor"])
def test_split_plan_operand_blocks(monkeypatch, floor):
    """Every 32-token operand block of a varlen batch (ragged last steps, a lone last chunk, an empty
    sequence) against the 32-token chunk form, with decays from random gates and at the floor."""
    lengths, H = [250, 0, 17, 64, 33], 2
    inp = I.make_inputs(1, lengths=lengths, num_heads=H, d=128, seed=31)
    if floor:
        inp["z"] = torch.full_like(inp["z"], 60.0)
    ws, _ = _run_split(inp, monkeypatch, 0)
    g, _ = oracle.gate(inp["z"], inp["A"])
    cu = inp["cu_seqlens"].numpy()
    x = _np(inp)
    worst = {}
    for n, L in enumerate(lengths):
        for h in range(H):
            for s in range((L + 31) // 32):
                t0 = int(cu[n]) + 32 * s
                t1 = min(t0 + 32, int(cu[n + 1]))
                got = decode_block(split_block(ws, cu, H, n, h, s))
                ref = pair_reference(x["q"], x["k"], x["v"], g, x["beta"], t0, t1, h)
                where = f"seq {n} head {h} step {s}"
                _bf16_rel_ok(got["QG"], ref["QG"], f"Q Gamma, {where}")
                # W is one bf16 operand; its second chunk's rows come from W_b Gamma_Ca - X W_a with
                # the bf16 W_a, so the bound is a bf16 ulp of the block's largest element
                e_w = err_max_rel(got["W"], ref["W"])
                worst["W"] = max(worst.get("W", 0.0), e_w)
                assert e_w <= 2.0 ** -7, f"W, {where}: max-rel {e_w:.3e}"
                for key in ("P", "KtT", "Ut"):
                    e = err_max_rel(got[key], ref[key])
                    worst[key] = max(worst.get(key, 0.0), e)
                    assert e <= TOL_FP32_STAGE, f"{key}, {where}: max-rel {e:.3e}"
                    assert np.isfinite(got[key]).all()
                gc_bad = np.abs(got["GC"] - ref["GC"]) > 1e-4 * ref["GC"] + 1e-30
                assert not gc_bad.any(), f"Gamma_C, {where}"
                # tokens beyond the sequence contribute nothing to the step
                c = t1 - t0
                assert not got["P"][:, c:].any() and not got["KtT"][:, c:].any() and not got["Ut"][c:].any()
                assert np.isfinite(got["W"]).all() and np.isfinite(got["QG"]).all()
    print("worst max-rel per stage:", {k: f"{v:.2e}" for k, v in worst.items()})


def test_split_plan_segment_summaries(monkeypatch):
    """Segments of 4 chunks: S_in (the scan's incoming state of every segment, the first one a copy of
    the initial state), S~ (end state from a zero start) and M (end state from the identity with
    v = 0: the segment's transition) against the oracle run over the same token ranges."""
    lengths, H, seg_tokens = [250, 100, 33, 0, 129], 2, 64
    inp = I.make_inputs(1, lengths=lengths, num_heads=H, d=128, seed=32)
    ws, plan = _run_split(inp, monkeypatch, 4)
    assert plan["seg_chunks"] == 4 and plan["num_segments"] == 4
    T, N, max_seg = sum(lengths), len(lengths), plan["num_segments"]
    _, seg_in, seg_st, seg_mt, _ = split_layout(T, N, H, max_seg)
    f32 = lambda off, cnt: ws[off:off + cnt * 4].view(np.float32).astype(np.float64)
    unit = 128 * 128
    S_in = f32(seg_in, N * H * max_seg * unit).reshape(N, H, max_seg, 128, 128)
    S_t = f32(seg_st, N * H * max_seg * unit).reshape(N, H, max_seg, 128, 128)
    mt = ws[seg_mt:seg_mt + N * H * max_seg * unit * 4].reshape(N, H, max_seg, unit * 4)
    cu = inp["cu_seqlens"].numpy()
    g, _ = oracle.gate(inp["z"], inp["A"])
    x = _np(inp)
    _, _, inter = chunk_forward(x["q"], x["k"], x["v"], g, x["beta"], S0=x["S0"], cu_seqlens=cu, keep=True)
    eye = np.broadcast_to(np.eye(128), (1, H, 128, 128)).copy()
    checked = 0
    for n, L in enumerate(lengths):
        nseg = max(1, -(-L // seg_tokens))
        for kseg in range(nseg):
            t0 = int(cu[n]) + kseg * seg_tokens
            t1 = min(t0 + seg_tokens, int(cu[n + 1]))
            if nseg >= 2:  # the scan writes incoming states of segmented sequences only
                ref_in = np.stack([inter[(n, h, 4 * kseg)]["S_in"] for h in range(H)])
                check(S_in[n, :, kseg], ref_in, torch.bfloat16, f"S_in seq {n} segment {kseg}")
            if kseg == nseg - 1:
                continue  # the last segment of a sequence needs no summary
            sl = lambda x: x[t0:t1]
            _, ref_st = oracle.forward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["z"]), inp["A"],
                                       sl(inp["beta"]))
            check(S_t[n, :, kseg], ref_st[0], torch.bfloat16, f"S~ seq {n} segment {kseg}")
            _, ref_m = oracle.forward(sl(inp["q"]), sl(inp["k"]), torch.zeros_like(sl(inp["v"])), sl(inp["z"]),
                                      inp["A"], sl(inp["beta"]), S0=torch.from_numpy(eye))
            for h in range(H):
                got_m = _decode_transition(mt[n, h, kseg])
                check(got_m, ref_m[0, h], torch.bfloat16, f"M seq {n} head {h} segment {kseg}")
            checked += 1
    assert checked == 6


def _decode_transition(buf):
    """A segment's M [c][j] from its 64 KiB scan operand: bf16 hi and lo planes of the row-major
    matrix, the 16-byte chunks of every 256-byte row permuted by XOR with c mod 8."""
    c = np.arange(128)[:, None]
    j = np.arange(128)[None, :]
    off = c * 256 + (((j // 8) ^ (c % 8)) * 16) + (j % 8) * 2
    u16 = lambda base: (buf[base + off].astype(np.uint32) | (buf[base + off + 1].astype(np.uint32) << 8)) << 16
    hi = u16(0).view(np.float32).astype(np.float64)
    lo = u16(128 * 128 * 2).view(np.float32).astype(np.float64)
    return hi + lo


@pytest.mark.parametrize("dk,dv", [(32, 64), (64, 128)])
def test_fp32_path_T_and_A(dk, dv):
    """T = (I + A)^-1 and A of every chunk of the fp32 path, recovered from the stored
    U~ = T diag(beta) V, against the chunk form's T and A."""
    lengths, H = [37, 0, 16, 50], 3
    inp = I.make_inputs(1, lengths=lengths, num_heads=H, d_k=dk, d_v=dv, io_dtype=torch.float32, seed=23 + dk)
    T, N = sum(lengths), len(lengths)
    d = to_dev(inp)
    prob = B.make_problem(N, T, max(lengths), H, dk, dv, torch.float32)
    ws = torch.zeros(B.kda_forward_workspace_bytes(prob), dtype=torch.uint8, device="cuda")
    B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"],
                  cu_seqlens=d["cu_seqlens"], max_seqlen=max(lengths), workspace=ws)
    torch.cuda.synchronize()
    _, _, Ut = fp32_stage_views(ws, T, H, dk, dv)
    g, _ = oracle.gate(inp["z"], inp["A"])
    cu = inp["cu_seqlens"].numpy()
    x = _np(inp)
    _, _, inter = chunk_forward(x["q"], x["k"], x["v"], g, x["beta"], S0=x["S0"], cu_seqlens=cu, keep=True)
    v = inp["v"].double().numpy()
    beta = inp["beta"].double().numpy()
    worst_t = worst_a = 0.0
    for (n, h, ci), st in inter.items():
        t0 = int(cu[n]) + 16 * ci
        c = st["Tinv"].shape[0]
        X = beta[t0:t0 + c, h, None] * v[t0:t0 + c, h]
        T_gpu = Ut[t0:t0 + c, h] @ np.linalg.pinv(X)
        e_t = err_max_rel(T_gpu, st["Tinv"])
        A_gpu = np.linalg.inv(T_gpu) - np.eye(c)
        e_a = np.abs(A_gpu - st["A"]).max() / max(1.0, np.abs(st["A"]).max())
        worst_t, worst_a = max(worst_t, e_t), max(worst_a, e_a)
        assert e_t <= TOL_FP32_STAGE, f"T, seq {n} head {h} chunk {ci}: {e_t:.3e}"
        assert e_a <= TOL_FP32_STAGE, f"A, seq {n} head {h} chunk {ci}: {e_a:.3e}"
        assert np.abs(np.triu(A_gpu)).max() <= TOL_FP32_STAGE  # strictly lower
    print(f"T max-rel {worst_t:.2e}, A {worst_a:.2e}")
