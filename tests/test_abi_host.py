"""C-ABI checks that need no GPU: the library loads, exports every symbol include/kda.h declares,
and rejects bad descriptors, pointers, aliasing and workspaces on the host before any launch.

Every kda_forward / kda_decode_step / kda_decode_replay / kda_prologue / kda_epilogue call below is built to fail in a host-only check (the fake
addresses are never dereferenced and nothing is launched)."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT
from linear_attention_recurrence_kda_gb300 import binding as B

HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(B.LIB_PATH):
        from linear_attention_recurrence_kda_gb300 import build
        build.build()
    return B.lib()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert set(_declared_functions()) == set(B.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True, check=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in _declared_functions():
        assert name in syms, name
        assert hasattr(L, name)


def test_abi_version_and_status_strings(L):
    assert B.kda_abi_version() == (1 << 16) | 5
    for code in range(7):
        s = B.status_string(code)
        assert s.startswith("KDA_")
    assert "unknown" in B.status_string(99)


def _prob(**kw):
    base = dict(num_seqs=1, total_tokens=64, max_seqlen=64, num_heads=2, d_k=32, d_v=32, io_dtype=B.KDA_F32, g_min=-5.0)
    base.update(kw)
    return B.make_problem(**base)


def test_workspace_bytes(L, monkeypatch):
    p = _prob()
    n = B.kda_forward_workspace_bytes(p)
    # check word + G, W (d_k) and U~ (d_v) in fp32 for every token-head
    assert n >= 256 + 64 * 2 * (32 + 32 + 32) * 4
    assert n % 256 == 0
    # bf16 inputs with d_k = d_v = 128: the fastest plan holds one 53,760-byte operand block per
    # 32-token step slot (T_tot / 32 + N + 1 slots) and head, plus per-segment states
    big = _prob(total_tokens=1 << 20, max_seqlen=1 << 20, num_heads=8, d_k=128, d_v=128, io_dtype=B.KDA_BF16)
    blocks = ((1 << 20) // 32 + 1 + 1) * 8 * 53760
    assert blocks <= B.kda_forward_workspace_bytes(big) < blocks + (1 << 30)
    # the fused kernel needs no per-token scratch
    monkeypatch.setenv("KDA_TC_PLAN", "fused")
    assert 256 <= B.kda_forward_workspace_bytes(big) < 1 << 30
    monkeypatch.delenv("KDA_TC_PLAN")
    simt_big = _prob(total_tokens=1 << 20, max_seqlen=1 << 20, num_heads=8, d_k=128, d_v=128)
    assert B.kda_forward_workspace_bytes(simt_big) > B.kda_forward_workspace_bytes(p)
    for bad in (_prob(d_k=96), _prob(num_heads=0), _prob(g_min=0.0), _prob(g_min=float("nan")),
                _prob(io_dtype=7), _prob(total_tokens=-1), _prob(num_seqs=0)):
        assert B.kda_forward_workspace_bytes(bad) == 0


# fake, 256-byte aligned, non-overlapping addresses; never dereferenced
_BASE = 0x7000_0000_0000


def _addr(i, size=1 << 24):
    return _BASE + i * size


def _fwd(L, prob, **over):
    names = ["q", "k", "v", "z", "A", "beta", "s0", "cu", "out", "sf"]
    ptr = {n: _addr(i) for i, n in enumerate(names)}
    ptr["s0"] = None
    ptr["cu"] = None
    ptr["sf"] = None
    ws = over.pop("ws", _addr(20))
    wsb = over.pop("wsb", 1 << 30)
    ptr.update(over)
    args = [ctypes.c_void_p(ptr[n]) if ptr[n] is not None else None for n in names]
    return L.kda_forward(*args, ctypes.byref(prob), ctypes.c_void_p(ws) if ws else None, ctypes.c_size_t(wsb), None)


def test_forward_rejects_bad_descriptors(L):
    assert L.kda_forward(None, None, None, None, None, None, None, None, None, None, None, None, 0, None) == B.KDA_ERR_INVALID_ARG
    assert _fwd(L, _prob(d_k=48)) == B.KDA_ERR_UNSUPPORTED
    assert _fwd(L, _prob(d_v=256)) == B.KDA_ERR_UNSUPPORTED
    assert _fwd(L, _prob(g_min=1.0)) == B.KDA_ERR_INVALID_ARG
    assert _fwd(L, _prob(num_heads=70000)) == B.KDA_ERR_INVALID_ARG
    assert _fwd(L, _prob(max_seqlen=-1)) == B.KDA_ERR_INVALID_ARG
    # equal lengths need T_tot divisible by N
    assert _fwd(L, _prob(num_seqs=3, total_tokens=64)) == B.KDA_ERR_INVALID_ARG


def test_forward_rejects_missing_and_misaligned_pointers(L):
    p = _prob()
    for name in ("q", "k", "v", "z", "A", "beta", "out"):
        assert _fwd(L, p, **{name: None}) == B.KDA_ERR_INVALID_ARG, name
    for name in ("q", "k", "v", "z", "out"):
        assert _fwd(L, p, **{name: _addr(3) + 8}) == B.KDA_ERR_INVALID_ARG, name
    assert _fwd(L, p, s0=_addr(11) + 4) == B.KDA_ERR_INVALID_ARG
    assert _fwd(L, p, A=_addr(4) + 2) == B.KDA_ERR_INVALID_ARG


def test_forward_rejects_overlap(L):
    p = _prob()
    assert _fwd(L, p, out=_addr(0)) == B.KDA_ERR_INVALID_ARG            # out == q
    assert _fwd(L, p, out=_addr(3) + 256) == B.KDA_ERR_INVALID_ARG      # out inside z
    assert _fwd(L, p, sf=_addr(1)) == B.KDA_ERR_INVALID_ARG             # final state on k
    assert _fwd(L, p, s0=_addr(11), sf=_addr(11) + 256) == B.KDA_ERR_INVALID_ARG  # partial overlap
    assert _fwd(L, p, ws=_addr(5)) == B.KDA_ERR_INVALID_ARG             # workspace on beta


def test_forward_rejects_bad_workspace(L):
    p = _prob()
    need = B.kda_forward_workspace_bytes(p)
    assert _fwd(L, p, ws=0) == B.KDA_ERR_WORKSPACE
    assert _fwd(L, p, ws=_addr(20) + 16) == B.KDA_ERR_WORKSPACE
    assert _fwd(L, p, wsb=need - 1) == B.KDA_ERR_WORKSPACE


def test_decode_rejects_bad_arguments(L):
    def dec(prob, **over):
        names = ["q", "k", "v", "z", "A", "beta", "state", "out"]
        ptr = {n: _addr(i) for i, n in enumerate(names)}
        ptr.update(over)
        args = [ctypes.c_void_p(ptr[n]) if ptr[n] is not None else None for n in names]
        return L.kda_decode_step(*args, ctypes.byref(prob), None)

    p = _prob(num_seqs=4, total_tokens=4, max_seqlen=1)
    assert dec(_prob(num_seqs=4, total_tokens=5)) == B.KDA_ERR_INVALID_ARG
    assert dec(_prob(num_seqs=4, total_tokens=4, d_k=16)) == B.KDA_ERR_UNSUPPORTED
    for name in ("q", "k", "v", "z", "A", "beta", "state", "out"):
        assert dec(p, **{name: None}) == B.KDA_ERR_INVALID_ARG, name
    assert dec(p, state=_addr(6) + 4) == B.KDA_ERR_INVALID_ARG
    assert dec(p, out=_addr(6)) == B.KDA_ERR_INVALID_ARG       # out on the state
    assert dec(p, state=_addr(2)) == B.KDA_ERR_INVALID_ARG     # state on v


def test_replay_rejects_bad_arguments(L):
    names = ["q", "k", "v", "z", "A", "beta", "state_in", "accepted", "state_out", "out"]

    def rep(prob, **over):
        ptr = {n: _addr(i) for i, n in enumerate(names)}
        ptr.update(over)
        args = [ctypes.c_void_p(ptr[n]) if ptr[n] is not None else None for n in names]
        return L.kda_decode_replay(*args, ctypes.byref(prob), None)

    p = _prob(num_seqs=4, total_tokens=12, max_seqlen=3)
    assert rep(_prob(num_seqs=4, total_tokens=10)) == B.KDA_ERR_INVALID_ARG   # not N equal windows
    assert rep(_prob(num_seqs=4, total_tokens=0)) == B.KDA_ERR_INVALID_ARG    # empty windows
    assert rep(_prob(num_seqs=4, total_tokens=12, d_v=16)) == B.KDA_ERR_UNSUPPORTED
    for name in ("q", "k", "v", "z", "A", "beta", "state_in"):
        assert rep(p, **{name: None}) == B.KDA_ERR_INVALID_ARG, name
    assert rep(p, out=None, state_out=None) == B.KDA_ERR_INVALID_ARG        # nothing to write
    assert rep(p, state_out=_addr(8) + 8) == B.KDA_ERR_INVALID_ARG          # misaligned
    assert rep(p, accepted=_addr(7) + 2) == B.KDA_ERR_INVALID_ARG
    assert rep(p, out=_addr(6)) == B.KDA_ERR_INVALID_ARG                    # out on the snapshot
    assert rep(p, state_out=_addr(0)) == B.KDA_ERR_INVALID_ARG              # state_out on q
    assert rep(p, state_out=_addr(7)) == B.KDA_ERR_INVALID_ARG              # state_out on accepted
    assert rep(p, state_out=_addr(6) + 16) == B.KDA_ERR_INVALID_ARG         # partly on the snapshot


def test_prologue_and_epilogue_reject_bad_arguments(L):
    pro_names = ["xq", "xk", "xv", "wq", "wk", "wv", "cu", "q", "k", "v"]

    def pro(prob, K=4, **over):
        ptr = {n: _addr(i) for i, n in enumerate(pro_names)}
        ptr["cu"] = None
        ptr.update(over)
        a = [ctypes.c_void_p(ptr[n]) if ptr[n] is not None else None for n in pro_names]
        return L.kda_prologue(*a[:6], ctypes.c_int32(K), *a[6:], ctypes.byref(prob), None)

    p = _prob(num_seqs=2, total_tokens=64)
    assert pro(p, K=0) == B.KDA_ERR_UNSUPPORTED
    assert pro(p, K=5) == B.KDA_ERR_UNSUPPORTED
    assert pro(_prob(num_seqs=3, total_tokens=64)) == B.KDA_ERR_INVALID_ARG   # unequal lengths without offsets
    for name in ("xq", "xk", "xv", "wq", "wk", "wv", "q", "k", "v"):
        assert pro(p, **{name: None}) == B.KDA_ERR_INVALID_ARG, name
    assert pro(p, q=_addr(7) + 8) == B.KDA_ERR_INVALID_ARG                   # misaligned
    assert pro(p, wk=_addr(4) + 2) == B.KDA_ERR_INVALID_ARG
    assert pro(p, q=_addr(0)) == B.KDA_ERR_INVALID_ARG                       # in place is not allowed
    assert pro(p, v=_addr(7)) == B.KDA_ERR_INVALID_ARG                       # outputs overlap
    assert pro(p, k=_addr(5)) == B.KDA_ERR_INVALID_ARG                       # output on the weights

    epi_names = ["o", "gate", "weight", "y"]

    def epi(prob, eps=1e-5, **over):
        ptr = {n: _addr(i) for i, n in enumerate(epi_names)}
        ptr.update(over)
        a = [ctypes.c_void_p(ptr[n]) if ptr[n] is not None else None for n in epi_names]
        return L.kda_epilogue(a[0], a[1], a[2], ctypes.c_float(eps), a[3], ctypes.byref(prob), None)

    for name in epi_names:
        assert epi(p, **{name: None}) == B.KDA_ERR_INVALID_ARG, name
    assert epi(p, eps=-1.0) == B.KDA_ERR_INVALID_ARG
    assert epi(p, eps=float("inf")) == B.KDA_ERR_INVALID_ARG
    assert epi(p, y=_addr(1)) == B.KDA_ERR_INVALID_ARG                       # y on the gate
    assert epi(p, y=_addr(0) + 16) == B.KDA_ERR_INVALID_ARG                  # partly on o
    assert epi(_prob(d_v=16)) == B.KDA_ERR_UNSUPPORTED


def test_workspace_status_rejects_null(L):
    assert L.kda_workspace_status(None, 0, None) == B.KDA_ERR_WORKSPACE



def test_forward_plan(L, monkeypatch):
    """kda_forward_plan reports the plan kda_forward would take for a workspace size."""
    monkeypatch.delenv("KDA_TC_PLAN", raising=False)
    monkeypatch.delenv("KDA_SEGMENT_CHUNKS", raising=False)
    p = _prob(total_tokens=4096, max_seqlen=4096, num_heads=16, d_k=128, d_v=128, io_dtype=B.KDA_BF16)
    fast = B.kda_forward_plan(p)
    assert fast["split"] and fast["num_segments"] > 1 and fast["seg_chunks"] * fast["num_segments"] >= 256
    assert B.kda_forward_plan(p, B.kda_forward_workspace_bytes(p)) == fast
    # the 256-byte minimum: fused kernel, one segment
    assert B.kda_forward_plan(p, 256) == {"split": False, "seg_chunks": 0, "num_segments": 1}
    monkeypatch.setenv("KDA_TC_PLAN", "fused")
    assert not B.kda_forward_plan(p)["split"]
    monkeypatch.setenv("KDA_SEGMENT_CHUNKS", "0")
    assert B.kda_forward_plan(p)["num_segments"] == 1
    monkeypatch.delenv("KDA_TC_PLAN")
    monkeypatch.setenv("KDA_SEGMENT_CHUNKS", "64")
    assert B.kda_forward_plan(p) == {"split": True, "seg_chunks": 64, "num_segments": 4}
    # the split plan steps the state by pairs of chunks: an odd count is rounded up
    monkeypatch.setenv("KDA_SEGMENT_CHUNKS", "3")
    assert B.kda_forward_plan(p) == {"split": True, "seg_chunks": 4, "num_segments": 64}
    monkeypatch.setenv("KDA_TC_PLAN", "fused")
    assert B.kda_forward_plan(p) == {"split": False, "seg_chunks": 3, "num_segments": 86}
    monkeypatch.delenv("KDA_TC_PLAN")
    monkeypatch.delenv("KDA_SEGMENT_CHUNKS")
    # the planner's own choice for the split plan is a whole number of pairs
    for T in (4096, 3000, 65536):
        pl = B.kda_forward_plan(_prob(total_tokens=T, max_seqlen=T, num_heads=16, d_k=128, d_v=128,
                                      io_dtype=B.KDA_BF16))
        assert pl["split"] and pl["seg_chunks"] % 2 == 0
    # the fp32 path needs per-token scratch: below it the call is refused
    with pytest.raises(B.KdaError) as e:
        B.kda_forward_plan(_prob(), 256)
    assert e.value.status == B.KDA_ERR_WORKSPACE
    with pytest.raises(B.KdaError) as e:
        B.kda_forward_plan(_prob(d_k=96))
    assert e.value.status == B.KDA_ERR_UNSUPPORTED
    assert L.kda_forward_plan(ctypes.byref(p), ctypes.c_size_t(1 << 40), None) == B.KDA_ERR_INVALID_ARG


@pytest.mark.parametrize("T,N,H", [(4096, 1, 16), (58337, 8, 32), (1 << 20, 1, 8), (300, 3, 4), (16, 1, 1)])
def test_forward_plan_properties(L, monkeypatch, T, N, H):
    """Over workspace sizes from the fastest plan's need down to the 256-byte minimum, every plan
    fits, its segments cover the longest sequence without an empty last segment, the split plan's
    segments hold whole pairs of chunks, and any workspace at least the reported need gets the
    fastest plan."""
    monkeypatch.delenv("KDA_TC_PLAN", raising=False)
    monkeypatch.delenv("KDA_SEGMENT_CHUNKS", raising=False)
    max_len = -(-T // N) if N > 1 else T
    p = _prob(num_seqs=N, total_tokens=T, max_seqlen=max_len, num_heads=H, d_k=128, d_v=128, io_dtype=B.KDA_BF16)
    full = B.kda_forward_workspace_bytes(p)
    assert full >= 256 and full % 256 == 0
    fastest = B.kda_forward_plan(p, full)
    assert B.kda_forward_plan(p, 2 * full) == fastest
    chunks = -(-max_len // 16)
    for frac in (1.0, 0.7, 0.5, 0.3, 0.1, 0.02, 0.005, 0.0):
        ws = max(256, int(full * frac))
        pl = B.kda_forward_plan(p, ws)
        if pl["num_segments"] > 1:
            sc, ns = pl["seg_chunks"], pl["num_segments"]
            assert sc * ns >= chunks and (ns - 1) * sc < chunks, (ws, pl)
            if pl["split"]:
                assert sc % 2 == 0, (ws, pl)
        else:
            assert pl["seg_chunks"] == 0
    assert B.kda_forward_plan(p, 256) == {"split": False, "seg_chunks": 0, "num_segments": 1}


def test_compute_entry_points_cite_their_passage():
    """Every computing entry point's declaration in include/kda.h is preceded by a comment that
    names the page and section defining the operation."""
    src = open(HEADER).read()
    for name in ("kda_forward", "kda_decode_step", "kda_decode_replay", "kda_prologue", "kda_epilogue",
                 "kda_backward", "kda_forward_summary", "kda_state_scan"):
        decl = src.index(f"kda_status_t {name}(")
        comment = src[src.rindex("/*", 0, decl):decl]
        assert "Kimi K3" in comment and "section" in comment, name


def test_fp32_stage_layout_matches_the_library():
    """The layout the stage-parity test reads (check word, G, W, U~) has exactly the size the
    library reports for the fp32 path, and packing then reading it round-trips."""
    import numpy as np
    import torch
    from stages import fp32_stage_layout, fp32_stage_views
    for (T, H, dk, dv) in ((120, 3, 32, 64), (1, 1, 128, 32), (1000, 2, 64, 128)):
        p = _prob(num_seqs=1, total_tokens=T, max_seqlen=T, num_heads=H, d_k=dk, d_v=dv)
        assert fp32_stage_layout(T, H, dk, dv)[3] == B.kda_forward_workspace_bytes(p)
    T, H, dk, dv = 37, 2, 32, 64
    g_off, w_off, ut_off, total = fp32_stage_layout(T, H, dk, dv)
    rng = np.random.default_rng(0)
    ref = [rng.normal(size=(T, H, d)).astype(np.float32) for d in (dk, dk, dv)]
    ws = torch.zeros(total, dtype=torch.uint8)
    for off, a in zip((g_off, w_off, ut_off), ref):
        ws[off:off + a.nbytes] = torch.from_numpy(a.reshape(-1).view(np.uint8).copy())
    for got, want in zip(fp32_stage_views(ws, T, H, dk, dv), ref):
        np.testing.assert_array_equal(got, want)


def test_split_stage_layout_matches_the_library(monkeypatch):
    """The split-plan layout the stage-parity tests read (check word, operand blocks, then S_in, S~
    and M per segment) has exactly the size the library reports, unsegmented and segmented."""
    from stages import split_layout
    for seg in ("0", "4", "2"):
        monkeypatch.setenv("KDA_SEGMENT_CHUNKS", seg)
        for (N, T, ml, H) in ((5, 464, 250, 2), (1, 4096, 4096, 16), (3, 97, 64, 1)):
            p = _prob(num_seqs=N, total_tokens=T, max_seqlen=ml, num_heads=H, d_k=128, d_v=128, io_dtype=B.KDA_BF16)
            wsb = B.kda_forward_workspace_bytes(p)
            pl = B.kda_forward_plan(p, wsb)
            assert pl["split"]
            assert split_layout(T, N, H, pl["num_segments"])[4] == wsb, (seg, N, T, H, pl)
