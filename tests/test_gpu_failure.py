"""The failure path of the bounded device waits, driven without any GPU fault.

The split plan's state pass hands work between its warp roles through mbarriers, and every such
wait is bounded: one that gives up raises the CTA's stop flag, everyone leaves at their next wait,
the control thread waits (with the full limit) for its copies and tensor-core work in flight, the
CTA frees its tensor memory, and the call's check word reports KDA_ERR_TIMEOUT.  The debugging
knob KDA_DEBUG_HANDOFF_TRIES shortens the hand-off waits so that they run out: with 0 tries every
hand-off wait gives up at once, with 1 or 3 tries some give up somewhere in the middle of a chain.
The tests check that the status is reported, that nothing faults, and that the next normal call in
the same context still matches the oracle.
"""
import pytest
import torch

from linear_attention_recurrence_kda_gb300 import binding as B
from linear_attention_recurrence_kda_gb300 import inputs as I
from parity import check, gpu_forward, oracle_forward, to_dev

pytestmark = pytest.mark.gpu


def _call(inp, ws=None):
    d = to_dev(inp)
    lengths = inp["lengths"]
    return B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"],
                         cu_seqlens=d["cu_seqlens"], max_seqlen=max(lengths), workspace=ws)


def _workspace(inp):
    lengths = inp["lengths"]
    prob = B.make_problem(len(lengths), sum(lengths), max(lengths), inp["q"].shape[1], 128, 128, torch.bfloat16)
    assert B.kda_forward_plan(prob)["split"]
    return torch.empty(B.kda_forward_workspace_bytes(prob), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("seg", ["0", "2"], ids=["unsegmented", "segmented"])
def test_handoff_timeout_is_reported(monkeypatch, seg):
    """0 tries: the first hand-off wait of every state-pass CTA gives up (T = 64, H = 1, d = 128)."""
    monkeypatch.delenv("KDA_TC_PLAN", raising=False)
    monkeypatch.setenv("KDA_SEGMENT_CHUNKS", seg)
    inp = I.make_inputs(1, lengths=[64], num_heads=1, d=128, seed=51)
    ws = _workspace(inp)
    monkeypatch.setenv("KDA_DEBUG_HANDOFF_TRIES", "0")
    _call(inp, ws)
    assert B.kda_workspace_status(ws) == B.KDA_ERR_TIMEOUT
    monkeypatch.delenv("KDA_DEBUG_HANDOFF_TRIES")
    # the context is intact: a normal call (fresh workspace) matches the oracle, and the same
    # workspace reports OK again after a normal call
    out, sf = gpu_forward(inp)
    ref_o, ref_s = oracle_forward(inp)
    check(out, ref_o, torch.bfloat16, "out after a timeout")
    check(sf, ref_s, torch.bfloat16, "final state after a timeout")
    _call(inp, ws)
    assert B.kda_workspace_status(ws) == B.KDA_OK


@pytest.mark.parametrize("tries", ["1", "3"])
def test_handoff_timeouts_mid_chain(monkeypatch, tries):
    """A few tries: hand-off waits give up at varying steps of the chains (or not at all).  Whatever
    happens the call reports OK with correct results or KDA_ERR_TIMEOUT, and the next normal call
    is correct."""
    monkeypatch.delenv("KDA_TC_PLAN", raising=False)
    monkeypatch.setenv("KDA_SEGMENT_CHUNKS", "8")
    inp = I.make_inputs(1, lengths=[512, 200, 33], num_heads=4, d=128, seed=52)
    ws = _workspace(inp)
    ref_o, ref_s = oracle_forward(inp)
    monkeypatch.setenv("KDA_DEBUG_HANDOFF_TRIES", tries)
    seen = set()
    for _ in range(3):
        out, sf = _call(inp, ws)
        st = B.kda_workspace_status(ws)
        assert st in (B.KDA_OK, B.KDA_ERR_TIMEOUT)
        seen.add(st)
        if st == B.KDA_OK:
            check(out, ref_o, torch.bfloat16, "out")
            check(sf, ref_s, torch.bfloat16, "final state")
    monkeypatch.delenv("KDA_DEBUG_HANDOFF_TRIES")
    out, sf = _call(inp, ws)
    assert B.kda_workspace_status(ws) == B.KDA_OK
    check(out, ref_o, torch.bfloat16, "out after the shortened waits")
    check(sf, ref_s, torch.bfloat16, "final state after the shortened waits")
    print(f"tries={tries}: statuses seen {sorted(seen)}")


def test_handoff_timeout_through_the_static_scratch(monkeypatch):
    """The same report for the entry point without a workspace, read with kda_static_scratch_status."""
    monkeypatch.delenv("KDA_TC_PLAN", raising=False)
    monkeypatch.delenv("KDA_SEGMENT_CHUNKS", raising=False)
    inp = I.make_inputs(1, lengths=[96], num_heads=2, d=128, seed=53)
    d = to_dev(inp)
    monkeypatch.setenv("KDA_DEBUG_HANDOFF_TRIES", "0")
    B.kda_forward_static_scratch(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"])
    assert B.kda_static_scratch_status() == B.KDA_ERR_TIMEOUT
    monkeypatch.delenv("KDA_DEBUG_HANDOFF_TRIES")
    out, sf = B.kda_forward_static_scratch(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"])
    assert B.kda_static_scratch_status() == B.KDA_OK
    ref_o, ref_s = oracle_forward(inp)
    check(out, ref_o, torch.bfloat16, "out")
    check(sf, ref_s, torch.bfloat16, "final state")
