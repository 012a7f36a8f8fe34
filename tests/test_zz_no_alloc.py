"""kda_forward_static_scratch: the prefill entry point for callers that cannot allocate device memory
(for example a plugin inside a host application that owns every device allocation and hands the
plugin no allocator).  It must give the same results as kda_forward, call after call, while its
scratch comes from the library's own fixed-size device array instead of a caller workspace.

This file is named so that pytest collects it last."""
import pytest
import torch

from linear_attention_recurrence_kda_gb300 import binding as B
from linear_attention_recurrence_kda_gb300 import inputs as I
from parity import check, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # bf16, d = 128: the tensor-core path (a few hundred bytes of scratch), varlen with a ragged tail
    dict(lengths=[300, 17, 0, 64], heads=3, d=128, io=torch.bfloat16),
    # fp32, d = 64: the fp32 path, whose per-token scratch (4 (2 d_k + d_v) B per token-head) fits
    dict(lengths=[150, 33], heads=2, d=64, io=torch.float32),
]


@pytest.mark.parametrize("case", CASES, ids=["bf16-d128", "f32-d64"])
def test_matches_kda_forward_on_two_calls_in_a_row(case):
    for call in range(2):
        inp = I.make_inputs(1, lengths=case["lengths"], num_heads=case["heads"], d=case["d"], io_dtype=case["io"],
                            seed=100 + call)
        d = to_dev(inp)
        ml = max(case["lengths"])
        ref_o, ref_s = B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"],
                                     cu_seqlens=d["cu_seqlens"], max_seqlen=ml)
        out, fin = B.kda_forward_static_scratch(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"],
                                                initial_state=d["S0"], cu_seqlens=d["cu_seqlens"], max_seqlen=ml)
        torch.cuda.synchronize()
        check(out, ref_o.double().cpu().numpy(), case["io"], f"out, call {call}")
        check(fin, ref_s.double().cpu().numpy(), case["io"], f"final state, call {call}")


def test_rejects_problems_larger_than_the_static_scratch():
    # fp32 path, 8 heads x 8192 tokens x d = 128 needs 48 MiB of scratch: refused before any launch
    T, H, d = 8192, 8, 128
    prob = B.make_problem(1, T, T, H, d, d, torch.float32)
    assert B.kda_forward_workspace_bytes(prob) > B.KDA_STATIC_SCRATCH_BYTES
    dev = torch.device("cuda")
    x = torch.zeros(T, H, d, device=dev)
    A = torch.zeros(H, device=dev)
    beta = torch.zeros(T, H, device=dev)
    out = torch.full((T, H, d), 3.0, device=dev)
    with pytest.raises(B.KdaError) as e:
        B.kda_forward_static_scratch(x, x.clone(), x.clone(), x.clone(), A, beta, out=out)
    assert e.value.status == B.KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)


def test_static_scratch_status_reports_bad_offsets():
    """The check word of a call without a workspace is read back through kda_static_scratch_status:
    offsets that violate the descriptor are reported (the bad sequences skipped, the good one
    computed), and the next valid call clears the word."""
    inp = I.make_inputs(1, lengths=[32, 32, 32], num_heads=2, d=32, io_dtype=torch.float32, seed=16)
    d = to_dev(inp)
    bad = torch.tensor([0, 32, 20, 96], dtype=torch.int32, device="cuda")  # lengths 32, -12, 76 > 64
    out = torch.full((96, 2, 32), 7.0, device="cuda")
    B.kda_forward_static_scratch(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"],
                                 cu_seqlens=bad, max_seqlen=64, out=out)
    assert B.kda_static_scratch_status() == B.KDA_ERR_DEVICE_CHECK
    assert torch.all(out[32:] == 7.0)
    ref_o, _ = B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"],
                             cu_seqlens=d["cu_seqlens"], max_seqlen=32)
    check(out[:32], ref_o[:32].double().cpu().numpy(), torch.float32, "sequence 0")
    B.kda_forward_static_scratch(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], cu_seqlens=d["cu_seqlens"],
                                 max_seqlen=32)
    assert B.kda_static_scratch_status() == B.KDA_OK
