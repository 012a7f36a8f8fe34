"""Context-parallel prefill pieces on the GPU through the C ABI: the affine summary of a token range
(kda_forward_summary), the prefix scan of summaries (kda_state_scan), and the whole KCP flow for R
ranks emulated one after another on one GPU (each range summarised, the summaries stacked as the
all-gather would deliver them, the scan, the re-run from the scanned state) against the unsplit
oracle run."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrence_kda_gb300 import binding as B
from linear_attention_recurrence_kda_gb300 import inputs as I
from parity import check, to_dev

pytestmark = pytest.mark.gpu


def _oracle_summary(inp):
    """(M, S~) per sequence and head from the oracle: S~ from zero; M from the identity, values zero."""
    T, H, dk = inp["k"].shape
    N = len(inp["lengths"])
    cu = inp["cu_seqlens"]
    _, St = oracle.forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"], cu_seqlens=cu)
    eye = np.broadcast_to(np.eye(dk), (N, H, dk, dk)).copy()
    _, M = oracle.forward(inp["q"], inp["k"], torch.zeros(T, H, dk), inp["z"], inp["A"], inp["beta"], S0=eye,
                          cu_seqlens=cu)
    return M, St


@pytest.mark.parametrize("io,dk,dv", [(torch.bfloat16, 128, 128), (torch.float32, 64, 32), (torch.bfloat16, 32, 64)],
                         ids=["bf16-128", "f32-64x32", "bf16-32x64"])
def test_summary_matches_the_oracle(io, dk, dv):
    lengths = [70, 0, 33, 250]
    inp = I.make_inputs(1, lengths=lengths, num_heads=2, d_k=dk, d_v=dv, io_dtype=io, seed=81 + dk)
    d = to_dev(inp)
    M, St = B.kda_forward_summary(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    rM, rS = _oracle_summary(inp)
    check(M, rM, io, "transition M")
    check(St, rS, io, "state from zero S~")
    # an empty range is the identity map
    assert torch.equal(M[1].cpu(), torch.eye(dk).expand(2, dk, dk)) and not St[1].any()


def test_state_scan_composes_in_order():
    g = torch.Generator().manual_seed(82)
    R, N, H, dk, dv = 5, 3, 2, 128, 64
    Ms = torch.randn(R, N, H, dk, dk, generator=g) / np.sqrt(dk)
    Ss = torch.randn(R, N, H, dk, dv, generator=g)
    S0 = torch.randn(N, H, dk, dv, generator=g)
    Md, Sd, S0d = Ms.cuda(), Ss.cuda(), S0.cuda()
    for count in (0, 1, 3, 5):
        got = B.kda_state_scan(Md, Sd, initial_state=S0d, count=count)
        ref = S0.double()
        for i in range(count):
            ref = Ms[i].double() @ ref + Ss[i].double()
        torch.cuda.synchronize()
        check(got, ref.numpy(), torch.float32, f"scan of {count}")
    zero = B.kda_state_scan(Md, Sd, count=2)
    ref = Ms[1].double() @ Ss[0].double() + Ss[1].double()
    check(zero, ref.numpy(), torch.float32, "scan from zeros")
    inplace = S0d.clone()
    B.kda_state_scan(Md, Sd, initial_state=inplace, count=4, state_out=inplace)
    check(inplace, B.kda_state_scan(Md, Sd, initial_state=S0d, count=4).double().cpu().numpy(), torch.float32,
          "in place")


@pytest.mark.parametrize("ranks", [2, 4])
@pytest.mark.parametrize("io,d", [(torch.bfloat16, 128), (torch.float32, 64)], ids=["bf16-128", "f32-64"])
def test_kcp_flow_emulated_on_one_gpu(ranks, io, d):
    """Two sequences of 1,024 tokens split into `ranks` token ranges: the rank-by-rank flow gives the
    unsplit result (outputs of every range, the final state after the last)."""
    N, T, H = 2, 1024, 3
    inp = I.make_inputs(1, lengths=[T] * N, num_heads=H, d=d, io_dtype=io, seed=83 + ranks)
    d_ = to_dev(inp)
    Tr = T // ranks
    rows = [torch.cat([torch.arange(n * T + r * Tr, n * T + (r + 1) * Tr) for n in range(N)]).cuda()
            for r in range(ranks)]
    local = [{x: d_[x][rows[r]].contiguous() for x in ("q", "k", "v", "z", "beta")} for r in range(ranks)]
    summ = [B.kda_forward_summary(l["q"], l["k"], l["v"], l["z"], d_["A"], l["beta"], num_seqs=N) for l in local]
    Ms = torch.stack([m for m, _ in summ])
    Ss = torch.stack([s for _, s in summ])
    outs, last = [], None
    for r in range(ranks):
        S_in = B.kda_state_scan(Ms, Ss, initial_state=d_["S0"], count=r)
        o, last = B.kda_forward(local[r]["q"], local[r]["k"], local[r]["v"], local[r]["z"], d_["A"], local[r]["beta"],
                                initial_state=S_in)
        outs.append(o.view(N, Tr, H, d))
    torch.cuda.synchronize()
    out = torch.cat(outs, dim=1).reshape(N * T, H, d)
    ref_o, ref_s = oracle.forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"], S0=inp["S0"],
                                  cu_seqlens=inp["cu_seqlens"])
    check(out, ref_o, io, f"KCP outputs over {ranks} ranges")
    check(last, ref_s, io, f"KCP final state over {ranks} ranges")


def test_summaries_compose_at_length():
    """A property that holds at any size: for a 65,536-token range split into halves r1, r2, the maps
    compose, M(r) = M(r2) M(r1) and S~(r) = M(r2) S~(r1) + S~(r2), with each summary computed by
    kda_forward_summary on the tensor-core path (segmented inside for the whole range and the halves)."""
    T, H, d = 65536, 2, 128
    g = torch.Generator(device="cuda").manual_seed(84)
    import cases
    q, k, v, z = cases.device_tokens(g, (T, H), d, torch.bfloat16, torch.device("cuda"))
    A = (torch.randn(H, generator=g, device="cuda") * I.A_STD).float()
    beta = torch.sigmoid(torch.randn(T, H, generator=g, device="cuda")).float()
    M, St = B.kda_forward_summary(q, k, v, z, A, beta)
    h = T // 2
    halves = [B.kda_forward_summary(*(t[a:b].contiguous() for t in (q, k, v, z)), A, beta[a:b].contiguous())
              for a, b in ((0, h), (h, T))]
    (M1, S1), (M2, S2) = halves
    Mc = M2.double() @ M1.double()
    Sc = M2.double() @ S1.double() + S2.double()
    torch.cuda.synchronize()
    check(M, Mc.cpu().numpy(), torch.bfloat16, "composed transition")
    check(St, Sc.cpu().numpy(), torch.bfloat16, "composed state from zero")
    # and applying the composed map to a state equals running the range from it
    S0 = (torch.randn(1, H, d, d, generator=g, device="cuda") * I.S0_STD).float()
    _, S_run = B.kda_forward(q, k, v, z, A, beta, initial_state=S0)
    S_map = B.kda_state_scan(torch.stack([M1, M2]), torch.stack([S1, S2]), initial_state=S0)
    torch.cuda.synchronize()
    check(S_map, S_run.double().cpu().numpy(), torch.bfloat16, "scanned halves vs the run")
