"""GPU parity: kda_forward / kda_decode_step through the C ABI against the fp64 oracle, element by
element on the same seeded inputs, plus bit-exact pins, edge cases and invariants."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrence_kda_gb300 import binding as B
from linear_attention_recurrence_kda_gb300 import inputs as I
from parity import check, gpu_forward, oracle_forward, to_dev, TOL_BF16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.lib()


def _f64(t):
    return t.detach().double().cpu().numpy()


# ---------------------------------------------------------------- small shapes, both dtypes

SMALL = [
    ([1], 32, 32), ([15], 32, 32), ([16], 64, 64), ([17], 32, 64), ([33], 128, 128), ([64], 128, 64),
    ([5, 0, 40, 16, 1], 64, 128), ([100, 3, 77], 128, 32), ([0], 32, 32), ([250], 128, 128),
]


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("lengths,dk,dv", SMALL)
@pytest.mark.parametrize("with_s0", [False, True], ids=["s0zero", "s0rand"])
def test_forward_small(io, lengths, dk, dv, with_s0):
    inp = I.make_inputs(1, lengths=lengths, num_heads=3, d_k=dk, d_v=dv, io_dtype=io,
                        seed=sum(lengths) + dk + dv, random_s0=with_s0)
    out, sf = gpu_forward(inp)
    ref_o, ref_s = oracle_forward(inp)
    check(out, ref_o, io, "out")
    check(sf, ref_s, io, "final_state")


def test_config0_full_fp32():
    inp = I.make_inputs(0)
    out, sf = gpu_forward(inp)
    ref_o, ref_s = oracle_forward(inp)
    e1 = check(out, ref_o, torch.float32, "out")
    e2 = check(sf, ref_s, torch.float32, "final_state")
    print(f"config 0: out max-rel {e1:.2e}, state max-rel {e2:.2e}")


def test_config1_full_bf16():
    inp = I.make_inputs(1)
    out, sf = gpu_forward(inp)
    ref_o, ref_s = oracle_forward(inp)
    e1 = check(out, ref_o, torch.bfloat16, "out")
    e2 = check(sf, ref_s, torch.bfloat16, "final_state")
    print(f"config 1: out max/RMS {e1:.2e}, state max/RMS {e2:.2e}")


def test_config2_varlen_full():
    inp = I.make_inputs(2)
    out, sf = gpu_forward(inp)
    ref_o, ref_s = oracle_forward(inp)
    e1 = check(out, ref_o, torch.bfloat16, "out")
    e2 = check(sf, ref_s, torch.bfloat16, "final_state")
    # per-sequence final states individually
    for n in range(len(inp["lengths"])):
        check(sf[n], ref_s[n], torch.bfloat16, f"final_state[{n}]")
    print(f"config 2 lengths {inp['lengths']}: out {e1:.2e}, state {e2:.2e}")


@pytest.mark.parametrize("io,d", [(torch.bfloat16, 128), (torch.float32, 64)], ids=["bf16-128-tc", "f32-64"])
def test_many_short_sequences(io, d):
    """300 sequences of 0 to 40 tokens (many empty, many shorter than a chunk, ragged pairs): the
    per-sequence block slots, chunk grids and final states at a large N."""
    g = torch.Generator().manual_seed(34)
    lengths = torch.randint(0, 41, (300,), generator=g).tolist()
    inp = I.make_inputs(1, lengths=lengths, num_heads=2, d=d, io_dtype=io, seed=35, random_s0=True)
    out, sf = gpu_forward(inp)
    ref_o, ref_s = oracle_forward(inp)
    check(out, ref_o, io, "out")
    check(sf, ref_s, io, "final_state")
    # a sequence without tokens hands its initial state through unchanged
    for n, L in enumerate(lengths):
        if L == 0:
            assert torch.equal(sf[n].cpu(), inp["S0"][n].float())


@pytest.mark.slow
def test_config3_long_context_sampled_and_split():
    """1M tokens, 8 heads.  The oracle checks heads 0-1 over the first 65,536 tokens and the
    final state of heads 0-1 after all 1,048,576 tokens; the chunk-carry invariant is checked by
    running the GPU on [0, T/2) and [T/2, T) with the state carried."""
    inp = I.make_inputs(3)
    T = sum(inp["lengths"])
    d = to_dev(inp)
    out, sf = B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"])
    torch.cuda.synchronize()
    P = 65536
    ref_o, _ = oracle_forward(inp, heads=[0, 1], tokens=P)
    check(out[:P, :2], ref_o, torch.bfloat16, "out[:65536, heads 0-1]")
    _, ref_s = oracle_forward(inp, heads=[0, 1], want_out=False)
    check(sf[:, :2], ref_s, torch.bfloat16, "final_state heads 0-1")
    # split at T/2 with the state carried
    h = T // 2
    sl = lambda t, a, b: t[a:b].contiguous()
    o1, s1 = B.kda_forward(*(sl(d[x], 0, h) for x in ("q", "k", "v", "z")), d["A"], sl(d["beta"], 0, h),
                           initial_state=d["S0"])
    o2, s2 = B.kda_forward(*(sl(d[x], h, T) for x in ("q", "k", "v", "z")), d["A"], sl(d["beta"], h, T),
                           initial_state=s1)
    torch.cuda.synchronize()
    o12 = torch.cat([o1, o2])
    check(o12[:P, :2], ref_o, torch.bfloat16, "split out")
    check(s2[:, :2], ref_s, torch.bfloat16, "split final state")
    diff = (o12.float() - out.float()).abs().max().item()
    rms = out.float().pow(2).mean().sqrt().item()
    assert diff <= TOL_BF16 * rms
    del out, o1, o2, o12, d
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_config4_decode_chain():
    """256 sequences x 32 heads: 512-token varlen prefill from a random state, then 64 chained
    decode steps; the oracle runs the 576 tokens of a sample of sequences."""
    inp = I.make_inputs(4)
    N, H = 256, 32
    d = to_dev(inp)
    _, state = B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"],
                             cu_seqlens=d["cu_seqlens"], max_seqlen=512)
    dec = {k_: (v_.cuda() if torch.is_tensor(v_) else v_) for k_, v_ in inp["dec"].items()}
    outs = []
    for s in range(dec["steps"]):
        outs.append(B.kda_decode_step(dec["q"][s], dec["k"][s], dec["v"][s], dec["z"][s], d["A"], dec["beta"][s],
                                      state))
    torch.cuda.synchronize()
    outs = torch.stack(outs)  # [steps, N, H, d]
    sample = list(range(0, N, 8))  # 32 sequences
    L, S = 512, dec["steps"]
    # token-major [576 * len(sample), H, d] per sampled sequence: 512 prefill tokens then 64 decode tokens
    def seq_tokens(key):
        pre = inp[key].view(N, L, H, -1)[sample]
        de = inp["dec"][key].permute(1, 0, 2, 3)[sample]
        return torch.cat([pre, de], dim=1).reshape(len(sample) * (L + S), H, -1)
    q, k, v, z = (seq_tokens(x) for x in ("q", "k", "v", "z"))
    beta = torch.cat([inp["beta"].view(N, L, H)[sample], inp["dec"]["beta"].permute(1, 0, 2)[sample]], 1)
    beta = beta.reshape(-1, H)
    cu = torch.arange(len(sample) + 1, dtype=torch.int64) * (L + S)
    ref_o, ref_s = oracle.forward(q, k, v, z, inp["A"], beta, S0=inp["S0"][sample], cu_seqlens=cu)
    ref_dec = ref_o.reshape(len(sample), L + S, H, -1)[:, L:]          # [n, steps, H, d]
    gpu_dec = outs[:, sample].permute(1, 0, 2, 3)
    check(gpu_dec, ref_dec, torch.bfloat16, "decode outputs (64 steps)")
    check(state[sample], ref_s, torch.bfloat16, "state after 64 steps")


# ---------------------------------------------------------------- decode step alone

@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128)])
def test_decode_step_small(io, dk, dv):
    N, H = 5, 3
    inp = I.make_inputs(1, lengths=[1] * N, num_heads=H, d_k=dk, d_v=dv, io_dtype=io, seed=dk * 7 + dv)
    S = inp["S0"] * 25.0  # a state of the size a prefill leaves behind
    ref_o, ref_s = oracle.decode_step(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"], S)
    d = to_dev(inp)
    st = S.cuda()
    out = B.kda_decode_step(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], st)
    torch.cuda.synchronize()
    check(out, ref_o, io, "decode out")
    check(st, ref_s, io, "decode state")


def test_decode_after_prefill_equals_prefill_of_t_plus_1():
    T, H, dk, dv = 37, 4, 128, 128
    inp = I.make_inputs(1, lengths=[T + 1], num_heads=H, d_k=dk, d_v=dv, seed=5)
    d = to_dev(inp)
    o_full, s_full = B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"])
    _, s_pre = B.kda_forward(*(d[x][:T].contiguous() for x in ("q", "k", "v", "z")), d["A"],
                             d["beta"][:T].contiguous(), initial_state=d["S0"])
    o_dec = B.kda_decode_step(*(d[x][T:].contiguous() for x in ("q", "k", "v", "z")), d["A"],
                              d["beta"][T:].contiguous(), s_pre)
    torch.cuda.synchronize()
    check(o_dec, _f64(o_full[T:]), torch.bfloat16, "decode vs prefill")
    check(s_pre, _f64(s_full), torch.bfloat16, "state")


# ---------------------------------------------------------------- exact pins, edge cases

@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 16, 17, 100, 128])
def test_bit_exact_identity_write_read(io, T):
    """alpha = 1 (z = -1e4, A = 0 saturates the sigmoid to 0), beta = 1, q_t = k_t = distinct
    standard basis vectors, zero state: every token writes its value into an empty row and the
    query reads exactly that row back, so o_t = v_t bit for bit."""
    H, d = 2, 128
    g = torch.Generator().manual_seed(T)
    perm = torch.stack([torch.randperm(d, generator=g)[:T] for _ in range(H)], 1)  # [T, H]
    k = torch.zeros(T, H, d)
    k.scatter_(2, perm.unsqueeze(-1), 1.0)
    v = torch.randn(T, H, d, generator=g).to(io)
    z = torch.full((T, H, d), -1e4)
    A = torch.zeros(H)
    beta = torch.ones(T, H)
    out, sf = B.kda_forward(k.to(io).cuda(), k.to(io).cuda(), v.cuda(), z.to(io).cuda(), A.cuda(), beta.cuda())
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), v)


def test_beta_zero_pure_decay():
    inp = I.make_inputs(1, lengths=[70], num_heads=2, d=64, io_dtype=torch.float32, seed=11)
    inp["beta"] = torch.zeros_like(inp["beta"])
    out, sf = gpu_forward(inp)
    ref_o, ref_s = oracle_forward(inp)
    check(out, ref_o, torch.float32, "out")
    check(sf, ref_s, torch.float32, "state")


def test_gate_floor_extreme_decay_fp32():
    """Every log-decay at g_min (z large): a 16-token chunk spans exp(-80); stays finite and exact."""
    inp = I.make_inputs(1, lengths=[48], num_heads=2, d=32, io_dtype=torch.float32, seed=12)
    inp["z"] = torch.full_like(inp["z"], 60.0)
    out, sf = gpu_forward(inp)
    ref_o, ref_s = oracle_forward(inp)
    check(out, ref_o, torch.float32, "out")
    check(sf, ref_s, torch.float32, "state")


@pytest.mark.parametrize("d", [32, 64, 128])
def test_gate_floor_extreme_decay_fp32_all_widths(d):
    """The fp32 path at the decay floor for every supported width, with a ragged varlen batch."""
    inp = I.make_inputs(1, lengths=[48, 17, 0, 33], num_heads=2, d=d, io_dtype=torch.float32, seed=12 + d)
    inp["z"] = torch.full_like(inp["z"], 60.0)
    out, sf = gpu_forward(inp)
    ref_o, ref_s = oracle_forward(inp)
    check(out, ref_o, torch.float32, "out")
    check(sf, ref_s, torch.float32, "state")


def _decay_floor(inp):
    inp["z"] = torch.full_like(inp["z"], 60.0)  # sigmoid saturates: every log-decay at g_min


def _half_floor(inp):
    z = inp["z"].float()
    z[..., :64] = -1e4  # no decay at all on half the key channels ...
    z[..., 64:] = 60.0  # ... and the floor on the other half
    inp["z"] = z.to(inp["z"].dtype)


def _large_a(inp):
    inp["A"] = torch.full_like(inp["A"], 4.0)  # e^A = 55: the gate is a near step function of z


def _small_a(inp):
    inp["A"] = torch.full_like(inp["A"], -4.0)  # e^A = 0.018: every log-decay near g_min / 2


DECAY_EXTREMES = {"floor": _decay_floor, "half-floor": _half_floor, "large-A": _large_a, "small-A": _small_a}


@pytest.mark.parametrize("case", list(DECAY_EXTREMES))
@pytest.mark.parametrize("plan,seg", [("split", "0"), ("split", "2"), ("split", "6"), ("fused", "0"), ("fused", "3")],
                         ids=["split-1seg", "split-seg2", "split-seg6", "fused-1seg", "fused-seg3"])
def test_tensor_core_decay_extremes(monkeypatch, case, plan, seg):
    """The bf16 d = 128 tensor-core path at the edges of the gate's range, on both plans, unsegmented
    and with several segments: every log-decay at the floor (a 16-token chunk spans e^-80 and a
    32-token step e^-160, so K / Gamma reaches e^80 and Q Gamma e^-80 inside the hi/lo operands), no
    decay on half the key channels next to the floor on the other half, and a near-step gate
    (large A^h) or a flat one (small A^h).  Lengths 17, 33 and 250 give ragged last chunks and steps."""
    monkeypatch.setenv("KDA_TC_PLAN", plan)
    monkeypatch.setenv("KDA_SEGMENT_CHUNKS", seg)
    inp = I.make_inputs(1, lengths=[17, 33, 250, 0, 64], num_heads=3, d=128, seed=41)
    DECAY_EXTREMES[case](inp)
    out, sf = gpu_forward(inp)
    ref_o, ref_s = oracle_forward(inp)
    e1 = check(out, ref_o, torch.bfloat16, "out")
    e2 = check(sf, ref_s, torch.bfloat16, "final_state")
    print(f"{case} {plan} seg={seg}: out {e1:.2e}, state {e2:.2e}")


@pytest.mark.parametrize("g_min", [-5.0, -5.4, -8.0, -20.0])
def test_steep_decay_floor_bf16_d128(g_min):
    """The tensor-core kernels carry a 16-token chunk's Gamma and 1/Gamma as bf16 hi/lo pairs, whose
    lo parts fall below the normal fp32 range (and are flushed) for floors steeper than K3's -5, so
    such problems run on the fp32 path (pairwise decays); at -5 the tensor-core path runs.  Every
    log-decay sits at the floor here."""
    inp = I.make_inputs(1, lengths=[40, 17, 64], num_heads=2, d=128, seed=43)
    inp["z"] = torch.full_like(inp["z"], 60.0)
    out, sf = gpu_forward(inp, g_min=g_min)
    ref_o, ref_s = oracle_forward(inp, g_min=g_min)
    check(out, ref_o, torch.bfloat16, "out")
    check(sf, ref_s, torch.bfloat16, "final_state")


def test_in_place_carry_and_no_final_state():
    inp = I.make_inputs(1, lengths=[40, 24], num_heads=2, d=64, io_dtype=torch.float32, seed=13)
    d = to_dev(inp)
    ref_o, ref_s = oracle_forward(inp)
    st = d["S0"].clone()
    out, sf = B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=st,
                            cu_seqlens=d["cu_seqlens"], final_state=st)
    out2, none = B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"],
                               cu_seqlens=d["cu_seqlens"], want_final=False)
    torch.cuda.synchronize()
    assert none is None and sf.data_ptr() == st.data_ptr()
    check(st, ref_s, torch.float32, "in-place state")
    check(out, ref_o, torch.float32, "out")
    assert torch.equal(out, out2)


def test_equal_lengths_without_cu_seqlens():
    inp = I.make_inputs(1, lengths=[48, 48, 48], num_heads=2, d=64, seed=14)
    d = to_dev(inp)
    out, sf = B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"])
    torch.cuda.synchronize()
    ref_o, ref_s = oracle_forward(inp)
    check(out, ref_o, torch.bfloat16, "out")
    check(sf, ref_s, torch.bfloat16, "state")


def test_deterministic():
    inp = I.make_inputs(1, lengths=[300, 77], num_heads=4, d=128, seed=15)
    o1, s1 = gpu_forward(inp)
    o2, s2 = gpu_forward(inp)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_bad_cu_seqlens_is_reported_not_faulted():
    """Offsets that violate the descriptor are caught on the device: the bad sequence is skipped,
    the good ones are still computed, and the workspace status reports it."""
    inp = I.make_inputs(1, lengths=[32, 32, 32], num_heads=2, d=32, io_dtype=torch.float32, seed=16)
    d = to_dev(inp)
    # sequence 1 has length -12, sequence 2 (76 tokens) exceeds max_seqlen = 64
    bad = torch.tensor([0, 32, 20, 96], dtype=torch.int32, device="cuda")
    prob = B.make_problem(3, 96, 64, 2, 32, 32, torch.float32)
    ws = torch.empty(B.kda_forward_workspace_bytes(prob), dtype=torch.uint8, device="cuda")
    out = torch.full((96, 2, 32), 7.0, device="cuda")
    _, sf = B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"],
                          cu_seqlens=bad, max_seqlen=64, out=out, workspace=ws)
    assert B.kda_workspace_status(ws) == B.KDA_ERR_DEVICE_CHECK
    ref_o, _ = oracle_forward(inp)
    check(out[:32], ref_o[:32], torch.float32, "sequence 0")
    assert torch.all(out[32:] == 7.0)  # skipped sequences are not written
    # a valid call on the same workspace clears the word
    B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], cu_seqlens=d["cu_seqlens"], max_seqlen=32,
                  workspace=ws)
    assert B.kda_workspace_status(ws) == B.KDA_OK


def test_pageable_host_pointer():
    """A pageable host pointer reaching the C ABI is either rejected before any launch (GPUs that
    cannot address pageable memory) or, where the device reports it addressable (Grace-based
    GB300: coherent access to system memory), accepted and computed correctly."""
    import ctypes
    inp = I.make_inputs(1, lengths=[16], num_heads=1, d=32, seed=17)
    d = to_dev(inp)
    prob = B.make_problem(1, 16, 16, 1, 32, 32, torch.bfloat16)
    ws = torch.empty(B.kda_forward_workspace_bytes(prob), dtype=torch.uint8, device="cuda")
    out = torch.empty(16, 1, 32, dtype=torch.bfloat16, device="cuda")
    host_q = inp["q"].contiguous()  # CPU, pageable
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = B.lib().kda_forward(p(host_q), p(d["k"]), p(d["v"]), p(d["z"]), p(d["A"]), p(d["beta"]), p(d["S0"]),
                             None, p(out), None, ctypes.byref(prob), p(ws), ctypes.c_size_t(ws.numel()), None)
    torch.cuda.synchronize()
    if st == B.KDA_OK:
        ref, _ = gpu_forward(inp)
        assert torch.equal(out, ref)
    else:
        assert st == B.KDA_ERR_INVALID_ARG


# ---------------------------------------------------------------- segmented prefill

@pytest.mark.parametrize("seg", [1, 2, 3, 5])
@pytest.mark.parametrize("lengths", [[250], [100, 3, 77, 0, 160], [33]])
@pytest.mark.parametrize("plan", ["split", "fused"])
def test_segmented_prefill(monkeypatch, seg, lengths, plan):
    """Sequences cut into segments of `seg` chunks: segment summaries (S~, M), the scan of
    incoming states and the re-run from them must reproduce the unsegmented result, on both
    tensor-core plans (parallel chunk preparation + state pass, and the fused kernel)."""
    monkeypatch.setenv("KDA_SEGMENT_CHUNKS", str(seg))
    monkeypatch.setenv("KDA_TC_PLAN", plan)
    inp = I.make_inputs(1, lengths=lengths, num_heads=3, d=128, seed=seg * 100 + len(lengths))
    out, sf = gpu_forward(inp)
    ref_o, ref_s = oracle_forward(inp)
    check(out, ref_o, torch.bfloat16, "out")
    check(sf, ref_s, torch.bfloat16, "final_state")


@pytest.mark.parametrize("plan", ["split", "fused"])
def test_segmented_in_place_carry(monkeypatch, plan):
    """Final state written over the initial state with many segments: every segment must start
    from the state the call was given, although the last segment's CTAs write the final state
    into the same buffer (the first segment reads the scan's copy)."""
    monkeypatch.setenv("KDA_SEGMENT_CHUNKS", "2")
    monkeypatch.setenv("KDA_TC_PLAN", plan)
    inp = I.make_inputs(1, lengths=[250, 96, 33], num_heads=3, d=128, seed=77)
    d = to_dev(inp)
    ref_o, ref_s = oracle_forward(inp)
    for _ in range(3):
        st = d["S0"].clone()
        out, sf = B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=st,
                                cu_seqlens=d["cu_seqlens"], final_state=st)
        torch.cuda.synchronize()
        assert sf.data_ptr() == st.data_ptr()
        check(out, ref_o, torch.bfloat16, "out")
        check(st, ref_s, torch.bfloat16, "in-place state")


def test_segmented_prefill_identity_transition(monkeypatch):
    """alpha = 1, beta = 0 keeps the state constant, so every segment's transition is the identity
    and every incoming state equals the initial state: the scan must carry it exactly."""
    monkeypatch.setenv("KDA_SEGMENT_CHUNKS", "2")
    inp = I.make_inputs(1, lengths=[200], num_heads=2, d=128, seed=7)
    inp["z"] = torch.full_like(inp["z"], -1e4)
    inp["beta"] = torch.zeros_like(inp["beta"])
    out, sf = gpu_forward(inp)
    ref_o, ref_s = oracle_forward(inp)
    check(out, ref_o, torch.bfloat16, "out")
    check(sf, ref_s, torch.bfloat16, "final_state")
    assert torch.allclose(sf.cpu(), inp["S0"], rtol=0, atol=1e-6)


def test_workspace_smaller_than_the_fastest_plan():
    """A workspace below kda_forward_workspace_bytes (here the 256-byte minimum of the
    tensor-core path) makes kda_forward fall back to the fused kernel without sequence segments;
    results are unchanged."""
    inp = I.make_inputs(1, lengths=[700], num_heads=2, d=128, seed=21)
    d = to_dev(inp)
    prob = B.make_problem(1, 700, 700, 2, 128, 128, torch.bfloat16)
    assert B.kda_forward_workspace_bytes(prob) > 256  # the fastest plan segments this sequence
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    out, sf = B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"], workspace=small)
    torch.cuda.synchronize()
    ref_o, ref_s = oracle_forward(inp)
    check(out, ref_o, torch.bfloat16, "out")
    check(sf, ref_s, torch.bfloat16, "final_state")


def test_reported_workspace_runs_the_segmented_plan():
    """With exactly kda_forward_workspace_bytes of workspace, a 4096-token, 16-head prefill runs
    the split, segmented plan (operand blocks, segment summaries, scan, outputs), one launch each."""
    import cases as P
    B.kda_profile_enable(True)
    P.prefill(4096, 16, 0, torch.bfloat16)
    prof = B.kda_profile_read()
    B.kda_profile_enable(False)
    assert set(prof) == {"kda_chunk_prep_tc", "kda_state_summary_tc", "kda_seg_scan", "kda_chunk_state_tc"}
    assert all(n == 1 for n, _ in prof.values())


def test_fused_plan_when_forced(monkeypatch):
    """KDA_TC_PLAN=fused selects the fused kernel (its three segmented passes) for the same
    prefill, with a correspondingly smaller reported workspace."""
    import cases as P
    prob = B.make_problem(1, 4096, 4096, 16, 128, 128, torch.bfloat16)
    split_ws = B.kda_forward_workspace_bytes(prob)
    monkeypatch.setenv("KDA_TC_PLAN", "fused")
    assert B.kda_forward_workspace_bytes(prob) < split_ws
    B.kda_profile_enable(True)
    P.prefill(4096, 16, 0, torch.bfloat16)
    prof = B.kda_profile_read()
    B.kda_profile_enable(False)
    assert set(prof) == {"kda_seg_summary_tc", "kda_seg_scan", "kda_chunk_fwd_tc"}


# ---------------------------------------------------------------- speculative-decode state replay

def _replay_case(N, L, H, dk, dv, io, seed):
    """N windows of L drafted tokens (token t of sequence n at row n*L + t) and a snapshot of the
    size a prefill leaves behind."""
    inp = I.make_inputs(1, lengths=[L] * N, num_heads=H, d_k=dk, d_v=dv, io_dtype=io, seed=seed)
    inp["S0"] = inp["S0"] * 25.0
    return inp


def _oracle_replay(inp, accepted=None):
    return oracle.replay(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"], inp["S0"],
                         accepted=None if accepted is None else accepted.cpu().numpy())


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 32), (128, 128)])
@pytest.mark.parametrize("L", [1, 3, 8, 19])
def test_replay_small(io, dk, dv, L):
    """Outputs of the whole window and the state after each accepted prefix (0 and L included),
    with the snapshot left bit-identical."""
    N, H = 6, 3
    inp = _replay_case(N, L, H, dk, dv, io, seed=L * 131 + dk + dv)
    accepted = torch.tensor([0, L, 1 % (L + 1), L // 2, max(L - 1, 0), (3 * L) // 4], dtype=torch.int32)
    ref_o, ref_s = _oracle_replay(inp, accepted)
    d = to_dev(inp)
    snap = d["S0"].clone()
    out, s_acc = B.kda_decode_replay(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["S0"],
                                     accepted=accepted.cuda())
    torch.cuda.synchronize()
    check(out, ref_o, io, "replay window outputs")
    check(s_acc, ref_s, io, "replay accepted state")
    assert torch.equal(d["S0"], snap)
    assert torch.equal(s_acc[0], snap[0])  # nothing accepted: the snapshot, bit for bit


def test_replay_verify_then_commit_in_place():
    """The serving round: verify the window (outputs only, no state written), then advance the
    snapshot in place over the accepted prefixes (no outputs)."""
    N, L, H, dk, dv = 16, 7, 4, 128, 128
    inp = _replay_case(N, L, H, dk, dv, torch.bfloat16, seed=77)
    accepted = torch.randint(0, L + 1, (N,), generator=torch.Generator().manual_seed(7), dtype=torch.int32)
    ref_o, ref_s = _oracle_replay(inp, accepted)
    d = to_dev(inp)
    snap = d["S0"].clone()
    out, none = B.kda_decode_replay(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["S0"], want_state=False)
    assert none is None
    torch.cuda.synchronize()
    assert torch.equal(d["S0"], snap)
    check(out, ref_o, torch.bfloat16, "verify outputs")
    none, st = B.kda_decode_replay(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["S0"],
                                   accepted=accepted.cuda(), state_out=d["S0"], want_out=False)
    torch.cuda.synchronize()
    assert none is None and st.data_ptr() == d["S0"].data_ptr()
    check(st, ref_s, torch.bfloat16, "committed state")
    # the outputs do not depend on what is accepted: same bits with and without the counts (one
    # kernel: both calls also write a state), and the verify-only kernel within the tolerance
    out2, _ = B.kda_decode_replay(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], snap,
                                  accepted=accepted.cuda())
    out3, _ = B.kda_decode_replay(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], snap)
    torch.cuda.synchronize()
    assert torch.equal(out2, out3)
    check(out, _f64(out2), torch.bfloat16, "verify-only vs outputs written with a state")


def test_replay_matches_chained_decode_steps():
    """All accepted: the window equals L chained kda_decode_step calls (different kernels, the same
    recurrence), outputs and final state within the bf16 tolerance of each other."""
    N, L, H, dk, dv = 8, 5, 2, 128, 128
    inp = _replay_case(N, L, H, dk, dv, torch.bfloat16, seed=78)
    d = to_dev(inp)
    out, s_all = B.kda_decode_replay(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["S0"])
    st = d["S0"].clone()
    view = lambda x: x.view(N, L, *x.shape[1:])
    steps = []
    for t in range(L):
        steps.append(B.kda_decode_step(*(view(d[x])[:, t].contiguous() for x in ("q", "k", "v", "z")), d["A"],
                                       view(d["beta"])[:, t].contiguous(), st))
    torch.cuda.synchronize()
    chained = torch.stack(steps, 1).reshape(N * L, H, dv)
    check(out, _f64(chained), torch.bfloat16, "replay vs chained decode outputs")
    check(s_all, _f64(st), torch.bfloat16, "replay vs chained decode state")


@pytest.mark.parametrize("L", [1, 2, 5, 8])
def test_replay_verify_only(L):
    """Outputs only (no state written): bf16 with d = 128 takes the in-window chunk form; 320
    (sequence, head) units, more than the persistent grid, so CTAs walk several units."""
    N, H, dk, dv = 40, 8, 128, 128
    inp = _replay_case(N, L, H, dk, dv, torch.bfloat16, seed=90 + L)
    ref_o, _ = _oracle_replay(inp)
    d = to_dev(inp)
    snap = d["S0"].clone()
    out, none = B.kda_decode_replay(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["S0"], want_state=False)
    torch.cuda.synchronize()
    assert none is None
    assert torch.equal(d["S0"], snap)
    check(out, ref_o, torch.bfloat16, f"verify outputs, L={L}")
    # the same outputs as the recurrence kernel (which runs when a state is also written)
    out_rec, _ = B.kda_decode_replay(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["S0"])
    torch.cuda.synchronize()
    check(out, _f64(out_rec), torch.bfloat16, "chunk-form verify vs recurrence")


@pytest.mark.parametrize("decay", ["floor", "none", "mixed"])
def test_replay_verify_only_decay_extremes(decay):
    """The verify form at the ends of the gate's range over a full 8-token window: every log-decay
    at g_min (Gamma down to e^-40, 1/Gamma up to e^40 in the split bf16 operands), no decay, and
    half the key channels at each end."""
    N, L, H, d_ = 24, 8, 4, 128
    inp = _replay_case(N, L, H, d_, d_, torch.bfloat16, seed=95)
    z = inp["z"].float()
    if decay == "floor":
        z = torch.full_like(z, 60.0)
    elif decay == "none":
        z = torch.full_like(z, -60.0)
    else:
        z[..., : d_ // 2] = 60.0
        z[..., d_ // 2:] = -60.0
    inp["z"] = z.to(torch.bfloat16)
    ref_o, _ = _oracle_replay(inp)
    d = to_dev(inp)
    out, _ = B.kda_decode_replay(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["S0"], want_state=False)
    torch.cuda.synchronize()
    check(out, ref_o, torch.bfloat16, f"verify outputs, decay {decay}")


def test_replay_clamps_accepted_counts():
    N, L, H, dk, dv = 4, 6, 2, 64, 64
    inp = _replay_case(N, L, H, dk, dv, torch.float32, seed=79)
    acc = torch.tensor([-3, 0, 6, 100], dtype=torch.int32)
    _, ref_s = _oracle_replay(inp, acc.clamp(0, L))
    d = to_dev(inp)
    _, s_acc = B.kda_decode_replay(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["S0"],
                                   accepted=acc.cuda(), want_out=False)
    torch.cuda.synchronize()
    check(s_acc, ref_s, torch.float32, "clamped accepted state")


def test_replay_full_size_sampled():
    """256 sequences x 32 heads, a 7-token window (the draft length the audit's speculative-decoding
    section trains for), random accepted counts; the oracle checks a sample of 32 sequences."""
    N, L, H, d_ = 256, 7, 32, 128
    inp = _replay_case(N, L, H, d_, d_, torch.bfloat16, seed=80)
    accepted = torch.randint(0, L + 1, (N,), generator=torch.Generator().manual_seed(80), dtype=torch.int32)
    d = to_dev(inp)
    out, s_acc = B.kda_decode_replay(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["S0"],
                                     accepted=accepted.cuda())
    torch.cuda.synchronize()
    sample = list(range(3, N, 8))
    rows = torch.cat([torch.arange(n * L, (n + 1) * L) for n in sample])
    ref_o, ref_s = oracle.replay(inp["q"][rows], inp["k"][rows], inp["v"][rows], inp["z"][rows], inp["A"],
                                 inp["beta"][rows], inp["S0"][sample], accepted=accepted[sample].numpy())
    check(out[rows.cuda()], ref_o, torch.bfloat16, "full-size window outputs (sample)")
    check(s_acc[sample], ref_s, torch.bfloat16, "full-size accepted states (sample)")
    # the verify launch alone (outputs, no state), as a speculation round issues it
    out_v, _ = B.kda_decode_replay(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["S0"], want_state=False)
    torch.cuda.synchronize()
    check(out_v[rows.cuda()], ref_o, torch.bfloat16, "full-size verify outputs (sample)")


# ---------------------------------------------------------------- layer prologue / epilogue

def _layer_inputs(lengths, H, dk, dv, K, io, seed):
    g = torch.Generator().manual_seed(seed)
    T = sum(lengths)
    x = [torch.randn(T, H, d, generator=g).to(io) for d in (dk, dk, dv)]
    w = [(torch.randn(H, d, K, generator=g) * 0.7).float() for d in (dk, dk, dv)]
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32)
    return x, w, cu


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 128)])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_prologue_matches_oracle(io, dk, dv, K):
    lengths = [5, 0, 40, 16, 1, 130, 17]
    H = 3
    x, w, cu = _layer_inputs(lengths, H, dk, dv, K, io, seed=dk + dv + K)
    q, k, v = B.kda_prologue(*(t.cuda() for t in x), *(t.cuda() for t in w), cu_seqlens=cu.cuda())
    torch.cuda.synchronize()
    for name, got, xi, wi, norm in (("q", q, x[0], w[0], True), ("k", k, x[1], w[1], True), ("v", v, x[2], w[2], False)):
        ref = oracle.prologue(xi, wi, cu_seqlens=cu.numpy(), normalise=norm)
        check(got, ref, io, f"prologue {name}")


@pytest.mark.parametrize("io,d,H", [(torch.bfloat16, 128, 4), (torch.float32, 32, 9), (torch.bfloat16, 64, 5)],
                         ids=["bf16-128", "f32-32", "bf16-64"])
def test_prologue_many_tiles_per_cta(io, d, H):
    """More 64-token tiles than the persistent grid has CTAs (over 2 x 152), so CTAs walk several
    consecutive tiles: double-buffered staging, taps kept across tiles of one head group and reloaded
    at the next, and the sequence bounds carried from tile to tile across ragged sequence starts."""
    lengths = [1000, 3, 0, 2049, 64, 1, 3500, 777, 130]
    x, w, cu = _layer_inputs(lengths, H, d, d, 4, io, seed=33 + d)
    q, k, v = B.kda_prologue(*(t.cuda() for t in x), *(t.cuda() for t in w), cu_seqlens=cu.cuda())
    torch.cuda.synchronize()
    for name, got, xi, wi, norm in (("q", q, x[0], w[0], True), ("k", k, x[1], w[1], True), ("v", v, x[2], w[2], False)):
        check(got, oracle.prologue(xi, wi, cu_seqlens=cu.numpy(), normalise=norm), io, f"many-tile prologue {name}")
    # and equal lengths without offsets over the same number of tokens
    T = sum(lengths)
    N = 7
    Teq = T - T % N
    xe = [t[:Teq].contiguous() for t in x]
    qe, _, ve = B.kda_prologue(*(t.cuda() for t in xe), *(t.cuda() for t in w), num_seqs=N)
    torch.cuda.synchronize()
    cue = np.arange(N + 1) * (Teq // N)
    check(qe, oracle.prologue(xe[0], w[0], cu_seqlens=cue), io, "many-tile prologue q, equal lengths")
    check(ve, oracle.prologue(xe[2], w[2], cu_seqlens=cue, normalise=False), io, "many-tile prologue v, equal lengths")


def test_prologue_equal_lengths_without_offsets():
    H, d, K, N, Ls = 2, 128, 4, 3, 50
    x, w, _ = _layer_inputs([Ls] * N, H, d, d, K, torch.bfloat16, seed=11)
    q, k, v = B.kda_prologue(*(t.cuda() for t in x), *(t.cuda() for t in w), num_seqs=N)
    torch.cuda.synchronize()
    cu = np.arange(N + 1) * Ls
    check(q, oracle.prologue(x[0], w[0], cu_seqlens=cu), torch.bfloat16, "q")
    check(v, oracle.prologue(x[2], w[2], cu_seqlens=cu, normalise=False), torch.bfloat16, "v")


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("dv", [32, 64, 128])
def test_epilogue_matches_oracle(io, dv):
    g = torch.Generator().manual_seed(dv)
    T, H = 301, 5
    o = (torch.randn(T, H, dv, generator=g) * 3).to(io)
    gate = torch.randn(T, H, dv, generator=g).to(io)
    wt = torch.randn(dv, generator=g).float()
    ref = oracle.epilogue(o, gate, wt, 1e-5)
    y = B.kda_epilogue(o.cuda(), gate.cuda(), wt.cuda(), eps=1e-5)
    od = o.cuda()
    y2 = B.kda_epilogue(od, gate.cuda(), wt.cuda(), eps=1e-5, y=od)  # in place
    torch.cuda.synchronize()
    check(y, ref, io, "epilogue")
    assert torch.equal(y, y2)


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_layer_kernels_at_extreme_inputs(io):
    """Inputs far out on both tails of the logistic function (convolution outputs and gates near
    +-100): Swish and the gate saturate to 0 and to the identity without NaNs, and both kernels
    still match the oracle; also nine heads at d = 32, so that a warp's group of heads is split."""
    lengths, H, d, K = [90, 3, 64], 9, 32, 4
    x, w, cu = _layer_inputs(lengths, H, d, d, K, io, seed=31)
    x = [(t.float() * 40).to(io) for t in x]
    q, k, v = B.kda_prologue(*(t.cuda() for t in x), *(t.cuda() for t in w), cu_seqlens=cu.cuda())
    torch.cuda.synchronize()
    for name, got, xi, wi, norm in (("q", q, x[0], w[0], True), ("v", v, x[2], w[2], False)):
        assert torch.isfinite(got).all()
        check(got, oracle.prologue(xi, wi, cu_seqlens=cu.numpy(), normalise=norm), io, f"extreme prologue {name}")
    g = torch.Generator().manual_seed(32)
    T = sum(lengths)
    o = torch.randn(T, H, d, generator=g).to(io)
    gate = (torch.randn(T, H, d, generator=g) * 60).to(io)
    wt = torch.randn(d, generator=g).float()
    y = B.kda_epilogue(o.cuda(), gate.cuda(), wt.cuda(), eps=1e-5)
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
    check(y, oracle.epilogue(o, gate, wt, 1e-5), io, "extreme epilogue")


def test_layer_chain_prologue_forward_epilogue():
    """prologue -> kda_forward -> epilogue through the C ABI on a varlen bf16 batch.  Each stage is
    checked against the oracle run on the previous GPU stage's output: the recurrence on the GPU
    prologue's q, k, v, the epilogue on the GPU recurrence output.  (The RMSNorm rescales every row
    to unit RMS, so a row of small outputs would magnify the recurrence's own tolerance.)"""
    lengths, H, d, K = [70, 0, 33, 200], 4, 128, 4
    x, w, cu = _layer_inputs(lengths, H, d, d, K, torch.bfloat16, seed=21)
    T = sum(lengths)
    g = torch.Generator().manual_seed(22)
    z = torch.randn(T, H, d, generator=g).to(torch.bfloat16)
    A = (torch.randn(H, generator=g) * 0.5).float()
    beta = torch.sigmoid(torch.randn(T, H, generator=g)).float()
    gate = torch.randn(T, H, d, generator=g).to(torch.bfloat16)
    wt = torch.randn(d, generator=g).float()
    cud = cu.cuda()
    q, k, v = B.kda_prologue(*(t.cuda() for t in x), *(t.cuda() for t in w), cu_seqlens=cud)
    o, _ = B.kda_forward(q, k, v, z.cuda(), A.cuda(), beta.cuda(), cu_seqlens=cud)
    y = B.kda_epilogue(o, gate.cuda(), wt.cuda(), eps=1e-5)
    torch.cuda.synchronize()
    ref_o, _ = oracle.forward(q.cpu(), k.cpu(), v.cpu(), z, A, beta, cu_seqlens=cu.numpy())
    check(o, ref_o, torch.bfloat16, "layer recurrence output")
    check(y, oracle.epilogue(o.cpu(), gate, wt, 1e-5), torch.bfloat16, "layer output")


# ---------------------------------------------------------------- stage parity (fp32 path)

@pytest.mark.parametrize("dk,dv", [(32, 64), (128, 32)])
def test_stage_parity_fp32_path(dk, dv):
    """The fp32 path's per-chunk intermediates as they sit in the workspace after kda_forward --
    the in-chunk cumulative log-decay G, W = T diag(beta)(K*Gamma) and U~ = T diag(beta) V -- against
    the fp64 chunk-form restatement (itself matched to the token oracle), on a varlen batch with an
    empty sequence and a ragged last chunk."""
    from stages import chunk_reference_stages, fp32_stage_views
    lengths, H = [37, 0, 16, 50], 3
    inp = I.make_inputs(1, lengths=lengths, num_heads=H, d_k=dk, d_v=dv, io_dtype=torch.float32, seed=13 + dk)
    T, N = sum(lengths), len(lengths)
    d = to_dev(inp)
    prob = B.make_problem(N, T, max(lengths), H, dk, dv, torch.float32)
    ws = torch.zeros(B.kda_forward_workspace_bytes(prob), dtype=torch.uint8, device="cuda")
    B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"],
                  cu_seqlens=d["cu_seqlens"], max_seqlen=max(lengths), workspace=ws)
    torch.cuda.synchronize()
    G, W, Ut = fp32_stage_views(ws, T, H, dk, dv)
    g, _ = oracle.gate(inp["z"], inp["A"])
    rG, rW, rUt = chunk_reference_stages(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["S0"],
                                         inp["cu_seqlens"].numpy())
    check(G, rG, torch.float32, "stage G")
    check(W, rW, torch.float32, "stage W")
    check(Ut, rUt, torch.float32, "stage U~")
