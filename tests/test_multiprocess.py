"""The multi-rank path on the CPU: two gloo ranks shard a varlen batch by sequences, each runs the
recurrence on its own shard (the oracle stands in for the kernels here), and the gathered result
must equal the whole batch computed in one process -- sequences never interact (Equation 1 of
"Kimi K3: the paper and proofs side by side", section 2.1.1, acts on one sequence's state)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from linear_attention_recurrence_kda_gb300 import inputs as I  # noqa: E402
from linear_attention_recurrence_kda_gb300.sharding import local_batch, split_sequences  # noqa: E402

LENGTHS = [40, 7, 0, 65, 23, 1]
HEADS, D = 2, 16


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _batch():
    return I.make_inputs(2, lengths=LENGTHS, num_heads=HEADS, d=D, io_dtype=torch.float32, seed=7)


def _rank_main(rank, world, port, out_path):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from linear_attention_recurrence_kda_gb300 import sharding as SH

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = _batch()
        cu = inp["cu_seqlens"].tolist()
        lo, hi = SH.split_sequences(LENGTHS, world)[rank]
        t_lo, t_hi, lcu = SH.local_batch(cu, lo, hi)
        sl = slice(t_lo, t_hi)
        if hi > lo:
            o, s = oracle.forward(inp["q"][sl], inp["k"][sl], inp["v"][sl], inp["z"][sl], inp["A"], inp["beta"][sl],
                                  S0=inp["S0"][lo:hi], cu_seqlens=np.asarray(lcu, dtype=np.int64), threads=1)
        else:
            o = np.zeros((0, HEADS, D))
            s = np.zeros((0, HEADS, D, D))
        go = SH.gather_rows(torch.from_numpy(np.ascontiguousarray(o)))
        gs = SH.gather_rows(torch.from_numpy(np.ascontiguousarray(s)))
        mx = SH.max_over_ranks(1.5 + rank)
        tot = SH.sum_over_ranks(float(t_hi - t_lo))
        if rank == 0:
            torch.save({"o": go, "s": gs, "max": mx, "sum": tot}, out_path)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_split_sequences_covers_in_order_and_balances():
    for lengths in ([40, 7, 0, 65, 23, 1], [5] * 9, [1000, 1, 1, 1], [0, 0, 0], [3]):
        total = sum(lengths)
        for world in (1, 2, 3, 4, 8):
            parts = split_sequences(lengths, world)
            assert len(parts) == world
            assert parts[0][0] == 0 and parts[-1][1] == len(lengths)
            for (a, b), (c, d) in zip(parts, parts[1:]):
                assert b == c and a <= b
            # each rank is within one sequence of the ideal share
            longest = max(lengths) if lengths else 0
            for lo, hi in parts:
                assert sum(lengths[lo:hi]) <= total / world + longest
    with pytest.raises(ValueError):
        split_sequences([1, 2], 0)
    with pytest.raises(ValueError):
        split_sequences([1, -2], 2)


def test_local_batch_rebases_cu_seqlens():
    cu = [0, 40, 47, 47, 112, 135, 136]
    assert local_batch(cu, 2, 5) == (47, 135, [0, 0, 65, 88])
    assert local_batch(cu, 3, 3) == (47, 47, [0])
    with pytest.raises(ValueError):
        local_batch(cu, 4, 7)


def test_two_gloo_ranks_reproduce_the_single_process_batch(tmp_path):
    import oracle

    world = 2
    out_path = str(tmp_path / "rank0.pt")
    mp.get_context("spawn")
    mp.spawn(_rank_main, args=(world, _free_port(), out_path), nprocs=world, join=True)
    got = torch.load(out_path)
    inp = _batch()
    o, s = oracle.forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"], S0=inp["S0"],
                          cu_seqlens=inp["cu_seqlens"], threads=1)
    # the same fp64 arithmetic on the same sequences: identical, bit for bit
    assert np.array_equal(got["o"].numpy(), o)
    assert np.array_equal(got["s"].numpy(), s)
    assert got["max"] == 2.5
    assert got["sum"] == float(sum(LENGTHS))


# ---------------------------------------------------------------- context-parallel prefill (KCP)

KCP_T, KCP_N, KCP_H, KCP_DK, KCP_DV = 24, 2, 2, 8, 6


class OracleKernels:
    """The three per-rank KCP steps computed by the fp64 oracle (the CPU stand-in for the kernels):
    S~ is a range's end state from zero; M its end state from the identity with every value zero
    (d_v = d_k); the scan applies the maps of the ranks before this one, in order."""

    @staticmethod
    def summary(q, k, v, z, A, beta, num_seqs):
        import oracle
        T, H, dk = k.shape
        cu = np.arange(num_seqs + 1) * (T // num_seqs)
        _, St = oracle.forward(q, k, v, z, A, beta, cu_seqlens=cu, threads=1)
        eye = np.broadcast_to(np.eye(dk), (num_seqs, H, dk, dk)).copy()
        _, M = oracle.forward(q, k, torch.zeros(T, H, dk, dtype=v.dtype), z, A, beta, S0=eye, cu_seqlens=cu, threads=1)
        return torch.from_numpy(M), torch.from_numpy(St)

    @staticmethod
    def scan(Ms, Ss, S0, count):
        S = torch.zeros_like(Ss[0]) if S0 is None else S0.double().clone()
        for i in range(count):
            S = Ms[i] @ S + Ss[i]
        return S

    @staticmethod
    def forward(q, k, v, z, A, beta, S_in, num_seqs):
        import oracle
        T = k.shape[0]
        cu = np.arange(num_seqs + 1) * (T // num_seqs)
        o, s = oracle.forward(q, k, v, z, A, beta, S0=S_in, cu_seqlens=cu, threads=1)
        return torch.from_numpy(o), torch.from_numpy(s)


def _kcp_batch():
    return I.make_inputs(2, lengths=[KCP_T] * KCP_N, num_heads=KCP_H, d_k=KCP_DK, d_v=KCP_DV,
                         io_dtype=torch.float32, seed=11)


def _kcp_rank_main(rank, world, port, out_path):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from linear_attention_recurrence_kda_gb300 import context_parallel as CP

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = _kcp_batch()
        Tr = KCP_T // world
        rows = torch.cat([torch.arange(n * KCP_T + rank * Tr, n * KCP_T + (rank + 1) * Tr) for n in range(KCP_N)])
        local = {x: inp[x][rows] for x in ("q", "k", "v", "z", "beta")}
        o, s = CP.kcp_forward(local["q"], local["k"], local["v"], local["z"], inp["A"], local["beta"],
                              initial_state=inp["S0"], num_seqs=KCP_N, kernels=OracleKernels)
        parts = [torch.empty_like(o) for _ in range(world)]
        dist.all_gather(parts, o.contiguous())
        if rank == world - 1:
            torch.save({"o": torch.stack(parts), "s": s}, out_path)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_kcp_ranks_reproduce_the_unsplit_sequences(tmp_path, world):
    """Each sequence split by tokens over 2 or 3 gloo ranks: per-rank summaries (M, S~), one
    all-gather, the prefix scan and the re-run from the scanned state give the outputs and final
    state of the unsplit run."""
    import oracle

    out_path = str(tmp_path / "last.pt")
    mp.spawn(_kcp_rank_main, args=(world, _free_port(), out_path), nprocs=world, join=True)
    got = torch.load(out_path)
    inp = _kcp_batch()
    o, s = oracle.forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"], S0=inp["S0"],
                          cu_seqlens=inp["cu_seqlens"], threads=1)
    Tr = KCP_T // world
    ref = o.reshape(KCP_N, world, Tr, KCP_H, KCP_DV).transpose(1, 0, 2, 3, 4)  # [rank, n, t, H, dv]
    got_o = got["o"].numpy().reshape(world, KCP_N, Tr, KCP_H, KCP_DV)
    np.testing.assert_allclose(got_o, ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(got["s"].numpy(), s, rtol=1e-10, atol=1e-12)


def test_kcp_detects_a_wrong_scan_order():
    """The scan must apply the earlier ranks' maps first: composing them in the reverse order (a
    plausible mistake) gives a different incoming state for the third rank."""
    inp = _kcp_batch()
    Tr = KCP_T // 3
    summaries = []
    for r in range(3):
        rows = torch.cat([torch.arange(n * KCP_T + r * Tr, n * KCP_T + (r + 1) * Tr) for n in range(KCP_N)])
        summaries.append(OracleKernels.summary(*(inp[x][rows] for x in ("q", "k", "v", "z")), inp["A"],
                                               inp["beta"][rows], KCP_N))
    Ms = torch.stack([m for m, _ in summaries])
    Ss = torch.stack([s for _, s in summaries])
    right = OracleKernels.scan(Ms, Ss, inp["S0"], 2)
    wrong = OracleKernels.scan(Ms.flip(0)[1:], Ss.flip(0)[1:], inp["S0"], 2)
    assert not torch.allclose(right, wrong)
