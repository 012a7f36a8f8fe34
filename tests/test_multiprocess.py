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
