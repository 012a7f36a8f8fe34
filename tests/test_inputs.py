"""The seeded input recipe: determinism, shapes, dtypes and the stated distributions."""
import torch

from linear_attention_recurrence_kda_gb300 import inputs as I


def test_same_seed_same_inputs_and_other_seed_differs():
    a = I.make_inputs(1, lengths=[100], num_heads=2)
    b = I.make_inputs(1, lengths=[100], num_heads=2)
    c = I.make_inputs(1, lengths=[100], num_heads=2, seed=99)
    for key in ("q", "k", "v", "z", "A", "beta", "S0"):
        assert torch.equal(a[key], b[key]), key
    assert not torch.equal(a["q"], c["q"])


def test_workload_shapes_and_dtypes():
    w0 = I.make_inputs(0)
    assert w0["q"].shape == (64, 2, 32) and w0["q"].dtype == torch.float32 and w0["S0"] is None
    w2 = I.make_inputs(2, num_heads=1, d=32)
    assert len(w2["lengths"]) == 8 and all(1024 <= n <= 16384 for n in w2["lengths"])
    assert w2["cu_seqlens"][-1].item() == sum(w2["lengths"]) == w2["q"].shape[0]
    w4 = I.make_inputs(4, num_heads=2, d=32)
    assert w4["q"].dtype == torch.bfloat16 and w4["S0"].dtype == torch.float32
    assert w4["dec"]["q"].shape == (64, 256, 2, 32) and w4["dec"]["beta"].shape == (64, 256, 2)
    assert w4["cu_seqlens"].tolist() == [512 * n for n in range(257)]


def test_distributions():
    """q, k regularised-normalised (norm one up to the fp32 rounding of the division: the 1e-6
    regulariser is far below it for 64 standard-normal channels); v, z standard normal; beta in
    (0, 1); A with standard deviation 0.5 and S0 with 0.02 (both read as standard deviations)."""
    x = I.make_inputs(1, lengths=[4096], num_heads=16, d=64, io_dtype=torch.float32)
    for key in ("q", "k"):
        n = x[key].double().norm(dim=-1)
        assert n.max() < 1.0 + 1e-6 and n.min() > 0.999
    for key in ("v", "z"):
        t = x[key].double()
        assert abs(t.mean()) < 0.01 and abs(t.std() - 1.0) < 0.01
    assert 0.0 < x["beta"].min() and x["beta"].max() < 1.0
    assert abs(x["S0"].double().std() - 0.02) < 0.001
    A = I.make_inputs(1, lengths=[1], num_heads=4096)["A"].double()
    assert abs(A.std() - 0.5) < 0.03
