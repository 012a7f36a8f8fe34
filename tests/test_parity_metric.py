"""The parity metric's bf16 allowance is exactly the format's rounding: it excuses the rounding of
the exact value to bf16 and nothing more."""
import numpy as np
import torch

from parity import bf16_half_ulp, err_rms_rel


def test_half_ulp_bounds_round_to_nearest():
    rng = np.random.default_rng(0)
    x = rng.normal(size=100000) * np.exp(rng.uniform(-20, 20, size=100000))
    xb = torch.tensor(x).to(torch.bfloat16).double().numpy()
    hu = bf16_half_ulp(x)
    assert np.all(np.abs(xb - x) <= hu * (1 + 1e-12))
    # and it is tight: some values sit close to the bound
    assert np.max(np.abs(xb - x) / hu) > 0.99


def test_allowance_does_not_hide_computation_errors():
    rng = np.random.default_rng(1)
    ref = rng.normal(size=4096) * 0.05
    ref[7] = 0.5  # heavy tail
    exact_rounded = torch.tensor(ref).to(torch.bfloat16).double().numpy()
    assert err_rms_rel(exact_rounded, ref, stored_bf16=True) == 0.0
    assert err_rms_rel(exact_rounded, ref, stored_bf16=False) > 0.0
    wrong = exact_rounded.copy()
    wrong[100] += 0.03 * np.sqrt(np.mean(ref ** 2))
    assert err_rms_rel(wrong, ref, stored_bf16=True) > 0.02
