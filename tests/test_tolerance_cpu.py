"""The output comparison's bf16 rounding allowance, checked against torch's
own round-to-nearest-even conversion (CPU only)."""
import numpy as np
import torch

from _common import bf16_half_ulp, compare_out


def test_half_ulp_bounds_torch_rounding_and_is_reached():
    rng = np.random.default_rng(0)
    # fp32 values, so that torch rounds once (its float64 -> bf16 conversion
    # goes through fp32 and can round twice)
    x = (rng.standard_normal(200_000) * np.exp(rng.uniform(-20, 20, 200_000))).astype(np.float32)
    x = x.astype(np.float64)
    r = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    hu = bf16_half_ulp(x)
    assert np.all(np.abs(r - x) <= hu)
    # a value halfway between two bf16 neighbours is off by exactly half an ulp
    assert bf16_half_ulp(np.array([1.0]))[0] == 2.0 ** -8
    assert bf16_half_ulp(np.array([3.0]))[0] == 2.0 ** -7
    assert bf16_half_ulp(np.array([0.0]))[0] == 0.0
    mid = 1.0 + 2.0 ** -8
    assert abs(float(torch.tensor(mid, dtype=torch.float64).to(torch.bfloat16)) - mid) == 2.0 ** -8


def test_compare_out_accepts_the_correctly_rounded_result_and_rejects_a_real_error():
    rng = np.random.default_rng(1)
    exact = (rng.standard_normal(100_000) ** 3).astype(np.float32).astype(np.float64)  # heavy tail
    rounded = torch.from_numpy(exact).to(torch.bfloat16).to(torch.float64).numpy()
    compare_out(rounded, exact)
    rms = np.sqrt(np.mean(exact ** 2))
    bad = rounded.copy()
    bad[123] += 0.05 * rms
    try:
        compare_out(bad, exact)
    except AssertionError:
        return
    raise AssertionError("an error of 5% rms passed")
