"""The output tolerance's allowance for the bf16 output format, checked on CPU against
torch's own round-to-nearest-even conversion to bfloat16."""
import numpy as np
import torch

from helpers import bf16_half_ulp, check_output


def test_half_ulp_bounds_bf16_rounding_and_is_attained():
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(200000) * 10.0 ** rng.integers(-30, 30, 200000),
                        [1.0, -1.0, 2.0 ** -126, 3.0e38]])
    r = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    err = np.abs(r - v)
    assert np.all(err <= bf16_half_ulp(r) * (1 + 1e-12))
    # tight: some values sit close to a midpoint (error near half an ulp)
    assert np.max(err / bf16_half_ulp(r)) > 0.99


def test_exactly_rounded_reference_passes_and_a_real_error_fails():
    rng = np.random.default_rng(6)
    ref = rng.standard_normal((8, 512)) * np.where(rng.random((8, 512)) < 0.01, 8.0, 1.0)
    rounded = torch.from_numpy(ref).to(torch.bfloat16).to(torch.float64).numpy()
    assert check_output(rounded, ref) <= 1e-12
    wrong = rounded.copy()
    wrong[3, 7] += 0.05 * np.sqrt(np.mean(ref ** 2))
    try:
        check_output(wrong, ref)
    except AssertionError:
        return
    raise AssertionError("an error of 5e-2 RMS passed the check")
