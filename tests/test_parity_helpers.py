"""The tolerance the GPU parity tests apply, pinned on the CPU: half a unit in the last
place of the 16-bit output format bounds the error of rounding to that format, and is
reached (so the bound is not looser than one rounding)."""

import numpy as np
import pytest
import torch

from _parity import ATOL, FLAT_EXCESS, assert_close, half_ulp


@pytest.mark.parametrize("dtype,tdt", [("bf16", torch.bfloat16), ("fp16", torch.float16)])
def test_half_ulp_bounds_round_to_nearest(dtype, tdt):
    g = torch.Generator().manual_seed(0)
    x = (torch.randn(200000, generator=g, dtype=torch.float64) * torch.exp2(
        torch.randint(-12, 8, (200000,), generator=g).double())).float().double()
    # (x is an fp32 value, so the conversion below is one rounding; from fp64 torch
    # rounds through fp32 first)
    r = x.float().to(tdt).double()
    err = (r - x).abs().numpy()
    hu = half_ulp(x.numpy(), dtype)
    assert np.all(err <= hu)
    # at the midpoint between two representable numbers the bound is attained
    one = 1.0 + half_ulp(1.0, dtype)
    assert float(abs(torch.tensor(one, dtype=torch.float64).to(tdt).double() - one)) == pytest.approx(half_ulp(1.0, dtype))


def test_half_ulp_values():
    assert half_ulp(1.0, "bf16") == 2.0 ** -8
    assert half_ulp(1.99, "bf16") == 2.0 ** -8
    assert half_ulp(5.1, "bf16") == 2.0 ** -6
    assert half_ulp(-8.0, "bf16") == 2.0 ** -5
    assert half_ulp(1.0, "fp16") == 2.0 ** -11
    assert half_ulp(0.0, "fp16") == 2.0 ** -25      # subnormal step 2^-24
    assert half_ulp(1e-9, "fp16") == 2.0 ** -25


def test_assert_close_bound():
    n0 = len(FLAT_EXCESS)
    # bf16 at |ref| = 5: flat 1.6e-2 plus 2^-6
    assert_close("x", [5.0 + 0.016 + 2.0 ** -6 - 1e-9], [5.0], ATOL["bf16"], "bf16")
    with pytest.raises(AssertionError):
        assert_close("x", [5.0 + 0.016 + 2.0 ** -6 + 1e-6], [5.0], ATOL["bf16"], "bf16")
    with pytest.raises(AssertionError):
        assert_close("x", [0.5 + 0.0161 + 2.0 ** -9 + 1e-6], [0.5], ATOL["bf16"], "bf16")
    with pytest.raises(AssertionError):
        assert_close("x", [float("nan")], [0.0], 1.0)
    del FLAT_EXCESS[n0:]  # these are not parity results
