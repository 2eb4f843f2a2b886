"""The polynomial exponential on the FMA pipe, the library's alternative to ex2.approx
(range reduction to f in [-1/2, 1/2] and a degree-3 polynomial for 2^f with constant term
1, fitted by csrc/gen_exp2_poly.py; the kernels measured faster with ex2.approx and use it).  The CPU tests pin the committed coefficients to
the closed form 2^f; the GPU test runs the device function through the library's
self-test entry point on a dense grid and compares it with the exact value and with the
special-function unit's ex2.approx."""

import ctypes
import math
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "exact_attention_38_gb300", "csrc", "exp2_poly.h")
REL_BOUND = 1.1e-4  # fit 1.013e-4 plus float32 evaluation, rounded up


def coefficients():
    text = open(HEADER).read()
    vals = dict(re.findall(r"kExp2PolyC(\d) = ([0-9a-fA-Fx.p+-]+)f;", text))
    return [1.0] + [float.fromhex(vals[str(k)]) for k in range(1, 4)]


def test_header_coefficients_approximate_two_to_the_f():
    c = coefficients()
    f = np.linspace(-0.5, 0.5, 200001)
    rel = np.abs((c[0] + f * (c[1] + f * (c[2] + f * c[3]))) / 2.0 ** f - 1.0)
    assert rel.max() <= 1.02e-4
    assert rel[100000] == 0.0  # f = 0 is exact
    # a minimax fit equi-oscillates: the error reaches its bound at both ends
    assert rel[0] > 0.9 * rel.max() and rel[-1] > 0.9 * rel.max()


def test_coefficients_are_the_series_to_leading_order():
    # 2^f = 1 + ln2 f + (ln2)^2/2 f^2 + ...: a plausible fit stays close to it
    c = coefficients()
    ln2 = math.log(2.0)
    assert c[0] == 1.0 and abs(c[1] - ln2) < 1e-3 and abs(c[2] - ln2 ** 2 / 2) < 5e-3


@pytest.mark.gpu
def test_device_polynomial_against_exact_and_ex2_approx(fa_lib):
    import torch

    fa = fa_lib
    rng = np.random.default_rng(0)
    grid = np.concatenate([
        np.linspace(-125.0, 8.0, 2_000_001),
        rng.uniform(-125.0, 8.0, 500_000),
        np.arange(-125, 9, dtype=np.float64),             # integers
        np.arange(-125, 8, dtype=np.float64) + 0.5,       # rounding boundaries
        np.arange(-125, 8, dtype=np.float64) + 0.4999999,
        [-125.0001, -126.0, -200.0, -1e30, -np.inf],       # below the range: exactly 0
    ]).astype(np.float32)
    x = torch.from_numpy(grid).cuda()
    yp, ym = torch.empty_like(x), torch.empty_like(x)
    st = fa.lib.fa_selftest_exp2(x.data_ptr(), yp.data_ptr(), ym.data_ptr(), x.numel(),
                                 torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    xs = grid.astype(np.float64)
    yp, ym = yp.cpu().numpy().astype(np.float64), ym.cpu().numpy().astype(np.float64)
    inside = xs >= -125.0
    exact = np.exp2(xs[inside])
    rel_p = np.abs(yp[inside] / exact - 1.0)
    rel_m = np.abs(ym[inside] / exact - 1.0)
    assert rel_p.max() <= REL_BOUND, rel_p.max()
    ints = inside & (xs == np.round(xs))
    assert np.all(yp[ints] == np.exp2(xs[ints]))  # integer exponents are exact
    assert np.all(yp[~inside] == 0.0)
    # ex2.approx on the same inputs, and the two forms against each other
    assert rel_m.max() <= 1e-6, rel_m.max()
    assert np.max(np.abs(yp[inside] / ym[inside] - 1.0)) <= REL_BOUND + 1e-6
