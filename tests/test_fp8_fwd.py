"""FP8 (E4M3) forward against the fp64 oracle evaluated on the dequantized inputs.

Tolerance, derived from the arithmetic (the pages and the problem statement fix none for
8-bit inputs): the scores are exact products of the stored values accumulated in fp32,
so lse is held to the usual 1e-3.  P is rounded to E4M3 as P * 2^7 before the P V
product: a relative error of at most 2^-4 per term (3 mantissa bits, round to nearest),
or an absolute 2^-17 where P * 2^7 falls in E4M3's subnormal range (half the 2^-9
subnormal step, divided by the 2^7; the kernel's row sum l >= 1, so the bound holds
for the normalised P); the bf16 output adds 2^-9 relative.  So element (i, c) of O may
differ by at most
    2^-4 * sum_j P_ij |v_jc| + 2^-17 * sum_j |v_jc| + 2^-8 |O_ic| (+ 1e-5 for fp32 sums),
computed per element from the oracle's P.  The relative-norm error is also reported
against a loose 2^-4 (every term at its worst)."""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_38_gb300.inputs import make_fp8_inputs

pytestmark = pytest.mark.gpu


def _dequant(x, name):
    return x[name].to(torch.float64).numpy() * x[name + "_descale"]


def _p_rows(q, k, causal, scale, b, h, rows, lse):
    """Rows of P for the bound (the definition, only to size the tolerance)."""
    g = q.shape[2] // k.shape[2]
    s = scale * q[b, rows, h, :] @ k[b, :, h // g, :].T
    if causal:
        s = np.where(np.arange(k.shape[1])[None, :] > np.asarray(rows)[:, None], -np.inf, s)
    return np.exp(s - lse[:, None])


def _check(fa, B, N, Hq, Hkv, causal, seed, rows=None, heads=None):
    d = 128
    x = make_fp8_inputs(B, N, Hq, Hkv, d, seed=seed)
    scale = 1.0 / math.sqrt(d)
    q8, k8, v8 = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward_fp8(q8, k8, v8, x["q_descale"], x["k_descale"], x["v_descale"], causal=causal, scale=scale)
    fa.check_device_error()
    o = o.cpu().to(torch.float64).numpy()
    lse = lse.cpu().numpy().astype(np.float64)
    q, k, v = _dequant(x, "q"), _dequant(x, "k"), _dequant(x, "v")
    g = Hq // Hkv
    rows = np.arange(N) if rows is None else rows
    heads = range(Hq) if heads is None else heads
    num = den = 0.0
    for b in range(B):
        for h in heads:
            ro, rl = oracle.attn_fwd_rows(q, k, v, causal, scale, b, h, rows)
            assert np.max(np.abs(lse[b, h, rows] - rl)) <= 1e-3
            p = _p_rows(q, k, causal, scale, b, h, rows, rl)
            av = np.abs(v[b, :, h // g, :])
            tol = 2.0 ** -4 * (p @ av) + 2.0 ** -17 * av.sum(axis=0)[None, :] + 2.0 ** -8 * np.abs(ro) + 1e-5
            got = o[b, rows, h, :]
            assert np.all(np.isfinite(got))
            bad = np.abs(got - ro) > tol
            assert not bad.any(), f"b={b} h={h}: {int(bad.sum())} elements over the bound, worst excess " \
                                  f"{float(np.max(np.abs(got - ro) - tol)):.3e}"
            num += float(np.sum((got - ro) ** 2))
            den += float(np.sum(ro ** 2))
    assert math.sqrt(num / den) <= 2.0 ** -4


@pytest.mark.parametrize("N", [1, 100, 128, 129, 300, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_small(fa_lib, N, causal):
    _check(fa_lib, 2, N, 2, 2, causal, 500 + N)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_gqa(fa_lib, causal):
    _check(fa_lib, 1, 700, 4, 2, causal, 510)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_benchmark_shape_sampled(fa_lib, causal):
    rng = np.random.default_rng(520)
    rows = np.unique(np.concatenate([rng.choice(4096, 40, replace=False), [0, 4095]]))
    _check(fa_lib, 4, 4096, 16, 16, causal, 521, rows=rows, heads=(0, 11))


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_bench_workload_16k_sampled(fa_lib, causal):
    """The shape and inputs `bench.py --fp8` times: B=1, Hq=Hkv=16, N=16384, seed 3.  At
    this length each row meets 128 key blocks, so the lazy rescale (threshold 1.5 in log2
    units) and the 2^7 pre-scale of P are exercised four times longer than at N=4096."""
    rng = np.random.default_rng(530)
    rows = np.unique(np.concatenate([rng.choice(16384, 48, replace=False), [0, 16383]]))
    _check(fa_lib, 1, 16384, 16, 16, causal, 3, rows=rows, heads=(0, 7, 15))
