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


# ---- per-block descales (fa_fwd_fp8_blockscaled)
#
# Same bound as above, with two changes that follow from the kernel's arithmetic: the
# scores take the query block's and key block's descales (still exact products of stored
# values, accumulated in fp32), and P is rounded to E4M3 as P * 2^7 * v_j / v_max, so its
# subnormal floor, 2^-17 / (v_j / v_max) per unit of P, times the dequantized |v| =
# |v8| v_j gives 2^-17 v_max sum_j |v8_jc| (v_max taken over all blocks of the key/value
# head, at least the kernel's per-tile maximum).


def _dequant_blocks(x, name):
    t = x[name].to(torch.float64)  # [B, N, H, d]
    ds = x[name + "_descale"].to(torch.float64)  # [B, H, nb]
    N = t.shape[1]
    f = ds.permute(0, 2, 1).repeat_interleave(128, dim=1)[:, :N, :, None]  # [B, N, H, 1]
    return (t * f).numpy(), t.numpy()


def _check_block(fa, B, N, Hq, Hkv, causal, seed, rows=None, heads=None, spread=4.0):
    from exact_attention_38_gb300.inputs import make_fp8_block_inputs

    d = 128
    x = make_fp8_block_inputs(B, N, Hq, Hkv, d, seed=seed, spread=spread)
    scale = 1.0 / math.sqrt(d)
    q8, k8, v8 = (x[n].cuda() for n in ("q", "k", "v"))
    qd, kd, vd = (x[n + "_descale"].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward_fp8_blockscaled(q8, k8, v8, qd, kd, vd, causal=causal, scale=scale)
    fa.check_device_error()
    o = o.cpu().to(torch.float64).numpy()
    lse = lse.cpu().numpy().astype(np.float64)
    q, _ = _dequant_blocks(x, "q")
    k, _ = _dequant_blocks(x, "k")
    v, v8n = _dequant_blocks(x, "v")
    vmax = x["v_descale"].to(torch.float64).amax(dim=2).numpy()  # [B, Hkv]
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
            av8 = np.abs(v8n[b, :, h // g, :])
            tol = (2.0 ** -4 * (p @ av) + 2.0 ** -17 * vmax[b, h // g] * av8.sum(axis=0)[None, :]
                   + 2.0 ** -8 * np.abs(ro) + 1e-5)
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
def test_fp8_blockscaled_small(fa_lib, N, causal):
    _check_block(fa_lib, 2, N, 2, 2, causal, 540 + N)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_blockscaled_gqa_wide_spread(fa_lib, causal):
    """GQA 4:2 with block descales spread over [1/64, 64] (the V factor v_j / v_max reaches
    2^-12, deep into the kernel's E4M3 subnormal handling of P)."""
    _check_block(fa_lib, 1, 700, 4, 2, causal, 550, spread=64.0)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_blockscaled_4096_sampled(fa_lib, causal):
    rng = np.random.default_rng(560)
    rows = np.unique(np.concatenate([rng.choice(4096, 40, replace=False), [0, 4095]]))
    _check_block(fa_lib, 2, 4096, 8, 8, causal, 561, rows=rows, heads=(0, 5))


def test_fp8_blockscaled_equal_blocks_match_per_tensor(fa_lib):
    """With every block's descale equal to a per-tensor descale the block-scaled kernel is
    the per-tensor one up to the rounding of the score multiplier (scale x descales folded
    in another order): both stay within the bound above; their outputs differ by at most
    one E4M3 step of P per term, here checked as a small relative norm."""
    from exact_attention_38_gb300.inputs import make_fp8_inputs

    B, N, H, d = 1, 1000, 4, 128
    x = make_fp8_inputs(B, N, H, H, d, seed=570)
    nb = (N + 127) // 128
    q8, k8, v8 = (x[n].cuda() for n in ("q", "k", "v"))
    bs = {n: torch.full((B, H, nb), x[n + "_descale"], dtype=torch.float32, device="cuda") for n in ("q", "k", "v")}
    o1, l1 = fa_lib.forward_fp8(q8, k8, v8, x["q_descale"], x["k_descale"], x["v_descale"], causal=True)
    o2, l2 = fa_lib.forward_fp8_blockscaled(q8, k8, v8, bs["q"], bs["k"], bs["v"], causal=True)
    fa_lib.check_device_error()
    a, c = o1.float(), o2.float()
    assert float((a - c).norm() / a.norm()) <= 2.0 ** -6
    assert float((l1 - l2).abs().max()) <= 1e-4
