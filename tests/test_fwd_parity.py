"""Forward parity: the CUDA path against the fp64 oracle, element by element on small
shapes (several tiles and a ragged tail), on sampled rows at full benchmark sizes,
and against closed forms that need no oracle."""

import math

import numpy as np
import pytest

import oracle
from _parity import (ATOL, LSE_ATOL, assert_close, f64, gpu_forward, make_inputs, sample_rows)

pytestmark = pytest.mark.gpu


def _check_full(fa, B, N, Hq, Hkv, d, dtype, causal, seed):
    x = make_inputs(B, N, Hq, Hkv, d, dtype=dtype, seed=seed, with_do=False)
    _, o, lse = gpu_forward(fa, x, causal)
    xo = {k: f64(v) for k, v in x.items()}
    want_o, want_lse = oracle.attn_fwd_ref(xo["q"], xo["k"], xo["v"], causal, 1.0 / math.sqrt(d))
    assert_close("O", f64(o.cpu()), want_o, ATOL[dtype], dtype)
    assert_close("lse", lse.cpu().double().numpy(), want_lse, LSE_ATOL)


def test_small_fp16_config(fa_lib):
    """B=1, H=2, N=128, d=64, fp16, seed 0, non-causal: every element of O and lse."""
    _check_full(fa_lib, 1, 128, 2, 2, 64, "fp16", False, 0)


@pytest.mark.parametrize("N", [1, 17, 127, 128, 129, 255, 256, 257, 383, 640])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_lengths(fa_lib, N, causal, d):
    _check_full(fa_lib, 2, N, 2, 2, d, "bf16", causal, 100 + N)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (6, 1), (3, 3)])
def test_gqa_and_dtypes(fa_lib, dtype, causal, Hq, Hkv):
    _check_full(fa_lib, 2, 700, Hq, Hkv, 128, dtype, causal, 7)
    _check_full(fa_lib, 1, 530, Hq, Hkv, 64, dtype, causal, 8)


def test_several_tiles_fp16_d128(fa_lib):
    _check_full(fa_lib, 1, 1536, 4, 4, 128, "fp16", True, 9)


# -------------------------------------------------- closed forms (no oracle needed)

@pytest.mark.parametrize("causal", [False, True])
def test_v_ones_gives_ones(fa_lib, causal):
    x = make_inputs(2, 300, 4, 2, 128, dtype="bf16", seed=3, with_do=False, special="v_ones")
    _, o, _ = gpu_forward(fa_lib, x, causal)
    assert_close("O", f64(o.cpu()), 1.0, 1e-6)


@pytest.mark.parametrize("causal", [False, True])
def test_q_zero_gives_visible_mean_and_log_count(fa_lib, causal):
    N = 300
    x = make_inputs(1, N, 2, 1, 64, dtype="fp16", seed=4, with_do=False, special="q_zero")
    _, o, lse = gpu_forward(fa_lib, x, causal)
    v = f64(x["v"])[0, :, 0, :]
    cnt = np.arange(1, N + 1) if causal else np.full(N, N)
    mean = np.cumsum(v, axis=0) / cnt[:, None] if causal else np.broadcast_to(v.mean(axis=0), v.shape)
    for h in range(2):
        assert_close("O", f64(o.cpu())[0, :, h, :], mean, ATOL["fp16"], "fp16")
        assert_close("lse", lse.cpu().double().numpy()[0, h], np.log(cnt), 1e-5)


def test_causal_row_zero_is_v0_and_rows_normalise(fa_lib):
    N, d = 400, 128
    x = make_inputs(1, N, 2, 2, d, dtype="bf16", seed=5, with_do=False)
    _, o, lse = gpu_forward(fa_lib, x, True)
    q, k, v = (f64(x[n])[0] for n in ("q", "k", "v"))
    og, lg = f64(o.cpu())[0], lse.cpu().double().numpy()[0]
    assert_close("O row 0", og[0], v[0], ATOL["bf16"], "bf16")
    # probabilities built from the GPU's lse sum to one on every sampled row
    for h in range(2):
        for i in sample_rows(N, 32, 1):
            s = (q[i, h] @ k[: i + 1, h].T) / math.sqrt(d)
            assert abs(np.exp(s - lg[h, i]).sum() - 1.0) < 1e-3


# -------------------------------------- full-size configurations, sampled rows

def _check_sampled(fa, B, N, Hq, Hkv, d, dtype, causal, seed, heads=2, rows=64):
    x = make_inputs(B, N, Hq, Hkv, d, dtype=dtype, seed=seed, with_do=False)
    _, o, lse = gpu_forward(fa, x, causal)
    o, lse = f64(o.cpu()), lse.cpu().double().numpy()
    xo = {k: f64(v) for k, v in x.items() if k != "do"}
    rng = np.random.default_rng(seed)
    for b in sorted(set([0, B - 1])):
        for h in rng.choice(Hq, size=min(heads, Hq), replace=False):
            r = sample_rows(N, rows, seed + int(h))
            wo, wl = oracle.attn_fwd_rows(xo["q"], xo["k"], xo["v"], causal, 1.0 / math.sqrt(d), b, int(h), r)
            assert_close(f"O b{b} h{h}", o[b, r, h], wo, ATOL[dtype], dtype)
            assert_close(f"lse b{b} h{h}", lse[b, h, r], wl, LSE_ATOL)


SWEEP = [512, 1024, 2048, 4096, 8192, 16384]


@pytest.mark.parametrize("N", SWEEP)
@pytest.mark.parametrize("causal", [False, True])
def test_sweep_d64_h32(fa_lib, N, causal):
    _check_sampled(fa_lib, 16384 // N, N, 32, 32, 64, "bf16", causal, 2)


@pytest.mark.parametrize("N", SWEEP)
@pytest.mark.parametrize("causal", [False, True])
def test_sweep_d128_h16(fa_lib, N, causal):
    _check_sampled(fa_lib, 16384 // N, N, 16, 16, 128, "bf16", causal, 3)


def test_long_context_gqa_forward(fa_lib):
    """B=1, Hq=32, Hkv=8, d=128, N=65536, causal."""
    _check_sampled(fa_lib, 1, 65536, 32, 8, 128, "bf16", True, 5, heads=2, rows=64)
