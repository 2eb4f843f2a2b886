"""The d=64 forward above the persistent range (fixed length, one CTA per 256 queries).

Checked against the oracle element by element: ragged lengths around the 128-key block, the
128-row tile and the 256-query unit, both masks, bf16 and fp16, GQA, several batches; and,
sampled, the 16k-token sweep shape with many CTAs per SM."""

import math

import pytest

import oracle
from _parity import ATOL, LSE_ATOL, assert_close, f64, gpu_forward, make_inputs, sample_rows

pytestmark = pytest.mark.gpu


def _check_full(fa, B, N, Hq, Hkv, dtype, causal, seed):
    x = make_inputs(B, N, Hq, Hkv, 64, dtype=dtype, seed=seed, with_do=False)
    _, o, lse = gpu_forward(fa, x, causal)
    xo = {k: f64(v) for k, v in x.items()}
    want_o, want_lse = oracle.attn_fwd_ref(xo["q"], xo["k"], xo["v"], causal, 1.0 / math.sqrt(64))
    assert_close("O", f64(o.cpu()), want_o, ATOL[dtype], dtype)
    assert_close("lse", lse.cpu().double().numpy(), want_lse, LSE_ATOL)


@pytest.mark.parametrize("N", [513, 577, 640, 1000, 1025, 1100, 1536, 2049])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(fa_lib, N, causal):
    if causal and N <= 1024:
        pytest.skip("the causal forward runs the persistent kernel up to N=1024")
    _check_full(fa_lib, 2, N, 2, 2, "bf16", causal, 600 + N)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (6, 1), (4, 4)])
def test_gqa_fp16(fa_lib, causal, Hq, Hkv):
    _check_full(fa_lib, 3, 1300, Hq, Hkv, "fp16", causal, 650 + Hq + Hkv)


@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_sampled(fa_lib, causal):
    """B=1, H=32, N=16384 (the d=64 sweep shape): 1024 CTAs, sampled rows of two heads."""
    B, N, H = 1, 16384, 32
    x = make_inputs(B, N, H, H, 64, dtype="bf16", seed=660 + causal, with_do=False)
    _, o, lse = gpu_forward(fa_lib, x, causal)
    o = f64(o.cpu())
    lse = lse.cpu().double().numpy()
    xo = {k: f64(v) for k, v in x.items()}
    rows = sample_rows(N, 48, 661 + causal)
    for h in (0, H - 1):
        want_o, want_lse = oracle.attn_fwd_rows(xo["q"], xo["k"], xo["v"], causal, 1.0 / math.sqrt(64), 0, h, rows)
        assert_close(f"O h{h}", o[0, rows, h], want_o, ATOL["bf16"], "bf16")
        assert_close(f"lse h{h}", lse[0, h, rows], want_lse, LSE_ATOL)
