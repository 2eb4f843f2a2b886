"""Deterministic backward (``fa_bwd_deterministic``): parity with the fp64 oracle within
the same bounds as ``fa_bwd``, results identical bit for bit across repeated runs, and
dK / dV identical to ``fa_bwd``'s (the dK/dV kernel runs the same products in the same
order, only without its dQ path)."""

import math

import pytest
import torch

import oracle
from _parity import ATOL, assert_close, assert_relnorm, f64, make_inputs, sample_rows, to_gpu

pytestmark = pytest.mark.gpu


def _grads(fa, x, causal, deterministic):
    q, k, v, do = (to_gpu(x[n]) for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(q.shape[-1])
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    g = fa.backward(do, q, k, v, o, lse, causal=causal, scale=scale, deterministic=deterministic)
    fa.check_device_error()
    return g


@pytest.mark.parametrize("N", [1, 63, 128, 129, 300, 513])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_parity_ragged(fa_lib, N, causal, d):
    x = make_inputs(2, N, 2, 2, d, dtype="bf16", seed=300 + N)
    dq, dk, dv = _grads(fa_lib, x, causal, True)
    xo = {n: f64(t) for n, t in x.items()}
    ref = oracle.attn_bwd_ref(xo["q"], xo["k"], xo["v"], xo["do"], causal, 1.0 / math.sqrt(d))
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close(name, f64(got.cpu()), ref[name], ATOL["bf16"], "bf16")
        assert_relnorm(name, f64(got.cpu()), ref[name])


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
def test_parity_gqa(fa_lib, dtype, causal):
    x = make_inputs(2, 700, 6, 2, 128, dtype=dtype, seed=310)
    dq, dk, dv = _grads(fa_lib, x, causal, True)
    xo = {n: f64(t) for n, t in x.items()}
    ref = oracle.attn_bwd_ref(xo["q"], xo["k"], xo["v"], xo["do"], causal, 1.0 / math.sqrt(128))
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close(name, f64(got.cpu()), ref[name], ATOL[dtype], dtype)
        assert_relnorm(name, f64(got.cpu()), ref[name])


@pytest.mark.parametrize("causal", [False, True])
def test_bitwise_repeatable_and_dkdv_match(fa_lib, causal):
    """Benchmark-shaped (16k tokens, 4 x 4096): five runs give identical bits; dK and dV
    equal fa_bwd's bit for bit; dQ agrees with the oracle on sampled rows."""
    fa = fa_lib
    B, N, H, d = 4, 4096, 16, 128
    x = make_inputs(B, N, H, H, d, dtype="bf16", seed=311)
    q, k, v, do = (to_gpu(x[n]) for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    runs = [fa.backward(do, q, k, v, o, lse, causal=causal, scale=scale, deterministic=True) for _ in range(5)]
    fa.check_device_error()
    for r in runs[1:]:
        for a, b_ in zip(runs[0], r):
            assert torch.equal(a, b_)
    _, dk_nd, dv_nd = fa.backward(do, q, k, v, o, lse, causal=causal, scale=scale)
    fa.check_device_error()
    assert torch.equal(runs[0][1], dk_nd) and torch.equal(runs[0][2], dv_nd)
    rows = sample_rows(N, 48, 312)
    xo = {n: f64(t) for n, t in x.items()}
    for h in (0, 9):
        ref = oracle.attn_bwd_dq_rows(xo["q"], xo["k"], xo["v"], xo["do"], causal, scale, 1, h, rows)
        got = f64(runs[0][0][1, rows, h, :].cpu())
        assert_close("dq", got, ref, ATOL["bf16"], "bf16")


@pytest.mark.parametrize("d,H,causal", [(128, 16, False), (128, 16, True), (64, 32, False)])
def test_bench_workload_16k_sampled(fa_lib, d, H, causal):
    """The `--deterministic` bench workload (B=1, N=16384): dQ on sampled rows of two heads
    against the oracle (the K / V rings wrap many times per CTA here), dK and dV equal to
    fa_bwd's bit for bit."""
    fa = fa_lib
    B, N = 1, 16384
    x = make_inputs(B, N, H, H, d, dtype="bf16", seed=320 + d + causal)
    q, k, v, do = (to_gpu(x[n]) for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(do, q, k, v, o, lse, causal=causal, scale=scale, deterministic=True)
    _, dk_nd, dv_nd = fa.backward(do, q, k, v, o, lse, causal=causal, scale=scale)
    fa.check_device_error()
    assert torch.equal(dk, dk_nd) and torch.equal(dv, dv_nd)
    dq_host = dq.cpu()
    del dq, dk, dv, dk_nd, dv_nd, o, lse
    torch.cuda.empty_cache()
    xo = {n: f64(t) for n, t in x.items()}
    for h in (0, H - 1):
        rows = sample_rows(N, 40, 330 + h)
        ref = oracle.attn_bwd_dq_rows(xo["q"], xo["k"], xo["v"], xo["do"], causal, scale, 0, h, rows)
        assert_close(f"dq h{h}", f64(dq_host[0, rows, h, :]), ref, ATOL["bf16"], "bf16")
