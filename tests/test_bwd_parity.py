"""Backward parity: dQ, dK, dV of the CUDA path against the fp64 oracle (max-abs and
relative-norm bounds), exhaustively on small shapes and on sampled rows at the
benchmark sizes, plus identities that hold at any size."""

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from _parity import ATOL, assert_close, assert_relnorm, f64, make_inputs, sample_rows, to_gpu

pytestmark = pytest.mark.gpu


def gpu_fwd_bwd(fa, x, causal):
    q, k, v, do = (to_gpu(x[n]) for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(q.shape[-1])
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(do, q, k, v, o, lse, causal=causal, scale=scale)
    fa.check_device_error()
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


def _check_full(fa, B, N, Hq, Hkv, d, dtype, causal, seed):
    x = make_inputs(B, N, Hq, Hkv, d, dtype=dtype, seed=seed)
    g = gpu_fwd_bwd(fa, x, causal)
    xo = {k: f64(v) for k, v in x.items()}
    ref = oracle.attn_bwd_ref(xo["q"], xo["k"], xo["v"], xo["do"], causal, 1.0 / math.sqrt(d))
    for name in ("dq", "dk", "dv"):
        got = f64(g[name].cpu())
        assert_close(name, got, ref[name], ATOL[dtype], dtype)
        assert_relnorm(name, got, ref[name])


def test_small_fp16(fa_lib):
    _check_full(fa_lib, 1, 128, 2, 2, 64, "fp16", False, 0)


@pytest.mark.parametrize("N", [1, 17, 63, 64, 65, 127, 128, 129, 255, 300, 513])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_lengths(fa_lib, N, causal, d):
    _check_full(fa_lib, 2, N, 2, 2, d, "bf16", causal, 200 + N)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (6, 1), (3, 3)])
def test_gqa_and_dtypes(fa_lib, dtype, causal, Hq, Hkv):
    _check_full(fa_lib, 2, 700, Hq, Hkv, 128, dtype, causal, 17)
    _check_full(fa_lib, 1, 530, Hq, Hkv, 64, dtype, causal, 18)


def test_several_blocks_fp16_d128(fa_lib):
    _check_full(fa_lib, 1, 1536, 4, 2, 128, "fp16", True, 19)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_sum_identities(fa_lib, causal):
    """sum_j dK_j = 0 (each row of dS sums to 0) and sum_j dV_j = sum over the group of sum_i dO_i."""
    B, N, Hq, Hkv, d = 2, 777, 4, 2, 128
    x = make_inputs(B, N, Hq, Hkv, d, dtype="bf16", seed=21)
    g = gpu_fwd_bwd(fa_lib, x, causal)
    dk, dv = f64(g["dk"].cpu()), f64(g["dv"].cpu())
    do = f64(x["do"])
    # Every dK_j / dV_j carries relative rounding of order 2^-9 from its 16-bit inputs
    # (P, dS) and its 16-bit output, so a sum over j may drift by up to about
    # 2^-8 * sum_j |.|; a wrong gradient misses these identities by O(sqrt(N)).
    tol_k = 2 ** -8 * np.abs(dk).sum(axis=1)
    assert np.all(np.abs(dk.sum(axis=1)) <= tol_k)
    want = do.sum(axis=1).reshape(B, Hkv, Hq // Hkv, d).sum(axis=2)
    tol_v = 2 ** -8 * np.abs(dv).sum(axis=1)
    assert np.all(np.abs(dv.sum(axis=1) - want) <= tol_v)


def test_repeated_calls_are_consistent(fa_lib):
    """The workspace is re-initialised by every call (dQ accumulates from zero)."""
    x = make_inputs(1, 300, 4, 2, 64, dtype="bf16", seed=22)
    a = gpu_fwd_bwd(fa_lib, x, True)
    b = gpu_fwd_bwd(fa_lib, x, True)
    for n in ("dq", "dk", "dv"):
        diff = (a[n].float() - b[n].float()).abs().max().item()
        assert diff <= 2 * ATOL["bf16"], (n, diff)


# ------------------------------------------------ full-size configurations, sampled

def _kv_rows(xo, causal, scale, b, hk, kr):
    """Oracle dK/dV rows of key/value head hk, as the sum of one oracle call per query
    head of its group (each call sees that head alone, so the group sum is the sum of
    the calls), run on threads: numpy releases the interpreter lock in its products
    and exponentials."""
    G = xo["q"].shape[2] // xo["k"].shape[2]

    def one(h):
        return oracle.attn_bwd_kv_rows(xo["q"][:, :, h:h + 1], xo["k"][:, :, hk:hk + 1], xo["v"][:, :, hk:hk + 1],
                                       xo["do"][:, :, h:h + 1], causal, scale, b, 0, kr)

    with ThreadPoolExecutor(max_workers=min(G, 4)) as ex:
        parts = list(ex.map(one, range(hk * G, (hk + 1) * G)))
    return sum(p[0] for p in parts), sum(p[1] for p in parts)


def _check_sampled(fa, B, N, Hq, Hkv, d, dtype, causal, seed, heads=2, rows=64, key_rows=None):
    """dQ on sampled query rows of `heads` heads and dK/dV on sampled key rows of one
    key/value head, in the first and the last batch (the tensor maps' batch offset)."""
    x = make_inputs(B, N, Hq, Hkv, d, dtype=dtype, seed=seed)
    g = gpu_fwd_bwd(fa, x, causal)
    dq, dk, dv = (f64(g[n].cpu()) for n in ("dq", "dk", "dv"))
    del g
    torch.cuda.empty_cache()
    xo = {k: f64(v) for k, v in x.items()}
    scale = 1.0 / math.sqrt(d)
    rng = np.random.default_rng(seed)
    kr = sample_rows(N, rows, seed + 99) if key_rows is None else np.asarray(key_rows)
    for b in sorted({0, B - 1}):
        for h in rng.choice(Hq, size=min(heads, Hq), replace=False):
            r = sample_rows(N, rows, seed + int(h) + 7 * b)
            want = oracle.attn_bwd_dq_rows(xo["q"], xo["k"], xo["v"], xo["do"], causal, scale, b, int(h), r)
            assert_close(f"dq b{b} h{h}", dq[b, r, h], want, ATOL[dtype], dtype)
            assert_relnorm(f"dq b{b} h{h}", dq[b, r, h], want)
        hk = int(rng.integers(Hkv))
        wk, wv = _kv_rows(xo, causal, scale, b, hk, kr)
        assert_close(f"dk b{b} hkv{hk}", dk[b, kr, hk], wk, ATOL[dtype], dtype)
        assert_relnorm(f"dk b{b} hkv{hk}", dk[b, kr, hk], wk)
        assert_close(f"dv b{b} hkv{hk}", dv[b, kr, hk], wv, ATOL[dtype], dtype)
        assert_relnorm(f"dv b{b} hkv{hk}", dv[b, kr, hk], wv)


@pytest.mark.parametrize("N", [512, 1024, 2048, 4096, 8192, 16384])
@pytest.mark.parametrize("causal", [False, True])
def test_sweep_d128_h16(fa_lib, N, causal):
    _check_sampled(fa_lib, 16384 // N, N, 16, 16, 128, "bf16", causal, 4)


@pytest.mark.parametrize("causal", [False, True])
def test_sweep_d64_h32_16k(fa_lib, causal):
    _check_sampled(fa_lib, 1, 16384, 32, 32, 64, "bf16", causal, 2)


@pytest.mark.slow
def test_long_context_gqa_backward(fa_lib):
    """B=1, Hq=32, Hkv=8, d=128, N=65536, causal.  dK/dV on 64 key rows drawn uniformly
    over all positions plus 8 below 2048 (whose column of P spans every query of the
    4-head group, the longest walk of the kernel), and the first and last keys."""
    N = 65536
    rng = np.random.default_rng(55)
    kr = np.unique(np.concatenate([rng.choice(N, 64, replace=False), rng.choice(2048, 8, replace=False), [0, N - 1]]))
    _check_sampled(fa_lib, 1, N, 32, 8, 128, "bf16", True, 5, heads=2, rows=64, key_rows=kr)
