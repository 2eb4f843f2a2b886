"""The backward's wave-tail split: in the one-CTA-per-key-block grid (fixed length,
non-causal, N above the persistent kernel's range) the last U mod S key blocks (U key
blocks, S SMs), when they are at most S / 2, run as two CTAs each, one per half of the
query walk, whose fp32 dK / dV partials are added by TMA reductions and converted by a
separate kernel.

Checked here against the oracle on shapes where the split applies on this device (the
shapes are picked from its SM count): a partial last wave, a grid of fewer key blocks than
half the SMs (every block split), GQA and fp16, d=64 with a ragged last key block; and for
fa_bwd_deterministic, which splits the same blocks, bitwise repeatability and dK / dV equal
to fa_bwd's."""

import math

import pytest
import torch

import oracle
from _parity import ATOL, assert_close, assert_relnorm, f64, make_inputs, to_gpu

pytestmark = pytest.mark.gpu


def _split_count(B, N, Hkv):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    units = B * Hkv * ((N + 127) // 128)
    r = units % sms
    return r if 0 < r <= sms // 2 else 0


def _pick_batch(N, Hkv, lo, hi):
    """A batch size in [lo, hi] for which the split applies, else None."""
    for B in range(lo, hi + 1):
        if _split_count(B, N, Hkv):
            return B
    return None


def _check(fa, B, N, Hq, Hkv, d, dtype, seed, deterministic=False):
    if not _split_count(B, N, Hkv):
        pytest.skip("no wave-tail split for this shape on this device")
    x = make_inputs(B, N, Hq, Hkv, d, dtype=dtype, seed=seed)
    q, k, v, do = (to_gpu(x[n]) for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.forward(q, k, v, causal=False, scale=scale)
    g = fa.backward(do, q, k, v, o, lse, causal=False, scale=scale, deterministic=deterministic)
    fa.check_device_error()
    xo = {n: f64(t) for n, t in x.items()}
    ref = oracle.attn_bwd_ref(xo["q"], xo["k"], xo["v"], xo["do"], False, scale)
    for name, got in zip(("dq", "dk", "dv"), g):
        got = f64(got.cpu())
        assert_close(name, got, ref[name], ATOL[dtype], dtype)
        assert_relnorm(name, got, ref[name])
    return (q, k, v, do, o, lse), g


def test_partial_last_wave_bf16(fa_lib):
    """N=1536 (12 key blocks), Hq=Hkv=8: a batch size whose last wave is split."""
    B = _pick_batch(1536, 8, 2, 8)
    if B is None:
        pytest.skip("no batch size in range splits on this device")
    _check(fa_lib, B, 1536, 8, 8, 128, "bf16", 900)


def test_every_block_split(fa_lib):
    """B=1, Hq=Hkv=4, N=1024: 32 key blocks, fewer than half the SMs, all split."""
    _check(fa_lib, 1, 1024, 4, 4, 128, "bf16", 901)


def test_gqa_fp16(fa_lib):
    """fp16, Hq=8, Hkv=4, N=1280 (10 key blocks of 2 query heads each)."""
    B = _pick_batch(1280, 4, 3, 10)
    if B is None:
        pytest.skip("no batch size in range splits on this device")
    _check(fa_lib, B, 1280, 8, 4, 128, "fp16", 902)


def test_d64_ragged(fa_lib):
    """d=64, N=1500: the last key block of each head is ragged, and split blocks include it."""
    B = _pick_batch(1500, 8, 2, 8)
    if B is None:
        pytest.skip("no batch size in range splits on this device")
    _check(fa_lib, B, 1500, 8, 8, 64, "bf16", 903)


def test_deterministic_split(fa_lib):
    """fa_bwd_deterministic splits the same key blocks (its partials use the unused fp32 dQ
    accumulator): five runs identical bit for bit, dK / dV equal to fa_bwd's."""
    fa = fa_lib
    B = _pick_batch(1536, 8, 2, 8)
    if B is None:
        pytest.skip("no batch size in range splits on this device")
    (q, k, v, do, o, lse), g = _check(fa, B, 1536, 8, 8, 128, "bf16", 904, deterministic=False)
    scale = 1.0 / math.sqrt(128)
    runs = [fa.backward(do, q, k, v, o, lse, causal=False, scale=scale, deterministic=True) for _ in range(5)]
    torch.cuda.synchronize()
    fa.check_device_error()
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)
    assert torch.equal(runs[0][1], g[1]) and torch.equal(runs[0][2], g[2])
    assert (runs[0][0].float() - g[0].float()).abs().max().item() <= 2 * ATOL["bf16"]


def test_dq_aliasing_dout_skips_split(fa_lib):
    """dq given the memory of dout (written only after the pass has read dout): the split,
    which would keep its partials in dq, is skipped, and the results are the oracle's."""
    fa = fa_lib
    B = _pick_batch(1536, 8, 2, 8)
    if B is None:
        pytest.skip("no batch size in range splits on this device")
    N, H, d = 1536, 8, 128
    x = make_inputs(B, N, H, H, d, dtype="bf16", seed=905)
    q, k, v, do = (to_gpu(x[n]) for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.forward(q, k, v, causal=False, scale=scale)
    shared = do.clone()
    dq, dk, dv = fa.backward(shared, q, k, v, o, lse, causal=False, scale=scale, dq=shared)
    fa.check_device_error()
    assert dq.data_ptr() == shared.data_ptr()
    xo = {n: f64(t) for n, t in x.items()}
    ref = oracle.attn_bwd_ref(xo["q"], xo["k"], xo["v"], xo["do"], False, scale)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close(name, f64(got.cpu()), ref[name], ATOL["bf16"], "bf16")
