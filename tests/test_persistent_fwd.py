"""The persistent forward that fa_fwd runs for short sequences: one CTA per SM takes
(batch, head, 256-query) units from a counter pair in device memory.

Checked here: the oracle's values on grids with fewer units than SMs and with several
units per CTA, both masks and both head sizes; that the counter pair is put back after
every launch (more launches back to back than the ring of pairs holds give identical
bits); and that launches on two streams at once take none of each other's units."""

import math

import pytest
import torch

import oracle
from _parity import ATOL, LSE_ATOL, assert_close, f64, gpu_forward, make_inputs, to_gpu

pytestmark = pytest.mark.gpu

# more launches than the library's ring of counter pairs (256)
RING_WRAP_LAUNCHES = 300


def _oracle_check(fa, B, N, Hq, Hkv, d, causal, seed, dtype="bf16"):
    x = make_inputs(B, N, Hq, Hkv, d, dtype=dtype, seed=seed, with_do=False)
    _, o, lse = gpu_forward(fa, x, causal)
    xo = {k: f64(v) for k, v in x.items()}
    want_o, want_lse = oracle.attn_fwd_ref(xo["q"], xo["k"], xo["v"], causal, 1.0 / math.sqrt(d))
    assert_close("O", f64(o.cpu()), want_o, ATOL[dtype], dtype)
    assert_close("lse", lse.cpu().double().numpy(), want_lse, LSE_ATOL)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_fewer_units_than_sms(fa_lib, causal, d):
    """B=1, Hq=3, Hkv=1, N=300: 6 units, the second tile of each last unit past N."""
    _oracle_check(fa_lib, 1, 300, 3, 1, d, causal, 700 + d + causal)


@pytest.mark.parametrize("causal", [False, True])
def test_many_units_per_cta(fa_lib, causal):
    """B=40, Hq=Hkv=4, N=512: 320 units on at most the SM count of CTAs, GQA off."""
    _oracle_check(fa_lib, 40, 512, 4, 4, 128, causal, 710 + causal)


def test_fp16_gqa_causal_1024(fa_lib):
    """fp16, B=2, Hq=8, Hkv=2, N=1000 with the mask (the persistent range of the causal
    forward), ragged last block."""
    _oracle_check(fa_lib, 2, 1000, 8, 2, 128, True, 720, dtype="fp16")


def _fwd(fa, q, k, v, causal, stream=None):
    return fa.forward(q, k, v, causal=causal, scale=1.0 / math.sqrt(q.shape[-1]), stream=stream)


@pytest.mark.parametrize("causal", [False, True])
def test_counter_reset_over_many_launches(fa_lib, causal):
    """Every launch must leave its counter pair at {0, 0}: a pair that was not put back
    would make the launch that next picks it skip units (their O stays as the buffer
    held it)."""
    fa = fa_lib
    x = make_inputs(2, 384, 4, 2, 128, dtype="bf16", seed=730 + causal, with_do=False)
    q, k, v = (to_gpu(x[n]) for n in ("q", "k", "v"))
    ref_o, ref_lse = _fwd(fa, q, k, v, causal)
    o = torch.full_like(ref_o, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    scale = 1.0 / math.sqrt(128)
    bad = 0
    for i in range(RING_WRAP_LAUNCHES):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        fa.forward(q, k, v, causal=causal, scale=scale, out=o, lse=lse)
        if i % 25 == 0 or i == RING_WRAP_LAUNCHES - 1:
            torch.cuda.synchronize()
            bad += int(not (torch.equal(o, ref_o) and torch.equal(lse, ref_lse)))
    torch.cuda.synchronize()
    fa.check_device_error()
    assert bad == 0
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)


def test_two_streams_take_their_own_units(fa_lib):
    """Persistent launches of two different shapes interleaved on two streams give the
    bits of separate launches."""
    fa = fa_lib
    xa = make_inputs(8, 512, 4, 4, 128, dtype="bf16", seed=740, with_do=False)
    xb = make_inputs(3, 256, 8, 2, 64, dtype="bf16", seed=741, with_do=False)
    a = [to_gpu(xa[n]) for n in ("q", "k", "v")]
    b = [to_gpu(xb[n]) for n in ("q", "k", "v")]
    ref_a = _fwd(fa, *a, False)
    ref_b = _fwd(fa, *b, True)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(20):
        with torch.cuda.stream(sa):
            ga = _fwd(fa, *a, False, stream=sa)
        with torch.cuda.stream(sb):
            gb = _fwd(fa, *b, True, stream=sb)
        outs.append((ga, gb))
    torch.cuda.synchronize()
    fa.check_device_error()
    for ga, gb in outs:
        for r, g in zip(ref_a, ga):
            assert torch.equal(r, g)
        for r, g in zip(ref_b, gb):
            assert torch.equal(r, g)
