"""The persistent backward that fa_bwd and fa_bwd_deterministic run for short sequences
(fixed length; one CTA per SM takes (batch, key/value head, 128-key block) units from a
counter pair in device memory).

Checked here: the oracle's values on grids with fewer units than SMs and with several
units per CTA, both masks, both head sizes, GQA and fp16; dK and dV identical bit for bit
to the one-CTA-per-block kernel's (reached through the variable-length entry point with
equal lengths, which runs that kernel on the same products in the same order); that the
counter pair is put back after every launch; and launches on two streams at once."""

import math

import pytest
import torch

import oracle
from _parity import ATOL, assert_close, assert_relnorm, f64, make_inputs, to_gpu

pytestmark = pytest.mark.gpu

# more launches than the library's ring of counter pairs (256)
RING_WRAP_LAUNCHES = 300


def _run(fa, x, causal, deterministic=False):
    q, k, v, do = (to_gpu(x[n]) for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(q.shape[-1])
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    g = fa.backward(do, q, k, v, o, lse, causal=causal, scale=scale, deterministic=deterministic)
    fa.check_device_error()
    return (q, k, v, do, o, lse), g


def _oracle_check(fa, B, N, Hq, Hkv, d, causal, seed, dtype="bf16", deterministic=False):
    x = make_inputs(B, N, Hq, Hkv, d, dtype=dtype, seed=seed)
    _, g = _run(fa, x, causal, deterministic)
    xo = {n: f64(t) for n, t in x.items()}
    ref = oracle.attn_bwd_ref(xo["q"], xo["k"], xo["v"], xo["do"], causal, 1.0 / math.sqrt(d))
    for name, got in zip(("dq", "dk", "dv"), g):
        got = f64(got.cpu())
        assert_close(name, got, ref[name], ATOL[dtype], dtype)
        assert_relnorm(name, got, ref[name])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_fewer_units_than_sms(fa_lib, causal, d):
    """B=1, Hq=3, Hkv=1, N=300: 3 units (GQA group of 3), the last key block ragged."""
    _oracle_check(fa_lib, 1, 300, 3, 1, d, causal, 800 + d + causal)


@pytest.mark.parametrize("causal", [False, True])
def test_many_units_per_cta(fa_lib, causal):
    """B=12, Hq=Hkv=16, N=512: 768 units on at most the SM count of CTAs."""
    _oracle_check(fa_lib, 12, 512, 16, 16, 128, causal, 810 + causal)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_fp16_d64_many_units(fa_lib, causal):
    """fp16, d=64, B=40, Hq=8, Hkv=2, N=500: 320 units of 4 query heads each, ragged last
    block."""
    _oracle_check(fa_lib, 40, 500, 8, 2, 64, causal, 820 + causal, dtype="fp16")


@pytest.mark.parametrize("causal", [False, True])
def test_deterministic_many_units(fa_lib, causal):
    """fa_bwd_deterministic on the persistent kernel without its dQ path: the oracle's
    values, five runs identical bit for bit, dK / dV equal to fa_bwd's."""
    fa = fa_lib
    x = make_inputs(16, 384, 8, 4, 128, dtype="bf16", seed=830 + causal)
    (q, k, v, do, o, lse), g = _run(fa, x, causal)
    scale = 1.0 / math.sqrt(128)
    runs = [fa.backward(do, q, k, v, o, lse, causal=causal, scale=scale, deterministic=True) for _ in range(5)]
    torch.cuda.synchronize()
    fa.check_device_error()
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)
    assert torch.equal(runs[0][1], g[1]) and torch.equal(runs[0][2], g[2])
    xo = {n: f64(t) for n, t in x.items()}
    ref = oracle.attn_bwd_ref(xo["q"], xo["k"], xo["v"], xo["do"], causal, scale)
    for name, got in zip(("dq", "dk", "dv"), runs[0]):
        assert_close(name, f64(got.cpu()), ref[name], ATOL["bf16"], "bf16")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_dkdv_match_one_cta_per_block_kernel(fa_lib, causal, d):
    """With every sequence of length N (a multiple of 128, so no tile crosses a sequence
    end) the variable-length backward runs the one-CTA-per-block kernel on the very
    products the persistent kernel issues, in the same order: dK and dV must agree bit
    for bit, dQ (fp32 additions in a run-dependent order) within the bound."""
    fa = fa_lib
    B, N, Hq, Hkv = 16, 384, 8, 4
    x = make_inputs(B, N, Hq, Hkv, d, dtype="bf16", seed=840 + d + causal)
    (q, k, v, do, o, lse), (dq, dk, dv) = _run(fa, x, causal)
    scale = 1.0 / math.sqrt(d)
    cu = torch.arange(0, (B + 1) * N, N, dtype=torch.int32, device="cuda")
    flat = lambda t: t.reshape(B * N, t.shape[2], d)  # noqa: E731
    lse_v = lse.permute(1, 0, 2).reshape(Hq, B * N).contiguous()
    vq, vk, vv = fa.backward_varlen(flat(do), flat(q), flat(k), flat(v), flat(o), lse_v, cu, cu, N, N,
                                    causal=causal, scale=scale)
    torch.cuda.synchronize()
    fa.check_device_error()
    assert torch.equal(flat(dk), vk)
    assert torch.equal(flat(dv), vv)
    assert_close("dq", f64(vq.cpu()), f64(flat(dq).cpu()), 2 * ATOL["bf16"])


@pytest.mark.parametrize("causal", [False, True])
def test_counter_reset_over_many_launches(fa_lib, causal):
    """Every launch must leave its counter pair at {0, 0}: a pair that was not put back
    would make the launch that next picks it skip key blocks (their dK / dV stay as the
    buffers held them)."""
    fa = fa_lib
    x = make_inputs(4, 384, 8, 2, 128, dtype="bf16", seed=850 + causal)
    (q, k, v, do, o, lse), (rq, rk, rv) = _run(fa, x, causal)
    scale = 1.0 / math.sqrt(128)
    dq, dk, dv = torch.empty_like(rq), torch.empty_like(rk), torch.empty_like(rv)
    bad = 0
    for i in range(RING_WRAP_LAUNCHES):
        dk.fill_(float("nan"))
        dv.fill_(float("nan"))
        fa.backward(do, q, k, v, o, lse, causal=causal, scale=scale, dq=dq, dk=dk, dv=dv)
        if i % 25 == 0 or i == RING_WRAP_LAUNCHES - 1:
            torch.cuda.synchronize()
            bad += int(not (torch.equal(dk, rk) and torch.equal(dv, rv)))
    torch.cuda.synchronize()
    fa.check_device_error()
    assert bad == 0
    assert torch.equal(dk, rk) and torch.equal(dv, rv)
    assert (dq.float() - rq.float()).abs().max().item() <= 2 * ATOL["bf16"]


def test_two_streams_take_their_own_units(fa_lib):
    """Persistent backward launches of two shapes, and persistent forwards, interleaved on
    two streams: dK and dV equal those of separate launches."""
    fa = fa_lib
    xa = make_inputs(8, 512, 4, 4, 128, dtype="bf16", seed=860)
    xb = make_inputs(6, 256, 8, 2, 64, dtype="bf16", seed=861)
    (qa, ka, va, doa, oa, la), ra = _run(fa, xa, False)
    (qb, kb, vb, dob, ob, lb), rb = _run(fa, xb, True)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(20):
        with torch.cuda.stream(sa):
            fa.forward(qa, ka, va, causal=False, stream=sa)
            ga = fa.backward(doa, qa, ka, va, oa, la, causal=False, stream=sa)
        with torch.cuda.stream(sb):
            gb = fa.backward(dob, qb, kb, vb, ob, lb, causal=True, stream=sb)
            fa.forward(qb, kb, vb, causal=True, stream=sb)
        outs.append((ga, gb))
    torch.cuda.synchronize()
    fa.check_device_error()
    for ga, gb in outs:
        assert torch.equal(ga[1], ra[1]) and torch.equal(ga[2], ra[2])
        assert torch.equal(gb[1], rb[1]) and torch.equal(gb[2], rb[2])


@pytest.mark.parametrize("deterministic", [False, True])
def test_cuda_graph_capture_and_replay(fa_lib, deterministic):
    """Forward and persistent backward captured in a CUDA graph (the backward's kernels
    are chained by programmatic dependent launches, which capture records as graph edges)
    and replayed: dK / dV (and, deterministic, dQ) equal the eager call's bits."""
    fa = fa_lib
    B, N, Hq, Hkv, d = 8, 448, 8, 4, 128
    x = make_inputs(B, N, Hq, Hkv, d, dtype="bf16", seed=870 + deterministic)
    q, k, v, do = (to_gpu(x[n]) for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, Hq, Hkv, N, d), dtype=torch.uint8, device="cuda")

    def step(stream):
        fa.forward(q, k, v, causal=False, scale=scale, out=o, lse=lse, stream=stream)
        fa.backward(do, q, k, v, o, lse, causal=False, scale=scale, workspace=ws, dq=dq, dk=dk, dv=dv,
                    stream=stream, deterministic=deterministic)

    step(None)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (o, lse, dq, dk, dv)]
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step(s)
    torch.cuda.synchronize()
    for _ in range(3):
        for t in (o, lse, dq, dk, dv):
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        fa.check_device_error()
        for name, r, t in zip(("o", "lse", "dq", "dk", "dv"), ref, (o, lse, dq, dk, dv)):
            if name == "dq" and not deterministic:
                assert (t.float() - r.float()).abs().max().item() <= 2 * ATOL["bf16"]
            else:
                assert torch.equal(r, t), name
