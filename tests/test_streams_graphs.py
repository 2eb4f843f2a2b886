"""Concurrency and graph capture: the entry points keep no per-call state (all but
fa_bwd_noalloc, whose calls share one scratch array and must be serialised), so calls on
two streams may overlap, and a forward + backward can be captured into a CUDA graph and
replayed.  The deterministic backward makes every comparison bit-exact."""

import math

import pytest
import torch

from _parity import make_inputs, to_gpu

pytestmark = pytest.mark.gpu


def _inputs(seed):
    x = make_inputs(2, 700, 4, 2, 128, dtype="bf16", seed=seed)
    return [to_gpu(x[n]) for n in ("q", "k", "v", "do")]


def _run(fa, q, k, v, do, causal, stream=None):
    scale = 1.0 / math.sqrt(q.shape[-1])
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale, stream=stream)
    dq, dk, dv = fa.backward(do, q, k, v, o, lse, causal=causal, scale=scale, stream=stream, deterministic=True)
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("causal", [False, True])
def test_two_streams_overlap(fa_lib, causal):
    fa = fa_lib
    xa, xb = _inputs(600), _inputs(601)
    ref_a, ref_b = _run(fa, *xa, causal), _run(fa, *xb, causal)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(3):  # interleave launches on both streams
        with torch.cuda.stream(sa):
            ga = _run(fa, *xa, causal, stream=sa)
        with torch.cuda.stream(sb):
            gb = _run(fa, *xb, causal, stream=sb)
        outs.append((ga, gb))
    torch.cuda.synchronize()
    fa.check_device_error()
    for ga, gb in outs:
        for r, g in zip(ref_a, ga):
            assert torch.equal(r, g)
        for r, g in zip(ref_b, gb):
            assert torch.equal(r, g)


def test_cuda_graph_capture_and_replay(fa_lib):
    fa = fa_lib
    q, k, v, do = _inputs(602)
    scale = 1.0 / math.sqrt(128)
    o = torch.empty_like(q)
    lse = torch.empty((2, 4, 700), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(2, 4, 2, 700, 128), dtype=torch.uint8, device="cuda")

    def step(stream):
        fa.forward(q, k, v, causal=True, scale=scale, out=o, lse=lse, stream=stream)
        fa.backward(do, q, k, v, o, lse, causal=True, scale=scale, workspace=ws, dq=dq, dk=dk, dv=dv,
                    stream=stream, deterministic=True)

    step(None)  # eager reference (also resolves the library's per-device lookups)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (o, lse, dq, dk, dv)]
    for t in (o, lse, dq, dk, dv):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step(s)
    torch.cuda.synchronize()
    for _ in range(2):
        for t in (o, lse, dq, dk, dv):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        fa.check_device_error()
        for r, t in zip(ref, (o, lse, dq, dk, dv)):
            assert torch.equal(r, t)


def _decode_inputs(seed):
    from exact_attention_38_gb300.inputs import make_decode_inputs

    x = make_decode_inputs(2, 1, 3000, 16, 2, 128, dtype="bf16", seed=seed)
    return x["q"].cuda(), x["k"].cuda(), x["v"].cuda()


def test_decode_split_combine_in_graph_and_back_to_back(fa_lib):
    """The split combine is launched as a programmatic dependent of the decode kernel:
    back-to-back calls that reuse one workspace, and a captured graph replayed with new
    cache lengths, give the bits of separate eager calls."""
    fa = fa_lib
    q, k, v = _decode_inputs(603)
    lens_list = [[3000, 1], [129, 2999], [1500, 1500]]
    refs = []
    for lens in lens_list:
        cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
        o, lse = fa.forward_decode(q, k, v, cl, num_splits=6)
        torch.cuda.synchronize()
        refs.append((o.clone(), lse.clone()))
    ws = torch.empty(fa.fa_decode_workspace_size(2, 16, 2, 1, 3000, 128, 6), dtype=torch.uint8, device="cuda")
    o, lse = torch.empty_like(q), torch.empty((2, 16, 1), dtype=torch.float32, device="cuda")
    outs = []
    for _ in range(2):  # back to back on one stream, one workspace
        for lens in lens_list:
            cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
            fa.forward_decode(q, k, v, cl, num_splits=6, out=o, lse=lse, workspace=ws)
            outs.append((o.clone(), lse.clone()))
    torch.cuda.synchronize()
    fa.check_device_error()
    for n, (og, lg) in enumerate(outs):
        assert torch.equal(og, refs[n % 3][0]) and torch.equal(lg, refs[n % 3][1])
    cl = torch.tensor(lens_list[0], dtype=torch.int32, device="cuda")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fa.forward_decode(q, k, v, cl, num_splits=6, out=o, lse=lse, workspace=ws, stream=s)
    torch.cuda.synchronize()
    for n, lens in enumerate(lens_list):
        cl.copy_(torch.tensor(lens, dtype=torch.int32))
        o.zero_()
        g.replay()
        torch.cuda.synchronize()
        fa.check_device_error()
        assert torch.equal(o, refs[n][0]) and torch.equal(lse, refs[n][1])
