"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no attention arithmetic: it only draws random numbers.  Recipe
(the pages name no generator; only the small fp16 case fixes seed 0): a CPU
``torch.Generator`` seeded with ``seed`` draws fp32 standard normals for q, k, v
and then dO, in that order, with shapes [B, N, Hq, d], [B, N, Hkv, d],
[B, N, Hkv, d], [B, N, Hq, d]; each is rounded to nearest into the 16-bit dtype.
The workload family is the one the FlashAttention-2 pages benchmark
(iid N(0,1) activations, head dim 64 or 128, 16k tokens per batch).
"""

from __future__ import annotations

import math

import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


def make_inputs(B, N, Hq, Hkv, d, dtype="bf16", seed=0, with_do=True, special=None):
    """Return a dict of CPU tensors q, k, v (and do) in the 16-bit ``dtype``.

    ``special`` optionally overrides the draw to build closed-form cases:
    "v_ones" sets V to 1, "q_zero" sets Q to 0 (the draw order is unchanged).
    """
    tdt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randn((B, N, Hq, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, N, Hkv, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, N, Hkv, d), generator=g, dtype=torch.float32)
    out = {}
    if with_do:
        out["do"] = torch.randn((B, N, Hq, d), generator=g, dtype=torch.float32).to(tdt)
    if special == "v_ones":
        v = torch.ones_like(v)
    elif special == "q_zero":
        q = torch.zeros_like(q)
    elif special is not None:
        raise ValueError(f"unknown special case {special!r}")
    out["q"] = q.to(tdt)
    out["k"] = k.to(tdt)
    out["v"] = v.to(tdt)
    return out


def to_f64(t):
    """Exact upcast of a 16-bit CPU tensor to a float64 numpy array."""
    return t.detach().to("cpu", torch.float64).numpy()


def make_varlen_inputs(seg_q, seg_k, Hq, Hkv, d, dtype="bf16", seed=0):
    """Packed variable-length batch: CPU tensors q, do [sum(seg_q), Hq, d] and k, v
    [sum(seg_k), Hkv, d] (16-bit ``dtype``) and int32 offsets cu_q, cu_k [B+1].

    ``seg_q[b]`` / ``seg_k[b]`` are the rows each sequence owns in the packed tensors
    (its length, or for a padded batch its padded length).  Same draw recipe as
    ``make_inputs``: one CPU generator, fp32 normals for q, k, v, dO in that order,
    rounded to nearest into the 16-bit type.
    """
    tdt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    tq, tk = int(sum(seg_q)), int(sum(seg_k))
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randn((tq, Hq, d), generator=g, dtype=torch.float32)
    k = torch.randn((tk, Hkv, d), generator=g, dtype=torch.float32)
    v = torch.randn((tk, Hkv, d), generator=g, dtype=torch.float32)
    do = torch.randn((tq, Hq, d), generator=g, dtype=torch.float32)
    cu_q = torch.zeros(len(seg_q) + 1, dtype=torch.int32)
    cu_k = torch.zeros(len(seg_k) + 1, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(torch.tensor(list(seg_q), dtype=torch.int64), 0).to(torch.int32)
    cu_k[1:] = torch.cumsum(torch.tensor(list(seg_k), dtype=torch.int64), 0).to(torch.int32)
    return {"q": q.to(tdt), "k": k.to(tdt), "v": v.to(tdt), "do": do.to(tdt), "cu_q": cu_q, "cu_k": cu_k}


def make_decode_inputs(B, Nq, Nmax, Hq, Hkv, d, dtype="bf16", seed=0):
    """Decode-shaped inputs: CPU tensors q [B, Nq, Hq, d] and caches k, v
    [B, Nmax, Hkv, d] (every cache row drawn, including rows past a sequence's length).
    Same recipe as ``make_inputs``: one CPU generator, fp32 normals in the order q, k, v,
    rounded to nearest into the 16-bit type."""
    tdt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randn((B, Nq, Hq, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, Nmax, Hkv, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, Nmax, Hkv, d), generator=g, dtype=torch.float32)
    return {"q": q.to(tdt), "k": k.to(tdt), "v": v.to(tdt)}


def make_fp8_block_inputs(B, N, Hq, Hkv, d, seed=0, spread=4.0):
    """E4M3 inputs with one descale per 128-row block of each head: q, k, v fp32 normals
    from one CPU generator, each 128-row block of each head multiplied by its own factor
    drawn log-uniformly from [1/spread, spread] (so the blocks' ranges differ), divided by
    the block's descale = block amax / 448 and rounded to nearest E4M3.  Returns a dict with
    CPU tensors q, k, v (E4M3) and q_descale [B, Hq, nb], k_descale and v_descale
    [B, Hkv, nb] (fp32, nb = ceil(N / 128)); real value = E4M3 value x its block's descale."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    nb = (N + 127) // 128
    out = {}
    for name, H in (("q", Hq), ("k", Hkv), ("v", Hkv)):
        x = torch.randn((B, N, H, d), generator=g, dtype=torch.float32)
        f = torch.exp((torch.rand((B, nb, H), generator=g) * 2.0 - 1.0) * math.log(spread))
        x = x * f.repeat_interleave(128, dim=1)[:, :N, :, None]
        xb = torch.zeros((B, nb * 128, H, d), dtype=torch.float32)
        xb[:, :N] = x
        amax = xb.abs().reshape(B, nb, 128, H, d).amax(dim=(2, 4))  # [B, nb, H]
        ds = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        out[name] = (x / ds.repeat_interleave(128, dim=1)[:, :N, :, None]).to(torch.float8_e4m3fn)
        out[name + "_descale"] = ds.permute(0, 2, 1).contiguous()  # [B, H, nb]
    return out


def make_fp8_inputs(B, N, Hq, Hkv, d, seed=0):
    """E4M3 inputs with one descale per tensor: the ``make_inputs`` draw (q, k, v fp32
    normals from one CPU generator), each tensor divided by its descale = amax / 448 and
    rounded to nearest E4M3 (torch.float8_e4m3fn).  Returns a dict with CPU tensors q, k,
    v (E4M3) and floats q_descale, k_descale, v_descale; real value = E4M3 value x
    descale."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    out = {}
    for name, shape in (("q", (B, N, Hq, d)), ("k", (B, N, Hkv, d)), ("v", (B, N, Hkv, d))):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        ds = float(x.abs().max()) / 448.0
        out[name] = (x / ds).to(torch.float8_e4m3fn)
        out[name + "_descale"] = ds
    return out
