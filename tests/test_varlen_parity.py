"""Variable-length batches and unequal query / key lengths: the CUDA path against the
fp64 oracle (``oracle.varlen``), forward and backward.

Covers packed batches with ragged lengths, query and key lengths that differ in both
directions (bottom-right-aligned causal mask, rows that see no key), empty sequences,
padded batches (seqused), GQA, both 16-bit types and both head dimensions, that rows
belonging to no sequence are never written, and that inconsistent offsets are
reported instead of read past the tensors."""

import math

import numpy as np
import pytest
import torch

import oracle
from _parity import ATOL, LSE_ATOL, assert_close, assert_relnorm, f64, half_ulp
from exact_attention_38_gb300.inputs import make_varlen_inputs

pytestmark = pytest.mark.gpu

SENTINEL = float("nan")


def _run(fa, x, seg_q, seg_k, used_q, used_k, causal, bwd=True):
    dev = "cuda"
    q, k, v, do = (x[n].to(dev).contiguous() for n in ("q", "k", "v", "do"))
    cu_q, cu_k = x["cu_q"].to(dev), x["cu_k"].to(dev)
    uq = None if used_q is None else torch.tensor(used_q, dtype=torch.int32, device=dev)
    uk = None if used_k is None else torch.tensor(used_k, dtype=torch.int32, device=dev)
    lq = used_q if used_q is not None else seg_q
    lk = used_k if used_k is not None else seg_k
    max_q, max_k = max(lq), max(lk)
    scale = 1.0 / math.sqrt(q.shape[-1])
    o = torch.full_like(q, SENTINEL)
    lse = torch.full((q.shape[1], q.shape[0]), SENTINEL, dtype=torch.float32, device=dev)
    fa.forward_varlen(q, k, v, cu_q, cu_k, max_q, max_k, causal=causal, scale=scale, seqused_q=uq, seqused_k=uk,
                      out=o, lse=lse)
    fa.check_device_error()
    out = {"o": o, "lse": lse}
    if bwd:
        dq, dk, dv = torch.full_like(q, SENTINEL), torch.full_like(k, SENTINEL), torch.full_like(v, SENTINEL)
        fa.backward_varlen(do, q, k, v, o, lse, cu_q, cu_k, max_q, max_k, causal=causal, scale=scale,
                           seqused_q=uq, seqused_k=uk, dq=dq, dk=dk, dv=dv)
        fa.check_device_error()
        out.update(dq=dq, dk=dk, dv=dv)
    return out, scale


def _check(fa, seg_q, seg_k, Hq, Hkv, d, dtype, causal, seed, used_q=None, used_k=None, bwd=True):
    x = make_varlen_inputs(seg_q, seg_k, Hq, Hkv, d, dtype=dtype, seed=seed)
    g, scale = _run(fa, x, seg_q, seg_k, used_q, used_k, causal, bwd)
    xo = {n: f64(x[n]) for n in ("q", "k", "v", "do")}
    cu_q, cu_k = x["cu_q"].numpy(), x["cu_k"].numpy()
    o_ref, lse_ref = oracle.attn_varlen_fwd_ref(xo["q"], xo["k"], xo["v"], cu_q, cu_k, causal, scale, used_q, used_k)
    got_o = f64(g["o"].cpu())
    got_lse = g["lse"].cpu().numpy().astype(np.float64)
    cov_q = ~np.isnan(o_ref[:, 0, 0])  # rows some sequence owns
    # rows outside every sequence keep the sentinel
    assert np.all(np.isnan(got_o[~cov_q])) and np.all(np.isnan(got_lse[:, ~cov_q]))
    assert_close("o", got_o[cov_q], o_ref[cov_q], ATOL[dtype], dtype)
    want_lse = lse_ref[:, cov_q]
    gl = got_lse[:, cov_q]
    assert np.array_equal(np.isneginf(gl), np.isneginf(want_lse)), "lse: rows without keys must be -inf"
    fin = np.isfinite(want_lse)
    if fin.any():
        assert np.max(np.abs(gl[fin] - want_lse[fin])) <= LSE_ATOL
    if not bwd:
        return
    dq_ref, dk_ref, dv_ref = oracle.attn_varlen_bwd_ref(xo["q"], xo["k"], xo["v"], xo["do"], cu_q, cu_k, causal,
                                                        scale, used_q, used_k)
    cov_k = ~np.isnan(dk_ref[:, 0, 0])
    for name, ref, cov in (("dq", dq_ref, cov_q), ("dk", dk_ref, cov_k), ("dv", dv_ref, cov_k)):
        got = f64(g[name].cpu())
        assert np.all(np.isnan(got[~cov])), f"{name}: a row outside every sequence was written"
        assert_close(name, got[cov], ref[cov], ATOL[dtype], dtype)
        assert_relnorm(name, got[cov], ref[cov])


RAGGED = [1, 17, 128, 129, 300, 64, 1000, 255]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_packed_ragged_equal_lengths(fa_lib, causal, d):
    _check(fa_lib, RAGGED, RAGGED, 4, 2, d, "bf16", causal, 31)


@pytest.mark.parametrize("causal", [False, True])
def test_unequal_lengths_both_ways(fa_lib, causal):
    # includes queries longer than keys (rows that see nothing under the mask), a
    # single-query decode shape, and empty sequences on either side
    seg_q = [5, 200, 130, 1, 0, 700, 3, 260]
    seg_k = [300, 60, 130, 1000, 7, 0, 129, 1]
    _check(fa_lib, seg_q, seg_k, 4, 2, 128, "bf16", causal, 32)


@pytest.mark.parametrize("causal", [False, True])
def test_fp16_gqa_d64(fa_lib, causal):
    _check(fa_lib, [400, 77, 513], [90, 600, 513], 6, 2, 64, "fp16", causal, 33)


@pytest.mark.parametrize("causal", [False, True])
def test_padded_batch_seqused(fa_lib, causal):
    # segments of 384 rows each; only the first seqused rows are real
    _check(fa_lib, [384, 384, 384], [384, 384, 384], 4, 4, 128, "bf16", causal, 34, used_q=[100, 384, 0],
           used_k=[250, 40, 384])


def _rounding_bound(q, k, v, do, causal, scale, u=2.0 ** -8):
    """Worst-case bound on |dQ|, |dK|, |dV| errors of one sequence for the 16-bit steps of
    the backward (dS and P rounded to 16 bits before the products, D formed from the
    16-bit O, outputs rounded), each relative error taken as u = 2^-8 (twice bf16's unit
    roundoff).  Derived from the arithmetic: every product term carries at most that
    relative error, and D's error enters dS through P * dD."""
    nq, hq, d = q.shape
    g = hq // k.shape[1]
    vis = oracle.varlen.visible(nq, k.shape[0], causal)
    bq, bk, bv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    o, lse = oracle.attn_fwd_qk(q, k, v, causal, scale)
    for h in range(hq):
        kh, vh = k[:, h // g], v[:, h // g]
        s = np.where(vis, scale * (q[:, h] @ kh.T), -np.inf)
        with np.errstate(invalid="ignore"):  # rows with no visible key: -inf - (-inf)
            p = np.where(vis, np.exp(s - lse[h][:, None]), 0.0)
        dp = do[:, h] @ vh.T
        dd = np.sum(do[:, h] * o[:, h], axis=1)
        ds = p * (dp - dd[:, None])
        e_dd = u * np.sum(np.abs(do[:, h] * o[:, h]), axis=1)          # D from the rounded O
        e_ds = u * np.abs(ds) + p * e_dd[:, None]                       # per dS element
        bq[:, h] = scale * (e_ds @ np.abs(kh)) + u * np.abs(scale * (ds @ kh))
        bk[:, h // g] += scale * (e_ds.T @ np.abs(q[:, h])) + u * np.abs(scale * (ds.T @ q[:, h]))
        bv[:, h // g] += u * (p.T @ np.abs(do[:, h])) + u * np.abs(p.T @ do[:, h])
    return bq, bk, bv


@pytest.mark.parametrize("causal", [False, True])
def test_few_keys_many_queries(fa_lib, causal):
    """3 keys seen by 384 queries: dS reaches ~10 while dK sums 384 such terms, so the
    16-bit rounding of dS alone moves dK by up to ~0.05 (an exact CPU model of the
    kernel's roundings gives 0.053), above the flat 1.6e-2.  Here the gradients are held
    to the relative-norm bound and, element by element, to the worst-case rounding
    bound of ``_rounding_bound``; the forward keeps the usual bounds."""
    seg_q, seg_k = [384, 384], [3, 384]
    x = make_varlen_inputs(seg_q, seg_k, 4, 4, 128, dtype="bf16", seed=37)
    g, scale = _run(fa_lib, x, seg_q, seg_k, None, None, causal)
    xo = {n: f64(x[n]) for n in ("q", "k", "v", "do")}
    cu_q, cu_k = x["cu_q"].numpy(), x["cu_k"].numpy()
    o_ref, _ = oracle.attn_varlen_fwd_ref(xo["q"], xo["k"], xo["v"], cu_q, cu_k, causal, scale)
    assert_close("o", f64(g["o"].cpu()), o_ref, ATOL["bf16"], "bf16")
    refs = oracle.attn_varlen_bwd_ref(xo["q"], xo["k"], xo["v"], xo["do"], cu_q, cu_k, causal, scale)
    for b in range(2):
        sq, sk = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
        bounds = _rounding_bound(xo["q"][sq], xo["k"][sk], xo["v"][sk], xo["do"][sq], causal, scale)
        for name, ref, bnd, sl in (("dq", refs[0], bounds[0], sq), ("dk", refs[1], bounds[1], sk),
                                   ("dv", refs[2], bounds[2], sk)):
            got = f64(g[name].cpu())[sl]
            want = ref[sl]
            assert_relnorm(name, got, want)
            tol = np.maximum(bnd, ATOL["bf16"] + half_ulp(want, "bf16"))
            assert np.all(np.abs(got - want) <= tol), (name, b, float(np.max(np.abs(got - want) - tol)))


def test_longer_sequences_several_tiles(fa_lib):
    _check(fa_lib, [2048, 1500], [1800, 2600], 2, 1, 128, "bf16", True, 35)


def test_inconsistent_offsets_are_reported(fa_lib):
    """A sequence longer than max_seqlen is skipped and reported as FA_ERR_INVALID
    by the next device-error check, with nothing read or written for it."""
    fa = fa_lib
    x = make_varlen_inputs([100, 300], [100, 300], 2, 2, 64, dtype="bf16", seed=36)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    cu = x["cu_q"].cuda()
    o = torch.full_like(q, SENTINEL)
    lse = torch.full((2, 400), SENTINEL, dtype=torch.float32, device="cuda")
    fa.forward_varlen(q, k, v, cu, cu, 200, 300, causal=False, out=o, lse=lse)  # max_q too small for seq 1
    with pytest.raises(fa.FaError) as e:
        fa.check_device_error()
    assert e.value.status == fa.FA_ERR_INVALID
    assert torch.isnan(o[100:]).all()  # sequence 1 untouched
    fa.check_device_error()  # the error word was cleared
