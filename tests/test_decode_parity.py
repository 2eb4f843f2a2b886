"""Decode forward (a few new queries against a key/value cache, keys split across CTAs
and merged by log-sum-exp): the CUDA path against the fp64 oracle.

Each sequence b is checked as one unequal-length problem of the oracle
(``oracle.attn_fwd_qk`` with Nq queries and the first len_b cache rows, mask aligned at
the bottom-right corner).  Covers one and several new queries, GQA group packing, split
counts 1 / automatic / forced, sequences shorter than Nq (rows that see no key), an empty
cache, both 16-bit types and head dimensions, and a length out of range."""

import math

import numpy as np
import pytest
import torch

import oracle
from _parity import ATOL, LSE_ATOL, assert_close, f64
from exact_attention_38_gb300.inputs import make_decode_inputs

pytestmark = pytest.mark.gpu


def _check(fa, B, Nq, Nmax, Hq, Hkv, d, lens, dtype, causal, num_splits, seed):
    x = make_decode_inputs(B, Nq, Nmax, Hq, Hkv, d, dtype=dtype, seed=seed)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.forward_decode(q, k, v, cl, causal=causal, scale=scale, num_splits=num_splits)
    fa.check_device_error()
    o, lse = f64(o.cpu()), lse.cpu().numpy().astype(np.float64)
    xo = {n: f64(x[n]) for n in ("q", "k", "v")}
    for b in range(B):
        ro, rl = oracle.attn_fwd_qk(xo["q"][b], xo["k"][b, :lens[b]], xo["v"][b, :lens[b]], causal, scale)
        assert_close(f"o[b={b}]", o[b], ro, ATOL[dtype], dtype)
        assert np.array_equal(np.isneginf(lse[b]), np.isneginf(rl)), f"lse[b={b}]: rows without keys must be -inf"
        fin = np.isfinite(rl)
        if fin.any():
            assert np.max(np.abs(lse[b][fin] - rl[fin])) <= LSE_ATOL


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("num_splits", [0, 1, 7])
def test_single_query_gqa(fa_lib, causal, num_splits):
    _check(fa_lib, 3, 1, 3000, 8, 2, 128, [1, 2999, 777], "bf16", causal, num_splits, 41)


@pytest.mark.parametrize("causal", [False, True])
def test_several_queries_short_caches(fa_lib, causal):
    # Nq = 4 new tokens; the second sequence is shorter than Nq (its first queries see
    # nothing under the mask), the third is empty
    _check(fa_lib, 3, 4, 1000, 16, 2, 128, [1000, 3, 0], "bf16", causal, 0, 42)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_full_tile_fp16_d64(fa_lib, causal, num_splits):
    # G * Nq = 8 * 16 = 128 packed rows: the whole tile
    _check(fa_lib, 2, 16, 2100, 16, 2, 64, [2100, 1234], "fp16", causal, num_splits, 43)


def test_long_cache_many_splits(fa_lib):
    _check(fa_lib, 1, 2, 40000, 32, 8, 128, [39999], "bf16", True, 0, 44)


@pytest.mark.parametrize("causal,Nq,num_splits", [(False, 1, 0), (True, 3, 0), (True, 1, 4), (False, 2, 1)])
def test_two_ctas_per_sm_shape(fa_lib, causal, Nq, num_splits):
    # 6 x 2 = 12 (batch, kv head) units at d = 128: the two-CTAs-per-SM ring (at most 8
    # units take the deep ring, which the tests above cover)
    _check(fa_lib, 6, Nq, 1700, 8, 2, 128, [1700, 1, 129, 0, 900, 1313], "bf16", causal, num_splits, 52)


def test_length_out_of_range_is_reported(fa_lib):
    fa = fa_lib
    x = make_decode_inputs(2, 1, 256, 4, 4, 64, dtype="bf16", seed=45)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    cl = torch.tensor([100, 300], dtype=torch.int32, device="cuda")  # 300 > Nmax
    o = torch.full_like(q, float("nan"))
    fa.forward_decode(q, k, v, cl, out=o, num_splits=1)
    with pytest.raises(fa.FaError) as e:
        fa.check_device_error()
    assert e.value.status == fa.FA_ERR_INVALID
    assert torch.isnan(o[1]).all() and not torch.isnan(o[0]).any()


def _paged(x, B, Nmax, lens, seed):
    """Scatter the contiguous caches into 128-row pages in a shuffled order: returns
    k_pages, v_pages [num_pages, 128, Hkv, d] and the block table [B, max_pages]."""
    max_pages = (Nmax + 127) // 128
    num_pages = B * max_pages + 3  # a few pages nobody uses
    perm = np.random.default_rng(seed).permutation(num_pages)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    shape = (num_pages, 128) + tuple(x["k"].shape[2:])
    kp = torch.zeros(shape, dtype=x["k"].dtype)
    vp = torch.zeros(shape, dtype=x["v"].dtype)
    n = 0
    for b in range(B):
        for j in range((lens[b] + 127) // 128):
            pg = int(perm[n])
            n += 1
            table[b, j] = pg
            rows = min(128, Nmax - 128 * j)
            kp[pg, :rows] = x["k"][b, 128 * j:128 * j + rows]
            vp[pg, :rows] = x["v"][b, 128 * j:128 * j + rows]
    return kp, vp, torch.from_numpy(table)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("num_splits", [0, 1, 5])
def test_paged_cache_matches_contiguous(fa_lib, causal, num_splits):
    """The paged cache gives the same bits as the contiguous one (the same products in the
    same order, only the K/V tile addresses differ), and both agree with the oracle."""
    fa = fa_lib
    B, Nq, Nmax, Hq, Hkv, d = 3, 2, 1200, 8, 2, 128
    lens = [1200, 1, 640]
    x = make_decode_inputs(B, Nq, Nmax, Hq, Hkv, d, dtype="bf16", seed=46)
    kp, vp, table = _paged(x, B, Nmax, lens, seed=47)
    q = x["q"].cuda()
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o_c, l_c = fa.forward_decode(q, x["k"].cuda(), x["v"].cuda(), cl, causal=causal, num_splits=num_splits)
    o_p, l_p = fa.forward_decode_paged(q, kp.cuda(), vp.cuda(), table.cuda(), cl, causal=causal,
                                       num_splits=num_splits)
    fa.check_device_error()
    assert torch.equal(o_c, o_p) and torch.equal(l_c, l_p)
    xo = {n: f64(x[n]) for n in ("q", "k", "v")}
    o = f64(o_p.cpu())
    for b in range(B):
        ro, _ = oracle.attn_fwd_qk(xo["q"][b], xo["k"][b, :lens[b]], xo["v"][b, :lens[b]], causal, 1 / math.sqrt(d))
        assert_close(f"o[b={b}]", o[b], ro, ATOL["bf16"], "bf16")


def test_paged_page_out_of_range_is_reported(fa_lib):
    fa = fa_lib
    x = make_decode_inputs(1, 1, 256, 4, 4, 64, dtype="bf16", seed=48)
    kp, vp, table = _paged(x, 1, 256, [256], seed=49)
    table[0, 1] = 10_000  # no such page
    fa.forward_decode_paged(x["q"].cuda(), kp.cuda(), vp.cuda(), table.cuda(),
                            torch.tensor([256], dtype=torch.int32, device="cuda"), num_splits=1)
    with pytest.raises(fa.FaError) as e:
        fa.check_device_error()
    assert e.value.status == fa.FA_ERR_INVALID


@pytest.mark.parametrize("dtype,d,Nq,G", [("fp16", 64, 4, 4), ("bf16", 64, 1, 8), ("fp16", 128, 3, 2)])
def test_paged_cache_other_shapes(fa_lib, dtype, d, Nq, G):
    """Paged caches with d = 64, fp16 and several queries under the bottom-right mask:
    the same bits as the contiguous cache, within tolerance of the oracle, lse included."""
    fa = fa_lib
    B, Nmax, Hkv = 2, 700, 2
    Hq = G * Hkv
    lens = [700, 257]
    x = make_decode_inputs(B, Nq, Nmax, Hq, Hkv, d, dtype=dtype, seed=50 + d + Nq)
    kp, vp, table = _paged(x, B, Nmax, lens, seed=51)
    q = x["q"].cuda()
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o_c, l_c = fa.forward_decode(q, x["k"].cuda(), x["v"].cuda(), cl, causal=True, num_splits=3)
    o_p, l_p = fa.forward_decode_paged(q, kp.cuda(), vp.cuda(), table.cuda(), cl, causal=True, num_splits=3)
    fa.check_device_error()
    assert torch.equal(o_c, o_p) and torch.equal(l_c, l_p)
    xo = {n: f64(x[n]) for n in ("q", "k", "v")}
    o, lse = f64(o_p.cpu()), l_p.cpu().numpy().astype(np.float64)
    for b in range(B):
        ro, rl = oracle.attn_fwd_qk(xo["q"][b], xo["k"][b, :lens[b]], xo["v"][b, :lens[b]], True, 1 / math.sqrt(d))
        assert_close(f"o[b={b}]", o[b], ro, ATOL[dtype], dtype)
        assert np.max(np.abs(lse[b] - rl)) <= LSE_ATOL
