"""Pins for the variable-length / unequal-length oracle (``oracle/varlen.py``).

Each test compares the oracle with something other than itself: scalar brute force,
the equal-length oracle (a separate implementation of the definition), central
finite differences, closed forms, or invariants the definition implies.  The last
test plants a mistake in the oracle (a top-left instead of bottom-right mask) and
checks that the pins catch it.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import varlen as ov


def _rand(shape, rng):
    return rng.standard_normal(shape)


def _seq(nq, nk, hq, hkv, d, seed):
    rng = np.random.default_rng(seed)
    return (_rand((nq, hq, d), rng), _rand((nk, hkv, d), rng), _rand((nk, hkv, d), rng),
            _rand((nq, hq, d), rng))


LEN_PAIRS = [(1, 1), (3, 7), (7, 3), (5, 5), (1, 9), (9, 1), (6, 0), (0, 4), (4, 12), (12, 4)]


@pytest.mark.parametrize("nq,nk", LEN_PAIRS)
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_qk_matches_scalar_brute_force(nq, nk, causal):
    q, k, v, _ = _seq(nq, nk, 4, 2, 3, seed=nq * 31 + nk)
    scale = 0.7
    o, lse = oracle.attn_fwd_qk(q, k, v, causal, scale)
    ob, lseb = oracle.brute_force_fwd_qk(q, k, v, causal, scale)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(lseb))
    fin = np.isfinite(lseb)
    np.testing.assert_allclose(lse[fin], lseb[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_lengths_reduce_to_square_oracle(causal):
    """Nq = Nk: bottom-right and top-left alignment coincide, so the result must equal
    the square-shape oracle (a separate implementation of the same definition)."""
    q, k, v, do = _seq(11, 11, 4, 2, 5, seed=5)
    scale = 1 / math.sqrt(5)
    o, lse = oracle.attn_fwd_qk(q, k, v, causal, scale)
    o2, lse2 = oracle.attn_fwd_ref(q[None], k[None], v[None], causal, scale)
    np.testing.assert_allclose(o, o2[0], atol=1e-12)
    np.testing.assert_allclose(lse, lse2[0], atol=1e-12)
    g = oracle.attn_bwd_qk(q, k, v, do, causal, scale)
    g2 = oracle.attn_bwd_ref(q[None], k[None], v[None], do[None], causal, scale)
    for a, name in zip(g, ("dq", "dk", "dv")):
        np.testing.assert_allclose(a, g2[name][0], atol=1e-12)


def test_single_query_sees_every_key_under_the_mask():
    """Decode shape (Nq = 1): with the mask aligned at the bottom-right corner the one
    query is the last position and sees the whole key sequence."""
    q, k, v, _ = _seq(1, 13, 2, 1, 4, seed=2)
    o_c, lse_c = oracle.attn_fwd_qk(q, k, v, True, 0.5)
    o_n, lse_n = oracle.attn_fwd_qk(q, k, v, False, 0.5)
    np.testing.assert_allclose(o_c, o_n, atol=1e-14)
    np.testing.assert_allclose(lse_c, lse_n, atol=1e-14)


def test_zero_queries_give_counts_and_means():
    """Q = 0: every visible score is 0, so lse_i = ln(#visible keys) and O_i is the mean
    of the visible V rows; the last query sees all Nk keys, the first Nk - Nq + 1 (or
    none when Nq > Nk)."""
    nq, nk = 6, 9
    _, k, v, _ = _seq(nq, nk, 2, 2, 3, seed=3)
    q = np.zeros((nq, 2, 3))
    o, lse = oracle.attn_fwd_qk(q, k, v, True, 1.0)
    for i in range(nq):
        cnt = nk - nq + 1 + i
        np.testing.assert_allclose(lse[:, i], np.full(2, math.log(cnt)), atol=1e-14)
        np.testing.assert_allclose(o[i], v[:cnt].mean(axis=0), atol=1e-14)
    nq, nk = 9, 4  # the first 5 queries see nothing
    _, k, v, _ = _seq(nq, nk, 2, 2, 3, seed=4)
    o, lse = oracle.attn_fwd_qk(np.zeros((nq, 2, 3)), k, v, True, 1.0)
    assert np.all(np.isneginf(lse[:, :5])) and np.all(o[:5] == 0)
    np.testing.assert_allclose(lse[:, 5:], np.tile(np.log(np.arange(1, 5)), (2, 1)), atol=1e-14)


def _loss(q, k, v, do, causal, scale):
    o, _ = oracle.attn_fwd_qk(q, k, v, causal, scale)
    return float(np.sum(o * do))


@pytest.mark.parametrize("nq,nk", [(3, 6), (6, 3), (4, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_qk_matches_finite_differences(nq, nk, causal):
    q, k, v, do = _seq(nq, nk, 4, 2, 3, seed=7 * nq + nk)
    scale, h = 0.8, 1e-6
    dq, dk, dv = oracle.attn_bwd_qk(q, k, v, do, causal, scale)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            fp = _loss(args["q"], args["k"], args["v"], do, causal, scale)
            args[name] = xm
            fm = _loss(args["q"], args["k"], args["v"], do, causal, scale)
            num[idx] = (fp - fm) / (2 * h)
        err = np.linalg.norm(g - num) / max(np.linalg.norm(num), 1e-30)
        assert err < 1e-6, (name, err)


def test_empty_rows_have_zero_gradient():
    """Queries that see no key (Nq > Nk under the mask) change nothing: their dQ is 0
    and perturbing them leaves the loss unchanged."""
    q, k, v, do = _seq(7, 3, 2, 1, 4, seed=9)
    dq, _, _ = oracle.attn_bwd_qk(q, k, v, do, True, 1.0)
    assert np.all(dq[:4] == 0)
    q2 = q.copy()
    q2[:4] += 3.0
    assert _loss(q, k, v, do, True, 1.0) == _loss(q2, k, v, do, True, 1.0)


def test_varlen_packing_and_padding():
    """The packed batch equals its sequences evaluated one by one; a padded batch
    (seqused < segment length) leaves the padding rows unwritten (NaN)."""
    rng = np.random.default_rng(12)
    lq, lk = [3, 0, 5, 1], [4, 2, 5, 6]
    cu_q, cu_k = np.concatenate([[0], np.cumsum(lq)]), np.concatenate([[0], np.cumsum(lk)])
    q, do = _rand((cu_q[-1], 4, 3), rng), _rand((cu_q[-1], 4, 3), rng)
    k, v = _rand((cu_k[-1], 2, 3), rng), _rand((cu_k[-1], 2, 3), rng)
    for causal in (False, True):
        o, lse = oracle.attn_varlen_fwd_ref(q, k, v, cu_q, cu_k, causal, 0.6)
        dq, dk, dv = oracle.attn_varlen_bwd_ref(q, k, v, do, cu_q, cu_k, causal, 0.6)
        for b in range(4):
            sq, sk = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
            ob, lb = oracle.attn_fwd_qk(q[sq], k[sk], v[sk], causal, 0.6)
            np.testing.assert_array_equal(o[sq], ob)
            np.testing.assert_array_equal(lse[:, sq], lb)
            g = oracle.attn_bwd_qk(q[sq], k[sk], v[sk], do[sq], causal, 0.6)
            np.testing.assert_array_equal(dq[sq], g[0])
            np.testing.assert_array_equal(dk[sk], g[1])
            np.testing.assert_array_equal(dv[sk], g[2])
    # padded: segments of 6 rows, 4 and 2 real
    cu = np.array([0, 6, 12])
    qp, kp, vp = _rand((12, 2, 3), rng), _rand((12, 2, 3), rng), _rand((12, 2, 3), rng)
    used = np.array([4, 2])
    o, lse = oracle.attn_varlen_fwd_ref(qp, kp, vp, cu, cu, True, 1.0, used, used)
    assert np.all(np.isnan(o[4:6])) and np.all(np.isnan(o[8:12])) and np.all(np.isnan(lse[:, 4:6]))
    ob, _ = oracle.attn_fwd_qk(qp[6:8], kp[6:8], vp[6:8], True, 1.0)
    np.testing.assert_array_equal(o[6:8], ob)


def test_planted_top_left_mask_is_caught(monkeypatch):
    """Plant a top-left-aligned mask in the oracle: the decode-shape pin must fail."""
    def top_left(nq, nk, causal):
        if not causal:
            return np.ones((nq, nk), dtype=bool)
        return np.arange(nk)[None, :] <= np.arange(nq)[:, None]

    monkeypatch.setattr(ov, "visible", top_left)
    with pytest.raises(AssertionError):
        test_single_query_sees_every_key_under_the_mask()


@pytest.mark.parametrize("cuts", [(0, 5, 13), (0, 1, 2, 3, 13), (0, 13), (0, 0, 7, 7, 13)])
def test_split_keys_merge_by_lse_weights(cuts):
    """Splitting the keys into consecutive ranges and merging the per-range results with
    lse = ln sum_s e^{lse_s} and O = sum_s e^{lse_s - lse} O_s gives attention over all
    keys: the identity split-key decoding relies on.  Empty ranges carry lse = -inf and
    weight 0.  Checked against the whole-range oracle and scalar brute force."""
    q, k, v, _ = _seq(3, 13, 4, 2, 5, seed=21)
    scale = 0.45
    parts = [oracle.attn_fwd_qk(q, k[a:b], v[a:b], False, scale) for a, b in zip(cuts[:-1], cuts[1:])]
    lses = np.stack([pl for _, pl in parts])  # [S, Hq, Nq]
    mx = np.max(lses, axis=0)
    lse = mx + np.log(np.sum(np.exp(lses - mx), axis=0))
    w = np.exp(lses - lse)  # [S, Hq, Nq]
    o = sum(np.transpose(w[s_], (1, 0))[:, :, None] * parts[s_][0] for s_ in range(len(parts)))
    ro, rl = oracle.attn_fwd_qk(q, k, v, False, scale)
    np.testing.assert_allclose(lse, rl, atol=1e-12)
    np.testing.assert_allclose(o, ro, atol=1e-12)
    bo, bl = oracle.brute_force_fwd_qk(q, k, v, False, scale)
    np.testing.assert_allclose(o, bo, atol=1e-12)
    np.testing.assert_allclose(lse, bl, atol=1e-12)
