"""Pins for the fp64 oracle, against what the pages and the mathematics fix.

None of these re-types the oracle's own formula: each compares it with an
independent computation (scalar brute force, a library softmax, finite
differences) or with a closed form / invariant the definition implies.
"""

import math

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import attention as oa
from exact_attention_38_gb300.inputs import make_inputs, to_f64


def _case(B, N, Hq, Hkv, d, seed, dtype="fp16"):
    t = make_inputs(B, N, Hq, Hkv, d, dtype=dtype, seed=seed)
    return {k_: to_f64(v_) for k_, v_ in t.items()}


SHAPES = [  # B, N, Hq, Hkv, d
    (1, 7, 2, 2, 5),
    (2, 9, 4, 2, 3),
    (1, 1, 1, 1, 4),
    (1, 16, 3, 1, 8),
]


# ---------------------------------------------------------------- (vii) brute force

@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_matches_scalar_brute_force(shape, causal):
    B, N, Hq, Hkv, d = shape
    x = _case(B, N, Hq, Hkv, d, seed=11)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attn_fwd_ref(x["q"], x["k"], x["v"], causal, scale)
    ob, lseb = oracle.brute_force_fwd(x["q"], x["k"], x["v"], causal, scale)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lseb, rtol=0, atol=1e-12)


def test_hand_worked_example():
    """N=2, d=1, scale=1: q=(0,1), k=(0,ln3), v=(1,5), dO=(1,1), worked by hand.

    Non-causal row 0 sees scores (0,0) -> P=(1/2,1/2), O=3, lse=ln2; row 1 sees
    (0,ln3) -> P=(1/4,3/4), O=4, lse=ln4.  Causal row 0 sees key 0 only.
    Backward (non-causal): D=(3,4), dS=((-1,1),(-3/4,3/4)), dQ=(ln3, 3/4 ln3),
    dK=(-3/4, 3/4), dV=(3/4, 5/4).
    """
    ln3 = math.log(3.0)
    q = np.array([0.0, 1.0]).reshape(1, 2, 1, 1)
    k = np.array([0.0, ln3]).reshape(1, 2, 1, 1)
    v = np.array([1.0, 5.0]).reshape(1, 2, 1, 1)
    do = np.ones((1, 2, 1, 1))
    o, lse = oracle.attn_fwd_ref(q, k, v, False, 1.0)
    np.testing.assert_allclose(o.ravel(), [3.0, 4.0], atol=1e-14)
    np.testing.assert_allclose(lse.ravel(), [math.log(2), math.log(4)], atol=1e-14)
    oc, lsec = oracle.attn_fwd_ref(q, k, v, True, 1.0)
    np.testing.assert_allclose(oc.ravel(), [1.0, 4.0], atol=1e-14)
    np.testing.assert_allclose(lsec.ravel(), [0.0, math.log(4)], atol=1e-14)
    g = oracle.attn_bwd_ref(q, k, v, do, False, 1.0)
    np.testing.assert_allclose(g["D"].ravel(), [3.0, 4.0], atol=1e-14)
    np.testing.assert_allclose(g["dq"].ravel(), [ln3, 0.75 * ln3], atol=1e-14)
    np.testing.assert_allclose(g["dk"].ravel(), [-0.75, 0.75], atol=1e-14)
    np.testing.assert_allclose(g["dv"].ravel(), [0.75, 1.25], atol=1e-14)


def test_matches_library_softmax_and_logsumexp():
    """Special case that reduces to a library routine: one head, P = softmax(S)."""
    x = _case(1, 33, 1, 1, 16, seed=3)
    scale = 0.25
    for causal in (False, True):
        s = scale * x["q"][0, :, 0, :] @ x["k"][0, :, 0, :].T
        if causal:
            s = np.where(np.triu(np.ones_like(s, dtype=bool), 1), -np.inf, s)
        p_lib = scipy.special.softmax(s, axis=1)
        lse_lib = scipy.special.logsumexp(s, axis=1)
        o, lse = oracle.attn_fwd_ref(x["q"], x["k"], x["v"], causal, scale)
        np.testing.assert_allclose(oracle.attn_probs(x["q"], x["k"], causal, scale, 0, 0), p_lib,
                                   atol=1e-13)
        np.testing.assert_allclose(lse[0, 0], lse_lib, atol=1e-12)
        np.testing.assert_allclose(o[0, :, 0, :], p_lib @ x["v"][0, :, 0, :], atol=1e-12)


# ----------------------------------------------- (i) online recurrence == full softmax

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block", [1, 3, 16, 40])
def test_online_recurrence_equals_full_softmax(causal, block):
    x = _case(2, 40, 4, 2, 8, seed=5)
    scale = 1.0 / math.sqrt(8)
    o, lse = oracle.attn_fwd_ref(x["q"], x["k"], x["v"], causal, scale)
    oo, lseo = oracle.attn_online_ref(x["q"], x["k"], x["v"], causal, scale, block)
    np.testing.assert_allclose(oo, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lseo, lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_blockwise_normalise_then_sum_is_not_attention(causal):
    """Negative control: per-block softmax summed over blocks is a different result."""
    x = _case(1, 40, 2, 2, 8, seed=6)
    scale = 1.0 / math.sqrt(8)
    o, _ = oracle.attn_fwd_ref(x["q"], x["k"], x["v"], causal, scale)
    bad = oracle.attn_blockwise_normalised_sum(x["q"], x["k"], x["v"], causal, scale, 16)
    assert np.max(np.abs(bad - o)) > 1e-1
    # with a single block it *is* the same computation
    one = oracle.attn_blockwise_normalised_sum(x["q"], x["k"], x["v"], causal, scale, 40)
    np.testing.assert_allclose(one, o, atol=1e-12)


# ---------------------------------------------------------- (ii)-(v) closed forms

@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    x = _case(1, 50, 2, 1, 16, seed=7)
    for h in range(2):
        p = oracle.attn_probs(x["q"], x["k"], causal, 0.3, 0, h)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
        assert np.all(p >= 0)
        if causal:
            assert np.all(p[np.triu_indices(50, 1)] == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_v_ones_gives_o_ones(causal):
    t = make_inputs(1, 37, 2, 2, 8, dtype="bf16", seed=8, special="v_ones")
    x = {k_: to_f64(v_) for k_, v_ in t.items()}
    o, _ = oracle.attn_fwd_ref(x["q"], x["k"], x["v"], causal, 0.35)
    np.testing.assert_allclose(o, 1.0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_q_zero_gives_mean_of_visible_v(causal):
    t = make_inputs(2, 21, 4, 2, 8, dtype="bf16", seed=9, special="q_zero")
    x = {k_: to_f64(v_) for k_, v_ in t.items()}
    o, lse = oracle.attn_fwd_ref(x["q"], x["k"], x["v"], causal, 0.35)
    N = 21
    for b in range(2):
        for h in range(4):
            v = x["v"][b, :, h // 2, :]
            for i in range(N):
                cnt = i + 1 if causal else N
                np.testing.assert_allclose(o[b, i, h], v[:cnt].mean(axis=0), atol=1e-13)
                assert abs(lse[b, h, i] - math.log(cnt)) < 1e-13


def test_causal_row_zero_is_v0():
    x = _case(2, 19, 4, 2, 8, seed=10)
    scale = 1.0 / math.sqrt(8)
    o, lse = oracle.attn_fwd_ref(x["q"], x["k"], x["v"], True, scale)
    for b in range(2):
        for h in range(4):
            g = h // 2
            np.testing.assert_allclose(o[b, 0, h], x["v"][b, 0, g], atol=1e-14)
            assert abs(lse[b, h, 0] - scale * float(x["q"][b, 0, h] @ x["k"][b, 0, g])) < 1e-13


# ------------------------------------------------------------------ invariances

def test_noncausal_key_permutation_invariance():
    x = _case(1, 30, 2, 1, 8, seed=12)
    perm = np.random.default_rng(0).permutation(30)
    o, lse = oracle.attn_fwd_ref(x["q"], x["k"], x["v"], False, 0.3)
    op, lsep = oracle.attn_fwd_ref(x["q"], x["k"][:, perm], x["v"][:, perm], False, 0.3)
    np.testing.assert_allclose(op, o, atol=1e-12)
    np.testing.assert_allclose(lsep, lse, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal):
    """Adding u to every key leaves O unchanged and shifts lse_i by scale*<q_i,u>."""
    x = _case(1, 25, 2, 2, 8, seed=13)
    u = np.linspace(-1, 1, 8)
    o, lse = oracle.attn_fwd_ref(x["q"], x["k"], x["v"], causal, 0.3)
    o2, lse2 = oracle.attn_fwd_ref(x["q"], x["k"] + u, x["v"], causal, 0.3)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    shift = 0.3 * np.einsum("bnhd,d->bhn", x["q"], u)
    np.testing.assert_allclose(lse2, lse + shift, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_mha_on_repeated_kv(causal):
    x = _case(2, 17, 6, 2, 4, seed=14)
    k_rep = np.repeat(x["k"], 3, axis=2)
    v_rep = np.repeat(x["v"], 3, axis=2)
    o, lse = oracle.attn_fwd_ref(x["q"], x["k"], x["v"], causal, 0.5)
    o2, lse2 = oracle.attn_fwd_ref(x["q"], k_rep, v_rep, causal, 0.5)
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, atol=1e-13)
    g = oracle.attn_bwd_ref(x["q"], x["k"], x["v"], x["do"], causal, 0.5)
    g2 = oracle.attn_bwd_ref(x["q"], k_rep, v_rep, x["do"], causal, 0.5)
    np.testing.assert_allclose(g["dq"], g2["dq"], atol=1e-12)
    np.testing.assert_allclose(g["dk"], g2["dk"].reshape(2, 17, 2, 3, 4).sum(axis=3), atol=1e-12)
    np.testing.assert_allclose(g["dv"], g2["dv"].reshape(2, 17, 2, 3, 4).sum(axis=3), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_sum_identities(causal):
    """sum_j dK_j = 0 (rows of dS sum to 0); sum_j dV_j = sum over the group of sum_i dO_i."""
    x = _case(2, 23, 4, 2, 8, seed=15)
    g = oracle.attn_bwd_ref(x["q"], x["k"], x["v"], x["do"], causal, 0.3)
    np.testing.assert_allclose(g["dk"].sum(axis=1), 0.0, atol=1e-12)
    do_sum = x["do"].sum(axis=1).reshape(2, 2, 2, 8).sum(axis=2)
    np.testing.assert_allclose(g["dv"].sum(axis=1), do_sum, atol=1e-12)
    # D_i = <dO_i, O_i>
    np.testing.assert_allclose(g["D"], np.einsum("bnhd,bnhd->bhn", x["do"], g["o"]), atol=1e-13)


# ----------------------------------------------------- (vi) finite differences

def _loss(q, k, v, do, causal, scale):
    o, _ = oa.attn_fwd_ref(q, k, v, causal, scale)
    return float(np.sum(o * do))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 9, 2, 1, 4), (2, 5, 2, 2, 3)])
def test_gradients_match_central_finite_differences(causal, shape):
    B, N, Hq, Hkv, d = shape
    x = _case(B, N, Hq, Hkv, d, seed=16)
    scale = 0.6
    g = oracle.attn_bwd_ref(x["q"], x["k"], x["v"], x["do"], causal, scale)
    h = 1e-6
    for name in ("q", "k", "v"):
        base = x[name]
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args = dict(x)
            plus = base.copy()
            plus[idx] += h
            minus = base.copy()
            minus[idx] -= h
            args[name] = plus
            fp = _loss(args["q"], args["k"], args["v"], x["do"], causal, scale)
            args[name] = minus
            fm = _loss(args["q"], args["k"], args["v"], x["do"], causal, scale)
            num[idx] = (fp - fm) / (2 * h)
        ana = g["d" + name]
        rel = np.linalg.norm(ana - num) / np.linalg.norm(num)
        assert rel < 1e-6, (name, rel)


# ------------------------------------------------------ row-subset evaluators

@pytest.mark.parametrize("causal", [False, True])
def test_row_subset_evaluators_match_full(causal):
    x = _case(2, 45, 4, 2, 8, seed=17)
    scale = 0.4
    o, lse = oracle.attn_fwd_ref(x["q"], x["k"], x["v"], causal, scale)
    g = oracle.attn_bwd_ref(x["q"], x["k"], x["v"], x["do"], causal, scale)
    rows = np.array([0, 3, 17, 44, 44, 20])
    for b, h in [(0, 0), (1, 3)]:
        orow, lrow = oracle.attn_fwd_rows(x["q"], x["k"], x["v"], causal, scale, b, h, rows)
        np.testing.assert_allclose(orow, o[b, rows, h], atol=1e-13)
        np.testing.assert_allclose(lrow, lse[b, h, rows], atol=1e-13)
        dqr = oracle.attn_bwd_dq_rows(x["q"], x["k"], x["v"], x["do"], causal, scale, b, h, rows)
        np.testing.assert_allclose(dqr, g["dq"][b, rows, h], atol=1e-12)
    for b, hk in [(0, 0), (1, 1)]:
        dkr, dvr = oracle.attn_bwd_kv_rows(x["q"], x["k"], x["v"], x["do"], causal, scale, b, hk, rows)
        np.testing.assert_allclose(dkr, g["dk"][b, rows, hk], atol=1e-12)
        np.testing.assert_allclose(dvr, g["dv"][b, rows, hk], atol=1e-12)


# ------------------------------------------- the pins catch planted mistakes

def _planted_mask_off_by_one(q_rows, k_all, rows, causal, scale):
    s = scale * (q_rows @ k_all.T)
    if causal:
        cols = np.arange(k_all.shape[0])
        s = np.where(cols[None, :] >= np.asarray(rows)[:, None], -np.inf, s)  # drops the diagonal
        s = np.where(np.all(np.isneginf(s), axis=1, keepdims=True), 0.0, s)
    return s


def _planted_scale_dropped(q_rows, k_all, rows, causal, scale):
    return _ORIG_SCORES(q_rows, k_all, rows, causal, 1.0)


_ORIG_SCORES = oa._row_scores


@pytest.mark.parametrize("mutant,causal", [(_planted_mask_off_by_one, True), (_planted_scale_dropped, False)])
def test_planted_mistakes_fail_the_pins(monkeypatch, mutant, causal):
    x = _case(1, 7, 2, 2, 5, seed=11)
    ob, lseb = oracle.brute_force_fwd(x["q"], x["k"], x["v"], causal, 0.45)
    monkeypatch.setattr(oa, "_row_scores", mutant)
    o, lse = oracle.attn_fwd_ref(x["q"], x["k"], x["v"], causal, 0.45)
    assert np.max(np.abs(o - ob)) > 1e-3 or np.max(np.abs(lse - lseb)) > 1e-3


def test_planted_gradient_sign_error_fails_finite_differences(monkeypatch):
    x = _case(1, 5, 1, 1, 3, seed=18)
    g = oracle.attn_bwd_ref(x["q"], x["k"], x["v"], x["do"], False, 0.6)
    bad_dk = -g["dk"]  # a sign slip in dS^T Q
    h = 1e-6
    num = np.zeros_like(x["k"])
    for idx in np.ndindex(*x["k"].shape):
        kp = x["k"].copy()
        kp[idx] += h
        km = x["k"].copy()
        km[idx] -= h
        num[idx] = (_loss(x["q"], kp, x["v"], x["do"], False, 0.6)
                    - _loss(x["q"], km, x["v"], x["do"], False, 0.6)) / (2 * h)
    assert np.linalg.norm(g["dk"] - num) / np.linalg.norm(num) < 1e-6
    assert np.linalg.norm(bad_dk - num) / np.linalg.norm(num) > 1.0
