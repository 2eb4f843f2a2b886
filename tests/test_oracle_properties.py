"""Randomised pins for the oracle (hypothesis): over random tiny shapes, GQA ratios,
masks and (for the unequal-length oracle) query / key length pairs, the vectorised
oracle must equal the scalar brute force, its gradients must match central finite
differences, and the softmax invariants must hold.  Skipped where hypothesis is not
installed."""

import math

import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")

import oracle  # noqa: E402

given, settings = hyp.given, hyp.settings


def _draw(seed, shape):
    return np.random.default_rng(seed).standard_normal(shape)


@settings(max_examples=40, deadline=None)
@given(n=st.integers(1, 10), d=st.integers(1, 6), hkv=st.integers(1, 2), g=st.integers(1, 3),
       causal=st.booleans(), seed=st.integers(0, 2**31 - 1), scale=st.floats(0.1, 2.0))
def test_fwd_equals_brute_force(n, d, hkv, g, causal, seed, scale):
    hq = hkv * g
    q, k, v = _draw(seed, (1, n, hq, d)), _draw(seed + 1, (1, n, hkv, d)), _draw(seed + 2, (1, n, hkv, d))
    o, lse = oracle.attn_fwd_ref(q, k, v, causal, scale)
    ob, lb = oracle.brute_force_fwd(q, k, v, causal, scale)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-11)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-11)


@settings(max_examples=40, deadline=None)
@given(nq=st.integers(0, 9), nk=st.integers(0, 9), d=st.integers(1, 5), g=st.integers(1, 3),
       causal=st.booleans(), seed=st.integers(0, 2**31 - 1))
def test_unequal_lengths_equal_brute_force(nq, nk, d, g, causal, seed):
    q, k, v = _draw(seed, (nq, 2 * g, d)), _draw(seed + 1, (nk, 2, d)), _draw(seed + 2, (nk, 2, d))
    o, lse = oracle.attn_fwd_qk(q, k, v, causal, 0.7)
    ob, lb = oracle.brute_force_fwd_qk(q, k, v, causal, 0.7)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-11)
    assert np.array_equal(np.isneginf(lse), np.isneginf(lb))
    fin = np.isfinite(lb)
    np.testing.assert_allclose(lse[fin], lb[fin], rtol=0, atol=1e-11)


@settings(max_examples=15, deadline=None)
@given(nq=st.integers(1, 5), nk=st.integers(1, 5), causal=st.booleans(), seed=st.integers(0, 2**31 - 1))
def test_unequal_length_gradients_match_finite_differences(nq, nk, causal, seed):
    q, k, v, do = (_draw(seed + i, s) for i, s in enumerate([(nq, 2, 3), (nk, 1, 3), (nk, 1, 3), (nq, 2, 3)]))
    scale, h = 0.9, 1e-6
    grads = oracle.attn_bwd_qk(q, k, v, do, causal, scale)

    def loss(qq, kk, vv):
        return float(np.sum(oracle.attn_fwd_qk(qq, kk, vv, causal, scale)[0] * do))

    for idx_arg, (x, gx) in enumerate(zip((q, k, v), grads)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            args = [q, k, v]
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args[idx_arg] = xp
            fp = loss(*args)
            args[idx_arg] = xm
            fm = loss(*args)
            num[idx] = (fp - fm) / (2 * h)
        den = max(np.linalg.norm(num), 1e-12)
        assert np.linalg.norm(gx - num) / den < 1e-5 or np.linalg.norm(gx - num) < 1e-8


@settings(max_examples=30, deadline=None)
@given(n=st.integers(1, 12), causal=st.booleans(), seed=st.integers(0, 2**31 - 1), shift=st.floats(-3, 3))
def test_probabilities_sum_to_one_and_shift_invariance(n, causal, seed, shift):
    q, k, v = _draw(seed, (1, n, 1, 4)), _draw(seed + 1, (1, n, 1, 4)), _draw(seed + 2, (1, n, 1, 4))
    p = oracle.attn_probs(q, k, causal, 0.5, 0, 0)
    np.testing.assert_allclose(p.sum(axis=1), np.ones(n), atol=1e-12)
    # adding a constant vector u to every key shifts each score row by scale * <q_i, u>:
    # O is unchanged and lse moves by exactly that amount
    u = np.full(4, shift)
    o1, l1 = oracle.attn_fwd_ref(q, k, v, causal, 0.5)
    o2, l2 = oracle.attn_fwd_ref(q, k + u, v, causal, 0.5)
    np.testing.assert_allclose(o1, o2, atol=1e-10)
    np.testing.assert_allclose(l2 - l1, 0.5 * (q[0, :, 0, :] @ u)[None, None, :], atol=1e-10)
