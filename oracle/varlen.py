"""fp64 CPU oracle for variable-length batches and unequal query / key lengths.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only the tests,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may use it, and it shares
nothing with the CUDA path.

What it computes:

* The same plain definition as ``oracle.attention`` ("FlashAttention-2: atención
  eficiente en GPU para contextos largos", section "Bloques pequeños,
  normalización global": the tiled method reaches exact attention), for one
  sequence whose query length Nq and key length Nk may differ.  The prefill /
  decode distinction of section "Cómo documentar una diferencia técnica" and the
  boundary handling named in "Tres mejoras en la utilización de la GPU" are where
  such shapes arise; the pages give no formula, so the readings are:

  - causal mask aligned at the bottom-right corner: query i sees key j iff
    j <= i + (Nk - Nq), so the last query sees every key (with Nq = Nk this is the
    usual j <= i);
  - a query that sees no key (Nk = 0, or i + Nk - Nq < 0 under the mask) has an
    empty softmax: its output row is 0, its log-sum-exp is ln 0 = -inf, and it
    contributes nothing to any gradient.

* A batch of such sequences packed along the token axis ("variable length"): the
  tokens of sequence b are rows [cu[b], cu[b] + len_b) of the packed tensors, with
  len_b = cu[b+1] - cu[b], or ``seqused[b]`` when given (a padded batch: sequence b
  owns rows [cu[b], cu[b+1]) but only the first seqused[b] are real).  Rows that no
  sequence covers are returned as NaN, meaning "not written".

Layouts: packed q, o, dq, do [total_q, Hq, d]; k, v, dk, dv [total_k, Hkv, d];
lse [Hq, total_q].  Per-sequence functions take q [Nq, Hq, d], k, v [Nk, Hkv, d]
and return lse [Hq, Nq].  Query head h reads key/value head h // (Hq // Hkv)
("FlashAttention-T: Optimización GPU para LLMs Escalables", section "Innovaciones
técnicas frente a FlashAttention original"; contiguous groups are a reading).
"""

from __future__ import annotations

import math

import numpy as np


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def visible(nq: int, nk: int, causal: bool) -> np.ndarray:
    """[nq, nk] boolean: query i sees key j (bottom-right-aligned causal mask)."""
    if not causal:
        return np.ones((nq, nk), dtype=bool)
    i = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    return j <= i + (nk - nq)


def _group(hq: int, hkv: int) -> int:
    if hkv <= 0 or hq % hkv != 0:
        raise ValueError("Hq must be a positive multiple of Hkv")
    return hq // hkv


def attn_fwd_qk(q, k, v, causal, scale):
    """One sequence: q [Nq,Hq,d], k/v [Nk,Hkv,d] -> (o [Nq,Hq,d], lse [Hq,Nq])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    nq, hq, d = q.shape
    nk, hkv = k.shape[0], k.shape[1]
    g = _group(hq, hkv)
    vis = visible(nq, nk, causal)
    o = np.zeros((nq, hq, v.shape[2]))
    lse = np.full((hq, nq), -np.inf)
    rows = vis.any(axis=1) if nk > 0 else np.zeros(nq, dtype=bool)
    for h in range(hq):
        kh, vh = k[:, h // g], v[:, h // g]
        s = np.where(vis, scale * (q[:, h] @ kh.T), -np.inf)
        for i in np.nonzero(rows)[0]:
            m = s[i].max()
            e = np.exp(s[i] - m)
            tot = e.sum()
            lse[h, i] = m + math.log(tot)
            o[i, h] = (e / tot) @ vh
    return o, lse


def attn_bwd_qk(q, k, v, do, causal, scale):
    """One sequence: gradients of L = sum(dO * O) -> (dq, dk, dv), shapes of q, k, v.

    dV = P^T dO, dP = dO V^T, D_i = <dO_i, O_i>, dS = P * (dP - D),
    dQ = scale * dS K, dK = scale * dS^T Q; rows with no visible key have P = 0.
    dK and dV of a key/value head sum over the query heads of its group.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    nq, hq, d = q.shape
    nk, hkv = k.shape[0], k.shape[1]
    g = _group(hq, hkv)
    vis = visible(nq, nk, causal)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    if nk == 0 or nq == 0:
        return dq, dk, dv
    for h in range(hq):
        kh, vh = k[:, h // g], v[:, h // g]
        s = np.where(vis, scale * (q[:, h] @ kh.T), -np.inf)
        p = np.zeros_like(s)
        for i in range(nq):
            if vis[i].any():
                e = np.exp(s[i] - s[i].max())
                p[i] = e / e.sum()
        o = p @ vh
        dp = do[:, h] @ vh.T
        dd = np.sum(do[:, h] * o, axis=1)
        ds = p * (dp - dd[:, None])
        dq[:, h] = scale * (ds @ kh)
        dk[:, h // g] += scale * (ds.T @ q[:, h])
        dv[:, h // g] += p.T @ do[:, h]
    return dq, dk, dv


def brute_force_fwd_qk(q, k, v, causal, scale):
    """Scalar loops with math.fsum (tiny shapes only): an independent evaluation of
    attn_fwd_qk used to pin it."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    nq, hq, d = q.shape
    nk, hkv, dv = k.shape[0], k.shape[1], v.shape[2]
    g = hq // hkv
    o = np.zeros((nq, hq, dv))
    lse = np.full((hq, nq), -np.inf)
    for h in range(hq):
        for i in range(nq):
            keys = [j for j in range(nk) if (not causal) or j - (nk - nq) <= i]
            if not keys:
                continue
            s = {j: scale * math.fsum(q[i, h, c] * k[j, h // g, c] for c in range(d)) for j in keys}
            m = max(s.values())
            z = math.fsum(math.exp(s[j] - m) for j in keys)
            lse[h, i] = m + math.log(z)
            for c in range(dv):
                o[i, h, c] = math.fsum(math.exp(s[j] - m) / z * v[j, h // g, c] for j in keys)
    return o, lse


def _spans(cu, seqused, b):
    start = int(cu[b])
    n = int(cu[b + 1]) - start if seqused is None else int(seqused[b])
    return start, n


def attn_varlen_fwd_ref(q, k, v, cu_q, cu_k, causal, scale, seqused_q=None, seqused_k=None):
    """Packed batch -> (o [total_q,Hq,d], lse [Hq,total_q]); uncovered rows are NaN."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    o = np.full((q.shape[0], q.shape[1], v.shape[2]), np.nan)
    lse = np.full((q.shape[1], q.shape[0]), np.nan)
    for b in range(len(cu_q) - 1):
        sq, nq = _spans(cu_q, seqused_q, b)
        sk, nk = _spans(cu_k, seqused_k, b)
        ob, lb = attn_fwd_qk(q[sq:sq + nq], k[sk:sk + nk], v[sk:sk + nk], causal, scale)
        o[sq:sq + nq] = ob
        lse[:, sq:sq + nq] = lb
    return o, lse


def attn_varlen_bwd_ref(q, k, v, do, cu_q, cu_k, causal, scale, seqused_q=None, seqused_k=None):
    """Packed batch -> (dq, dk, dv) in the packed layouts; uncovered rows are NaN."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    for b in range(len(cu_q) - 1):
        sq, nq = _spans(cu_q, seqused_q, b)
        sk, nk = _spans(cu_k, seqused_k, b)
        g = attn_bwd_qk(q[sq:sq + nq], k[sk:sk + nk], v[sk:sk + nk], do[sq:sq + nq], causal, scale)
        dq[sq:sq + nq], dk[sk:sk + nk], dv[sk:sk + nk] = g
    return dq, dk, dv

