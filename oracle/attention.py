"""fp64 CPU oracle for exact scaled-dot-product attention (forward and backward).

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call or run this
module: only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it. It shares no code, constant or
helper with the CUDA path; it takes numpy arrays and returns numpy arrays.

What it computes, and where that is said:

* "FlashAttention-2: atención eficiente en GPU para contextos largos",
  section "Bloques pequeños, normalización global" (and the same section of its
  Chinese edition, "分块处理仍需保持全局归一化"): the tiled method keeps *exact*
  attention; only the floating-point order of operations differs, so outputs and
  gradients are compared within a tolerance.  The oracle is therefore the plain
  definition, evaluated in fp64:

      s_ij   = scale * <q_i, k_j>              (j visible to i)
      lse_i  = ln sum_j exp(s_ij)
      P_ij   = exp(s_ij - lse_i)
      O_i    = sum_j P_ij v_j

  Causal masking (section "Tres mejoras en la utilización de la GPU"): key j is
  visible to query i iff j <= i (queries and keys have the same length N, so the
  mask is aligned at the top-left corner; reading, the pages give no formula).

* Backward: the pages only say gradients are compared within tolerance; the
  gradient of L = sum(dO * O) is the textbook closed form

      dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij = <dO_i, O_i>,
      dS = P * (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q.

* Grouped-query attention ("FlashAttention-T: Optimización GPU para LLMs
  Escalables", section "Innovaciones técnicas frente a FlashAttention original"):
  query head h reads key/value head h // (Hq // Hkv) (reading: contiguous groups);
  dK and dV of a key/value head sum over the query heads of its group.

* ``attn_online_ref`` is the running-max / running-sum recurrence the pages
  describe in words ("Bloques pequeños, normalización global": statistics and
  partial outputs are updated and rescaled block by block so the final result is
  globally normalised).  It exists only to prove, in the tests, that this
  recurrence equals the plain definition.  ``attn_blockwise_normalised_sum`` is
  the computation the same section says is *not* equivalent (normalise each block
  by itself and sum); it is a negative control.

Layouts: q, o, dq, do are [B, N, Hq, d]; k, v, dk, dv are [B, N, Hkv, d]; lse is
[B, Hq, N].  All arithmetic is float64.  Rows are evaluated independently (a row
of attention depends only on its own query), so functions that take a subset of
rows compute exactly the same numbers as the full evaluation for those rows.
"""

from __future__ import annotations

import math

import numpy as np

# Rows evaluated per matrix product; only bounds memory, each row is still the
# plain definition above.
_ROW_CHUNK = 512


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _kv_head(h: int, hq: int, hkv: int) -> int:
    if hq % hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return h // (hq // hkv)


def _row_scores(q_rows, k_all, rows, causal, scale):
    """Scaled scores of the given query rows against every key, masked entries -inf."""
    s = scale * (q_rows @ k_all.T)
    if causal:
        cols = np.arange(k_all.shape[0])
        s = np.where(cols[None, :] > np.asarray(rows)[:, None], -np.inf, s)
    return s


def _row_lse(s):
    m = np.max(s, axis=1, keepdims=True)
    return (m + np.log(np.sum(np.exp(s - m), axis=1, keepdims=True)))[:, 0]


# --------------------------------------------------------------------------- forward

def attn_fwd_rows(q, k, v, causal, scale, b, h, rows):
    """O and lse for query rows ``rows`` of batch ``b``, query head ``h``.

    With the causal mask a chunk of rows only reads keys up to its last row (the
    probabilities of later keys are exactly zero).  Returns (o [len(rows), d],
    lse [len(rows)]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    hkv = _kv_head(h, q.shape[2], k.shape[2])
    rows = np.asarray(rows, dtype=np.int64)
    kb, vb = k[b, :, hkv, :], v[b, :, hkv, :]
    o = np.empty((rows.size, q.shape[3]))
    lse = np.empty(rows.size)
    for c0 in range(0, rows.size, _ROW_CHUNK):
        r = rows[c0:c0 + _ROW_CHUNK]
        kmax = int(r.max()) + 1 if causal else kb.shape[0]
        s = _row_scores(q[b, r, h, :], kb[:kmax], r, causal, scale)
        l = _row_lse(s)
        p = np.exp(s - l[:, None])
        o[c0:c0 + r.size] = p @ vb[:kmax]
        lse[c0:c0 + r.size] = l
    return o, lse


def attn_fwd_ref(q, k, v, causal, scale):
    """Full forward: O [B,N,Hq,d] and lse [B,Hq,N], both float64."""
    q = _f64(q)
    B, N, Hq, d = q.shape
    o = np.empty((B, N, Hq, d))
    lse = np.empty((B, Hq, N))
    rows = np.arange(N)
    for b in range(B):
        for h in range(Hq):
            o[b, :, h, :], lse[b, h, :] = attn_fwd_rows(q, k, v, causal, scale, b, h, rows)
    return o, lse


def attn_probs(q, k, causal, scale, b, h):
    """The full probability matrix P [N, N] of one (batch, query head)."""
    q, k = _f64(q), _f64(k)
    hkv = _kv_head(h, q.shape[2], k.shape[2])
    rows = np.arange(q.shape[1])
    s = _row_scores(q[b, :, h, :], k[b, :, hkv, :], rows, causal, scale)
    return np.exp(s - _row_lse(s)[:, None])


# -------------------------------------------------------------------------- backward

def attn_bwd_ref(q, k, v, do, causal, scale):
    """Gradients of L = sum(dO * O) with respect to q, k, v (float64).

    Returns dict with dq, dk, dv, o, lse and D (= rowsum(dO * O), [B,Hq,N]).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    o = np.empty_like(q)
    lse = np.empty((B, Hq, N))
    D = np.empty((B, Hq, N))
    rows = np.arange(N)
    for b in range(B):
        for h in range(Hq):
            g = _kv_head(h, Hq, Hkv)
            kb, vb = k[b, :, g, :], v[b, :, g, :]
            s = _row_scores(q[b, :, h, :], kb, rows, causal, scale)
            l = _row_lse(s)
            p = np.exp(s - l[:, None])
            ob = p @ vb
            dob = do[b, :, h, :]
            dp = dob @ vb.T
            Di = np.sum(dob * ob, axis=1)
            ds = p * (dp - Di[:, None])
            dq[b, :, h, :] = scale * (ds @ kb)
            dk[b, :, g, :] += scale * (ds.T @ q[b, :, h, :])
            dv[b, :, g, :] += p.T @ dob
            o[b, :, h, :] = ob
            lse[b, h, :] = l
            D[b, h, :] = Di
    return {"dq": dq, "dk": dk, "dv": dv, "o": o, "lse": lse, "D": D}


def attn_bwd_dq_rows(q, k, v, do, causal, scale, b, h, rows):
    """dQ for query rows ``rows`` of (b, h): [len(rows), d].

    Row i of dQ needs only row i of P and dP and D_i = <dO_i, O_i>, all of which
    come from query row i alone.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    g = _kv_head(h, q.shape[2], k.shape[2])
    kb, vb = k[b, :, g, :], v[b, :, g, :]
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((rows.size, q.shape[3]))
    for c0 in range(0, rows.size, _ROW_CHUNK):
        r = rows[c0:c0 + _ROW_CHUNK]
        kmax = int(r.max()) + 1 if causal else kb.shape[0]
        s = _row_scores(q[b, r, h, :], kb[:kmax], r, causal, scale)
        p = np.exp(s - _row_lse(s)[:, None])
        dob = do[b, r, h, :]
        Di = np.sum(dob * (p @ vb[:kmax]), axis=1)
        ds = p * (dob @ vb[:kmax].T - Di[:, None])
        out[c0:c0 + r.size] = scale * (ds @ kb[:kmax])
    return out


def attn_bwd_kv_rows(q, k, v, do, causal, scale, b, hkv, key_rows):
    """dK and dV for key rows ``key_rows`` of (b, key/value head ``hkv``).

    Column j of P and dS over the query rows that see key j, for every query head
    in the group, is needed: all rows without the mask (cost ~2*N^2*d per query
    head), rows i >= min(key_rows) with it.  Returns (dk [len, d], dv [len, d]).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    N, Hq = q.shape[1], q.shape[2]
    Hkv = k.shape[2]
    grp = Hq // Hkv
    kb, vb = k[b, :, hkv, :], v[b, :, hkv, :]
    key_rows = np.asarray(key_rows, dtype=np.int64)
    dk = np.zeros((key_rows.size, k.shape[3]))
    dv = np.zeros((key_rows.size, v.shape[3]))
    first = int(key_rows.min()) if causal else 0
    for h in range(hkv * grp, (hkv + 1) * grp):
        for c0 in range(first, N, _ROW_CHUNK):
            r = np.arange(c0, min(N, c0 + _ROW_CHUNK))
            kmax = max(int(r.max()), int(key_rows.max())) + 1 if causal else N
            s = _row_scores(q[b, r, h, :], kb[:kmax], r, causal, scale)
            p = np.exp(s - _row_lse(s)[:, None])
            dob = do[b, r, h, :]
            Di = np.sum(dob * (p @ vb[:kmax]), axis=1)
            pj = p[:, key_rows]
            dsj = pj * (dob @ vb[key_rows].T - Di[:, None])
            dv += pj.T @ dob
            dk += scale * (dsj.T @ q[b, r, h, :])
    return dk, dv


# ------------------------------------------------- the block recurrence (invariant i)

def attn_online_ref(q, k, v, causal, scale, block_n):
    """Forward by the online-softmax recurrence over key blocks of ``block_n`` keys.

    For each key block B_t (in order): m' = max(m, rowmax S_t),
    l' = l*exp(m - m') + rowsum exp(S_t - m'), O' = O*exp(m - m') + exp(S_t - m') V_t,
    and finally O / l, lse = m + ln l.  Returns (o, lse) like ``attn_fwd_ref``.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, Hq, d = q.shape
    o = np.empty((B, N, Hq, d))
    lse = np.empty((B, Hq, N))
    rows = np.arange(N)
    for b in range(B):
        for h in range(Hq):
            g = _kv_head(h, Hq, k.shape[2])
            qb = q[b, :, h, :]
            m = np.full(N, -np.inf)
            l = np.zeros(N)
            acc = np.zeros((N, d))
            for j0 in range(0, N, block_n):
                cols = np.arange(j0, min(N, j0 + block_n))
                s = scale * (qb @ k[b, cols, g, :].T)
                if causal:
                    s = np.where(cols[None, :] > rows[:, None], -np.inf, s)
                m_new = np.maximum(m, np.max(s, axis=1))
                # rows whose every key so far is masked keep m = -inf; exp(-inf - -inf)
                # is undefined, and such a row has nothing to rescale yet.
                alpha = np.where(np.isneginf(m_new), 1.0, np.exp(m - m_new))
                p = np.where(np.isneginf(m_new)[:, None], 0.0, np.exp(s - m_new[:, None]))
                l = l * alpha + np.sum(p, axis=1)
                acc = acc * alpha[:, None] + p @ v[b, cols, g, :]
                m = m_new
            o[b, :, h, :] = acc / l[:, None]
            lse[b, h, :] = m + np.log(l)
    return o, lse


def attn_blockwise_normalised_sum(q, k, v, causal, scale, block_n):
    """NEGATIVE CONTROL: softmax each key block by itself, then add the block outputs.

    The pages say this is not the same computation as attention; the tests check
    that it differs from ``attn_fwd_ref`` whenever there is more than one block.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, Hq, d = q.shape
    o = np.zeros((B, N, Hq, d))
    rows = np.arange(N)
    for b in range(B):
        for h in range(Hq):
            g = _kv_head(h, Hq, k.shape[2])
            for j0 in range(0, N, block_n):
                cols = np.arange(j0, min(N, j0 + block_n))
                s = scale * (q[b, :, h, :] @ k[b, cols, g, :].T)
                if causal:
                    s = np.where(cols[None, :] > rows[:, None], -np.inf, s)
                m = np.max(s, axis=1, keepdims=True)
                ok = ~np.isneginf(m)
                e = np.where(ok, np.exp(s - np.where(ok, m, 0.0)), 0.0)
                den = np.sum(e, axis=1, keepdims=True)
                o[b, :, h, :] += np.where(ok, e / np.where(den > 0, den, 1.0), 0.0) @ v[b, cols, g, :]
    return o


# ------------------------------------------------------------ brute force (vii)

def brute_force_fwd(q, k, v, causal, scale):
    """Scalar Python loops over every (b, h, i, j); tiny shapes only.

    Independent of numpy's matrix routines: dot products and sums are done with
    ``math.fsum`` on Python floats.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    o = np.zeros((B, N, Hq, d))
    lse = np.zeros((B, Hq, N))
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            for i in range(N):
                vis = [j for j in range(N) if not (causal and j > i)]
                s = [scale * math.fsum(float(q[b, i, h, c]) * float(k[b, j, g, c]) for c in range(d))
                     for j in vis]
                mx = max(s)
                z = math.fsum(math.exp(x - mx) for x in s)
                lse[b, h, i] = mx + math.log(z)
                for c in range(d):
                    o[b, i, h, c] = math.fsum(math.exp(x - mx) / z * float(v[b, j, g, c])
                                              for x, j in zip(s, vis))
    return o, lse
