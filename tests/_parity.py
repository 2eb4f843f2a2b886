"""Helpers for the GPU parity tests: run the CUDA path, compare with the oracle."""

import math

import numpy as np
import torch

from exact_attention_38_gb300.inputs import make_inputs, to_f64

# max-abs tolerance on O, dQ, dK, dV by input dtype; relative-norm bound on gradients
ATOL = {"fp16": 2e-3, "bf16": 1.6e-2}
GRAD_RELNORM = 1e-2
LSE_ATOL = 1e-3

# mantissa bits and smallest normal exponent of the 16-bit output formats
_FORMAT = {"bf16": (7, -126), "fp16": (10, -14)}

# (name, elements above the flat bound, elements compared, largest |ref| among them),
# one entry per comparison that had any; printed at the end of the session
FLAT_EXCESS = []


def to_gpu(t):
    return t.to("cuda", non_blocking=False).contiguous()


def gpu_forward(fa, x, causal, scale=None):
    q, k, v = to_gpu(x["q"]), to_gpu(x["k"]), to_gpu(x["v"])
    d = q.shape[-1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    fa.check_device_error()
    return (q, k, v), o, lse


def f64(t):
    return to_f64(t)


def half_ulp(x, out_dtype):
    """Half a unit in the last place of the 16-bit format `out_dtype` at |x| (the largest
    error of rounding an exact value x to nearest in that format)."""
    mant, emin = _FORMAT[out_dtype]
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(np.where(ax > 0, e, emin), emin)  # subnormals share the smallest step
    return np.ldexp(1.0, (e - mant - 1).astype(np.int64))


def assert_close(name, got, want, atol, out_dtype=None):
    """Max-abs bound on every element: `atol`, plus, when the values are outputs rounded
    to the 16-bit format `out_dtype`, half a unit in the last place of that format at the
    reference value.

    Reading of the bound (it names no magnitude): 1.6e-2 (bf16) and 2e-3 (fp16) are about
    one unit in the last place of the 16-bit format at magnitudes in [1, 2).  Above that
    the output's own final rounding grows with the value (a correctly rounded bf16 number
    in [4, 8) can be 2^-6 away from the exact value), so the bound allows exactly one more
    such rounding on top of the flat figure: atol + ulp(|ref|) / 2.  The number of
    elements that exceed the flat figure alone is recorded in FLAT_EXCESS.
    """
    got = np.asarray(got, dtype=np.float64)
    want = np.broadcast_to(np.asarray(want, dtype=np.float64), got.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    if got.size == 0:
        return 0.0
    err = np.abs(got - want)
    tol = atol + (half_ulp(want, out_dtype) if out_dtype is not None else 0.0)
    tol = np.broadcast_to(tol, err.shape)
    worst = int(np.argmax(err - tol))
    assert err.flat[worst] <= tol.flat[worst], (
        f"{name}: error {err.flat[worst]:.3e} > {tol.flat[worst]:.3e} at |ref|={abs(want.flat[worst]):.3f}")
    over = err > atol
    if over.any():
        FLAT_EXCESS.append((name, int(over.sum()), int(err.size), float(np.abs(want[over]).max())))
    return float(err.max())


def assert_relnorm(name, got, want, bound=GRAD_RELNORM):
    den = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(got - want)) / den if den > 0 else float(np.linalg.norm(got))
    assert rel <= bound, f"{name}: relative-norm error {rel:.3e} > {bound:.0e}"
    return rel


def sample_rows(N, count, seed):
    rng = np.random.default_rng(seed)
    rows = rng.choice(N, size=min(count, N), replace=False)
    # always include the first and last rows (causal row 0, ragged tail)
    return np.unique(np.concatenate([rows, [0, N - 1]]))


__all__ = ["make_inputs", "to_f64", "ATOL", "GRAD_RELNORM", "LSE_ATOL", "FLAT_EXCESS", "gpu_forward", "f64",
           "half_ulp", "assert_close", "assert_relnorm", "sample_rows", "to_gpu"]
