"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Plugins or engines that only get their input and output buffers, programs whose
allocator is frozen after start-up, and real-time paths cannot hand fa_bwd a
workspace; fa_bwd_noalloc uses a scratch array inside the library instead.  These tests
call it through the C ABI, twice in a row, and check each call's gradients against the
fp64 oracle and against fa_bwd with a caller-provided workspace, within the parity
tolerance.  The file name sorts last so that a run stopping at its first failure has run
every other test.  (The size limit is checked without a GPU in test_abi.py.)
"""

import ctypes
import math

import pytest

import oracle
from _parity import ATOL, assert_close, assert_relnorm, f64, make_inputs, to_gpu

pytestmark = pytest.mark.gpu


def _noalloc(fa):
    f = fa.lib.fa_bwd_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp] * 9 + [i] * 6 + [ctypes.c_float, i, vp]
    f.restype = i
    return f


@pytest.mark.parametrize("dtype,causal,shape", [
    ("bf16", True, (2, 700, 4, 2, 128)),
    ("fp16", False, (1, 333, 4, 4, 64)),
])
def test_noalloc_backward_matches_oracle_and_workspace_backward_twice(fa_lib, dtype, causal, shape):
    import torch

    fa = fa_lib
    f = _noalloc(fa)
    B, N, Hq, Hkv, d = shape
    x = make_inputs(B, N, Hq, Hkv, d, dtype=dtype, seed=31)
    q, k, v, do = (to_gpu(x[n]) for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    with_ws = fa.backward(do, q, k, v, o, lse, causal=causal, scale=scale)
    fa.check_device_error()
    with_ws = [f64(t.cpu()) for t in with_ws]
    xo = {n: f64(t) for n, t in x.items()}
    ref = oracle.attn_bwd_ref(xo["q"], xo["k"], xo["v"], xo["do"], causal, scale)
    stream = torch.cuda.current_stream().cuda_stream
    code = fa.FA_BF16 if dtype == "bf16" else fa.FA_FP16
    for call in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        st = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
               dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, N, d, int(causal), scale, code, stream)
        assert st == fa.FA_OK, fa.status_string(st)
        fa.check_device_error()
        for name, got, other in zip(("dq", "dk", "dv"), (dq, dk, dv), with_ws):
            g = f64(got.cpu())
            assert_close(f"{name} vs oracle (call {call + 1})", g, ref[name], ATOL[dtype], dtype)
            assert_relnorm(f"{name} vs oracle (call {call + 1})", g, ref[name])
            assert_close(f"{name} vs fa_bwd (call {call + 1})", g, other, ATOL[dtype], dtype)


def test_noalloc_rejects_sizes_beyond_its_scratch(fa_lib):
    fa = fa_lib
    f = _noalloc(fa)
    # B=1, Hq=16, d=128, N=8192 needs 64 MiB of workspace > 32 MiB; rejected before any launch
    fake = 1 << 20
    st = f(fake, fake, fake, fake, fake, fake, fake, fake, fake, 1, 16, 16, 8192, 128, 0, 0.088, fa.FA_BF16, None)
    assert st == fa.FA_ERR_UNSUPPORTED
