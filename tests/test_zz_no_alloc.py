"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Plugins or engines that only get their input and output buffers, programs whose
allocator is frozen after start-up, and real-time paths cannot hand fa_bwd a
workspace; fa_bwd_noalloc uses a scratch array inside the library instead.  This test
calls it through the C ABI and checks that two calls in a row give the same gradients
as fa_bwd with a caller-provided workspace, within the parity tolerance.  The file name
sorts last so that a run stopping at its first failure has run every other test.
"""

import ctypes
import math

import pytest

from _parity import ATOL, assert_close, f64, make_inputs, to_gpu

pytestmark = pytest.mark.gpu


def _noalloc(fa):
    f = fa.lib.fa_bwd_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp] * 9 + [i] * 6 + [ctypes.c_float, i, vp]
    f.restype = i
    return f


def test_noalloc_backward_matches_workspace_backward_twice(fa_lib):
    import torch

    fa = fa_lib
    f = _noalloc(fa)
    B, N, Hq, Hkv, d, causal = 2, 700, 4, 2, 128, True
    x = make_inputs(B, N, Hq, Hkv, d, dtype="bf16", seed=31)
    q, k, v, do = (to_gpu(x[n]) for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    want = fa.backward(do, q, k, v, o, lse, causal=causal, scale=scale)
    fa.check_device_error()
    want = [f64(t.cpu()) for t in want]
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        st = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
               dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, N, d, int(causal), scale, fa.FA_BF16,
               stream)
        assert st == fa.FA_OK, fa.status_string(st)
        fa.check_device_error()
        for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), want):
            assert_close(f"{name} (call {call + 1})", f64(got.cpu()), ref, ATOL["bf16"])


def test_noalloc_rejects_sizes_beyond_its_scratch(fa_lib):
    fa = fa_lib
    f = _noalloc(fa)
    # B=1, Hq=16, d=128, N=8192 needs 64 MiB of workspace > 32 MiB; rejected before any launch
    fake = 1 << 20
    st = f(fake, fake, fake, fake, fake, fake, fake, fake, fake, 1, 16, 16, 8192, 128, 0, 0.088, fa.FA_BF16, None)
    assert st == fa.FA_ERR_UNSUPPORTED
