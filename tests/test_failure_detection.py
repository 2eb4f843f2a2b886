"""Failure detection without a GPU fault: a kernel's bounded wait runs out on a barrier
that nothing arrives on, the kernel records the timeout and exits, the host reads
FA_ERR_TIMEOUT, and the context keeps working."""

import ctypes
import math

import pytest

from _parity import ATOL, assert_close, f64, gpu_forward, make_inputs

LIB_ARGS = [ctypes.c_int, ctypes.c_void_p]


def test_selftest_rejects_out_of_range_limits_without_a_device():
    import os

    lib = ctypes.CDLL(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                                   "exact_attention_38_gb300", "libfa.so"))
    lib.fa_selftest_wait_timeout.argtypes = LIB_ARGS
    lib.fa_selftest_wait_timeout.restype = ctypes.c_int
    assert lib.fa_selftest_wait_timeout(0, None) == 1
    assert lib.fa_selftest_wait_timeout(2_000_000, None) == 1


@pytest.mark.gpu
def test_bounded_wait_reports_timeout_and_context_survives(fa_lib):
    import torch

    fa = fa_lib
    s = torch.cuda.current_stream().cuda_stream
    assert fa.fa_check_device_error(s) == fa.FA_OK          # clean start
    assert fa.fa_selftest_wait_timeout(2000, s) == fa.FA_OK  # 2 ms limit
    assert fa.fa_check_device_error(s) == fa.FA_ERR_TIMEOUT
    assert fa.fa_check_device_error(s) == fa.FA_OK          # the word was cleared
    # the context still runs real work correctly
    import oracle

    x = make_inputs(1, 200, 2, 2, 64, dtype="bf16", seed=41, with_do=False)
    _, o, _ = gpu_forward(fa, x, True)
    xo = {k: f64(v) for k, v in x.items()}
    want, _ = oracle.attn_fwd_ref(xo["q"], xo["k"], xo["v"], True, 1.0 / math.sqrt(64))
    assert_close("O", f64(o.cpu()), want, ATOL["bf16"], "bf16")
