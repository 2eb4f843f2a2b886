"""The C ABI library loads on a host without a GPU, exports every entry point that
include/fa.h declares, and rejects bad arguments before touching the device."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")
LIB = os.path.join(ROOT, "exact_attention_38_gb300", "libfa.so")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from exact_attention_38_gb300 import build

        build.build()
    return ctypes.CDLL(LIB)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_check_device_error", "fa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_status_string.argtypes = [ctypes.c_int]
    for code, word in [(0, b"FA_OK"), (1, b"INVALID"), (2, b"UNSUPPORTED"), (3, b"CUDA"), (4, b"TIMEOUT")]:
        assert word in lib.fa_status_string(code)


def _fwd(lib, **kw):
    a = dict(q=0x10000, k=0x20000, v=0x30000, o=0x40000, lse=0x50000, B=1, Hq=2, Hkv=2, N=128, d=64,
             causal=0, scale=0.125, dtype=0)
    a.update(kw)
    f = lib.fa_fwd
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_float, i, vp]
    f.restype = i
    return f(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["N"], a["d"], a["causal"],
             a["scale"], a["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(k=0x20008), 1), (dict(lse=0x50004), 1),
    (dict(N=0), 1), (dict(B=0), 1), (dict(Hq=3, Hkv=2), 1), (dict(Hkv=0), 1),
    (dict(scale=0.0), 1), (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1), (dict(dtype=7), 1),
    (dict(d=96), 2), (dict(d=256), 2), (dict(d=0), 1), (dict(N=(1 << 20) + 1), 2),
])
def test_fwd_argument_errors_need_no_device(lib, kw, code):
    assert _fwd(lib, **kw) == code


def _bwd(lib, **kw):
    a = dict(q=0x10000, k=0x20000, v=0x30000, o=0x40000, lse=0x50000, do=0x60000, dq=0x70000, dk=0x80000,
             dv=0x90000, B=1, Hq=4, Hkv=2, N=300, d=128, causal=1, scale=0.088, dtype=0, ws=0x100000,
             ws_bytes=None)
    a.update(kw)
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd_workspace_size.argtypes = [ctypes.c_int] * 5
    need = lib.fa_bwd_workspace_size(a["B"], a["Hq"], a["Hkv"], a["N"], a["d"])
    ws_bytes = need if a["ws_bytes"] is None else a["ws_bytes"]
    vp, i = ctypes.c_void_p, ctypes.c_int
    f = lib.fa_bwd
    f.argtypes = [vp] * 9 + [i] * 6 + [ctypes.c_float, i, vp, ctypes.c_size_t, vp]
    f.restype = i
    return f(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"], a["B"], a["Hq"],
             a["Hkv"], a["N"], a["d"], a["causal"], a["scale"], a["dtype"], a["ws"], ws_bytes, None)


def test_workspace_size(lib):
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd_workspace_size.argtypes = [ctypes.c_int] * 5
    B, Hq, N, d = 2, 4, 300, 128
    rows = B * Hq * N
    npad = (N + 63) // 64 * 64
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    want = up(B * Hq * d * npad * 4) + 2 * up(B * Hq * npad * 4)
    assert lib.fa_bwd_workspace_size(B, Hq, 2, N, d) == want
    assert lib.fa_bwd_workspace_size(B, Hq, 3, N, d) == 0
    assert lib.fa_bwd_workspace_size(B, Hq, 2, N, 80) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(do=None), 1), (dict(dk=0x80002), 1), (dict(ws=None), 1), (dict(ws=0x100010), 1),
    (dict(ws_bytes=1024), 1), (dict(Hq=5), 1), (dict(d=32), 2), (dict(N=-5), 1),
])
def test_bwd_argument_errors_need_no_device(lib, kw, code):
    assert _bwd(lib, **kw) == code


def _fwd_varlen(lib, **kw):
    a = dict(q=0x10000, k=0x20000, v=0x30000, o=0x40000, lse=0x50000, cu_q=0x60000, cu_k=0x70000, used_q=None,
             used_k=None, B=3, Hq=4, Hkv=2, total_q=300, total_k=500, max_q=200, max_k=300, d=128, causal=1,
             scale=0.088, dtype=0)
    a.update(kw)
    vp, i = ctypes.c_void_p, ctypes.c_int
    f = lib.fa_fwd_varlen
    f.argtypes = [vp] * 9 + [i] * 9 + [ctypes.c_float, i, vp]
    f.restype = i
    return f(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cu_q"], a["cu_k"], a["used_q"], a["used_k"], a["B"],
             a["Hq"], a["Hkv"], a["total_q"], a["total_k"], a["max_q"], a["max_k"], a["d"], a["causal"],
             a["scale"], a["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(cu_q=None), 1), (dict(cu_k=0x70002), 1), (dict(used_q=0x80001), 1), (dict(q=0x10008), 1),
    (dict(total_q=-1), 1), (dict(max_k=-3), 1), (dict(B=0), 1), (dict(Hq=3), 1), (dict(scale=0.0), 1),
    (dict(d=96), 2), (dict(max_q=(1 << 20) + 1), 2),
    (dict(total_q=0, q=None, o=None, lse=None), 0),  # no query row: nothing is enqueued
])
def test_fwd_varlen_argument_errors_need_no_device(lib, kw, code):
    assert _fwd_varlen(lib, **kw) == code


def _bwd_varlen(lib, **kw):
    a = dict(q=0x10000, k=0x20000, v=0x30000, o=0x40000, lse=0x50000, do=0x60000, dq=0x70000, dk=0x80000,
             dv=0x90000, cu_q=0xa0000, cu_k=0xb0000, used_q=None, used_k=None, B=3, Hq=4, Hkv=2, total_q=300,
             total_k=500, max_q=200, max_k=300, d=64, causal=0, scale=0.125, dtype=1, ws=0x100000, ws_bytes=None)
    a.update(kw)
    lib.fa_bwd_varlen_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd_varlen_workspace_size.argtypes = [ctypes.c_int] * 4
    need = lib.fa_bwd_varlen_workspace_size(a["B"], a["Hq"], a["max_q"], a["d"])
    ws_bytes = need if a["ws_bytes"] is None else a["ws_bytes"]
    vp, i = ctypes.c_void_p, ctypes.c_int
    f = lib.fa_bwd_varlen
    f.argtypes = [vp] * 13 + [i] * 9 + [ctypes.c_float, i, vp, ctypes.c_size_t, vp]
    f.restype = i
    return f(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"], a["cu_q"], a["cu_k"],
             a["used_q"], a["used_k"], a["B"], a["Hq"], a["Hkv"], a["total_q"], a["total_k"], a["max_q"], a["max_k"],
             a["d"], a["causal"], a["scale"], a["dtype"], a["ws"], ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(do=None), 1), (dict(dk=0x80004), 1), (dict(cu_q=None), 1), (dict(ws=None), 1), (dict(ws_bytes=4096), 1),
    (dict(Hkv=3), 1), (dict(d=80), 2), (dict(total_k=-2), 1),
    (dict(total_q=0, total_k=0, q=None, k=None, v=None, o=None, lse=None, do=None, dq=None, dk=None, dv=None), 0),
])
def test_bwd_varlen_argument_errors_need_no_device(lib, kw, code):
    assert _bwd_varlen(lib, **kw) == code


def test_varlen_workspace_size(lib):
    lib.fa_bwd_varlen_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd_varlen_workspace_size.argtypes = [ctypes.c_int] * 4
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd_workspace_size.argtypes = [ctypes.c_int] * 5
    # the fixed-length layout with N = max_seqlen_q (at least one 64-row block)
    assert lib.fa_bwd_varlen_workspace_size(3, 4, 200, 128) == lib.fa_bwd_workspace_size(3, 4, 4, 200, 128)
    assert lib.fa_bwd_varlen_workspace_size(3, 4, 0, 128) == lib.fa_bwd_workspace_size(3, 4, 4, 64, 128)
    assert lib.fa_bwd_varlen_workspace_size(3, 4, 10, 96) == 0


def _decode(lib, **kw):
    a = dict(q=0x10000, k=0x20000, v=0x30000, cl=0x40000, o=0x50000, lse=0x60000, B=2, Hq=8, Hkv=2, Nq=1,
             Nmax=4096, d=128, causal=1, scale=0.088, splits=0, dtype=0, ws=0x100000, ws_bytes=None)
    a.update(kw)
    i = ctypes.c_int
    lib.fa_decode_workspace_size.restype = ctypes.c_size_t
    lib.fa_decode_workspace_size.argtypes = [i] * 7
    need = lib.fa_decode_workspace_size(a["B"], a["Hq"], a["Hkv"], a["Nq"], a["Nmax"], a["d"], a["splits"])
    ws_bytes = need if a["ws_bytes"] is None else a["ws_bytes"]
    vp = ctypes.c_void_p
    f = lib.fa_fwd_decode
    f.argtypes = [vp] * 6 + [i] * 7 + [ctypes.c_float, i, i, vp, ctypes.c_size_t, vp]
    f.restype = i
    return f(a["q"], a["k"], a["v"], a["cl"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["Nq"], a["Nmax"],
             a["d"], a["causal"], a["scale"], a["splits"], a["dtype"], a["ws"], ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(v=0x30008), 1), (dict(cl=None), 1), (dict(cl=0x40002), 1), (dict(Nq=0), 1),
    (dict(Nmax=0), 1), (dict(Hq=6, Hkv=4), 1), (dict(splits=-1), 1), (dict(scale=-1.0), 1), (dict(d=256), 2),
    (dict(Hq=32, Hkv=1, Nq=8), 2),  # 256 packed rows > one 128-row tile
    (dict(ws=None), 1), (dict(ws_bytes=16), 1),
])
def test_decode_argument_errors_need_no_device(lib, kw, code):
    assert _decode(lib, **kw) == code


def _decode_paged(lib, **kw):
    a = dict(q=0x10000, kp=0x20000, vp=0x30000, table=0x70000, cl=0x40000, o=0x50000, lse=0x60000, B=2, Hq=8, Hkv=2,
             Nq=1, num_pages=64, max_pages=32, d=128, causal=1, scale=0.088, splits=0, dtype=0, ws=0x100000,
             ws_bytes=None)
    a.update(kw)
    i = ctypes.c_int
    lib.fa_decode_workspace_size.restype = ctypes.c_size_t
    lib.fa_decode_workspace_size.argtypes = [i] * 7
    need = lib.fa_decode_workspace_size(a["B"], a["Hq"], a["Hkv"], a["Nq"], 128 * a["max_pages"], a["d"],
                                        a["splits"])
    ws_bytes = need if a["ws_bytes"] is None else a["ws_bytes"]
    vp = ctypes.c_void_p
    f = lib.fa_fwd_decode_paged
    f.argtypes = [vp] * 7 + [i] * 8 + [ctypes.c_float, i, i, vp, ctypes.c_size_t, vp]
    f.restype = i
    return f(a["q"], a["kp"], a["vp"], a["table"], a["cl"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["Nq"],
             a["num_pages"], a["max_pages"], a["d"], a["causal"], a["scale"], a["splits"], a["dtype"], a["ws"],
             ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(table=None), 1), (dict(table=0x70002), 1), (dict(kp=0x20008), 1), (dict(cl=None), 1),
    (dict(num_pages=0), 1), (dict(max_pages=0), 1), (dict(max_pages=1 << 20), 2), (dict(Hq=6, Hkv=4), 1),
    (dict(d=256), 2), (dict(ws_bytes=16), 1), (dict(scale=float("nan")), 1),
])
def test_decode_paged_argument_errors_need_no_device(lib, kw, code):
    assert _decode_paged(lib, **kw) == code


def test_decode_split_targets_one_wave(lib):
    """Automatic split count: one wave of CTAs on 152 SMs, 304 slots at two CTAs per SM,
    or 152 when the deep K/V ring (one CTA per SM) is used, i.e. at d = 128 with at most
    8 (batch, kv head) units; never more splits than 128-key blocks.  Splits take equal
    block counts, cps = ceil(blocks / target), so the count is ceil(blocks / cps)."""
    i = ctypes.c_int
    lib.fa_decode_num_splits.restype = i
    lib.fa_decode_num_splits.argtypes = [i] * 7
    n = lambda B, Hkv, N, d: lib.fa_decode_num_splits(B, 4 * Hkv, Hkv, 1, N, d, 0)
    assert n(1, 8, 65536, 128) == 19  # deep ring: 8 units x 19 = 152 CTAs
    assert n(2, 4, 65536, 128) == 19
    assert n(2, 8, 65536, 128) == 19  # 16 units: 304 // 16
    assert n(4, 8, 65536, 128) == 9
    assert n(1, 8, 65536, 64) == 37  # d = 64 keeps two CTAs per SM: target 38, 14 blocks each
    assert n(1, 1, 65536, 128) == 128  # target 152: 4 of the 512 blocks each
    assert n(1, 8, 1000, 128) == 8  # capped by the 8 key blocks
    assert n(64, 8, 65536, 128) == 1


def test_decode_split_count_and_workspace(lib):
    i = ctypes.c_int
    lib.fa_decode_num_splits.restype = i
    lib.fa_decode_num_splits.argtypes = [i] * 7
    lib.fa_decode_workspace_size.restype = ctypes.c_size_t
    lib.fa_decode_workspace_size.argtypes = [i] * 7
    # forced counts are capped by the number of 128-key blocks, then trimmed so no
    # split is empty (9 blocks in 4 splits of 3 -> 3 splits)
    assert lib.fa_decode_num_splits(1, 8, 2, 1, 1152, 128, 4) == 3
    assert lib.fa_decode_num_splits(1, 8, 2, 1, 200, 128, 50) == 2
    assert lib.fa_decode_num_splits(1, 8, 2, 1, 200, 128, 1) == 1
    # automatic: more splits when batch x kv-heads is small
    assert lib.fa_decode_num_splits(1, 32, 8, 1, 65536, 128, 0) > lib.fa_decode_num_splits(64, 32, 8, 1, 65536, 128, 0)
    # one split needs no workspace; otherwise partial outputs + partial lse
    assert lib.fa_decode_workspace_size(1, 8, 2, 1, 4096, 128, 1) == 0
    S = lib.fa_decode_num_splits(1, 8, 2, 2, 4096, 128, 5)
    rows = 1 * 2 * S * 4 * 2
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert lib.fa_decode_workspace_size(1, 8, 2, 2, 4096, 128, 5) == up(rows * 128 * 4) + up(rows * 4)


def test_fp8_argument_errors_need_no_device(lib):
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd_fp8_workspace_size.restype = ctypes.c_size_t
    lib.fa_fwd_fp8_workspace_size.argtypes = [i] * 4
    assert lib.fa_fwd_fp8_workspace_size(2, 4, 300, 128) == 2 * 4 * 128 * 384
    assert lib.fa_fwd_fp8_workspace_size(2, 4, 300, 64) == 0
    fn = lib.fa_fwd_fp8
    fn.argtypes = [vp] * 5 + [i] * 6 + [f, f, f, f, vp, ctypes.c_size_t, vp]
    fn.restype = i
    base = [0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 2, 4, 4, 300, 128, 1, 0.088, 0.01, 0.01, 0.01, 0x100000,
            2 * 4 * 128 * 384, None]
    for idx, val, code in [(0, None, 1), (1, 0x20008, 1), (9, 64, 2), (12, 0.0, 1), (14, float("nan"), 1),
                           (15, None, 1), (16, 1024, 1), (6, 3, 1)]:
        a = list(base)
        a[idx] = val
        assert fn(*a) == code, (idx, val)


def test_fp8_blockscaled_argument_errors_need_no_device(lib):
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn = lib.fa_fwd_fp8_blockscaled
    fn.argtypes = [vp] * 8 + [i] * 6 + [f, vp, ctypes.c_size_t, vp]
    fn.restype = i
    base = [0x10000, 0x20000, 0x30000, 0x40000, 0x40100, 0x40200, 0x50000, 0x60000, 2, 4, 4, 300, 128, 1, 0.088,
            0x100000, 2 * 4 * 128 * 384, None]
    # null or misaligned tensors / descales, d != 128, bad scale, short or null workspace,
    # Hq % Hkv != 0: rejected before any CUDA call
    for idx, val, code in [(0, None, 1), (3, None, 1), (5, 0x40202, 1), (6, 0x50008, 1), (12, 64, 2),
                           (14, 0.0, 1), (15, None, 1), (16, 1024, 1), (10, 3, 1)]:
        a = list(base)
        a[idx] = val
        assert fn(*a) == code, (idx, val)


def test_noalloc_scratch_limit_needs_no_device(lib):
    """fa_bwd_noalloc's fixed scratch: with B=1, Hq=16, d=128 the backward workspace fits
    up to N=4032 (Npad 4032) and not at N=4033 (Npad 4096); there the call is rejected
    with FA_ERR_UNSUPPORTED before any CUDA call, so it answers on a host without a GPU."""
    m = re.search(r"#define\s+FA_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", open(HEADER).read())
    limit = int(m.group(1)) << int(m.group(2))
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd_workspace_size.argtypes = [ctypes.c_int] * 5
    assert lib.fa_bwd_workspace_size(1, 16, 16, 4032, 128) <= limit
    assert lib.fa_bwd_workspace_size(1, 16, 16, 4033, 128) > limit
    f = lib.fa_bwd_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp] * 9 + [i] * 6 + [ctypes.c_float, i, vp]
    f.restype = i
    fake = 1 << 20
    assert f(*([fake] * 9), 1, 16, 16, 4033, 128, 0, 0.088, 0, None) == 2
    assert f(*([fake] * 9), 1, 16, 16, 8192, 128, 1, 0.088, 1, None) == 2
