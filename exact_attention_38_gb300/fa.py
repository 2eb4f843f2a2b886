"""ctypes binding of libfa.so: argument marshalling only, every step runs in the library.

The C names are mirrored one to one (``fa_fwd``, ``fa_bwd``, ``fa_bwd_workspace_size``,
``fa_fwd_varlen``, ``fa_bwd_varlen``, ``fa_bwd_varlen_workspace_size``,
``fa_check_device_error``, ``fa_status_string``).  ``forward`` / ``backward`` and
``forward_varlen`` / ``backward_varlen`` are conveniences that allocate the outputs
with torch (device memory and streams are the only things torch provides here) and
call the C entry points on the current stream.  Importing this module loads the library and raises if it is missing: there
is no fallback path.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

FA_OK, FA_ERR_INVALID, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
FA_BF16, FA_FP16 = 0, 1
_DT = {torch.bfloat16: FA_BF16, torch.float16: FA_FP16}


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libfa.so not found at {LIB_PATH}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
    lib.fa_fwd.restype = i
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_deterministic.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp]
    lib.fa_bwd_deterministic.restype = i
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_bwd_workspace_size.argtypes = [i, i, i, i, i]
    lib.fa_bwd_workspace_size.restype = sz
    lib.fa_fwd_varlen.argtypes = [vp] * 9 + [i] * 9 + [f, i, vp]
    lib.fa_fwd_varlen.restype = i
    lib.fa_bwd_varlen.argtypes = [vp] * 13 + [i] * 9 + [f, i, vp, sz, vp]
    lib.fa_bwd_varlen.restype = i
    lib.fa_bwd_varlen_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd_varlen_workspace_size.restype = sz
    lib.fa_fwd_decode.argtypes = [vp] * 6 + [i] * 7 + [f, i, i, vp, sz, vp]
    lib.fa_fwd_decode.restype = i
    lib.fa_fwd_decode_paged.argtypes = [vp] * 7 + [i] * 8 + [f, i, i, vp, sz, vp]
    lib.fa_fwd_decode_paged.restype = i
    lib.fa_decode_workspace_size.argtypes = [i] * 7
    lib.fa_decode_workspace_size.restype = sz
    lib.fa_decode_num_splits.argtypes = [i] * 7
    lib.fa_decode_num_splits.restype = i
    lib.fa_fwd_fp8.argtypes = [vp] * 5 + [i] * 6 + [f, f, f, f, vp, sz, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_fwd_fp8_workspace_size.argtypes = [i] * 4
    lib.fa_fwd_fp8_workspace_size.restype = sz
    lib.fa_fwd_fp8_blockscaled.argtypes = [vp] * 8 + [i] * 6 + [f, vp, sz, vp]
    lib.fa_fwd_fp8_blockscaled.restype = i
    lib.fa_selftest_wait_timeout.argtypes = [i, vp]
    lib.fa_selftest_wait_timeout.restype = i
    lib.fa_selftest_exp2.argtypes = [vp, vp, vp, i, vp]
    lib.fa_selftest_exp2.restype = i
    lib.fa_check_device_error.argtypes = [vp]
    lib.fa_check_device_error.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    return lib


lib = _load()


# ------------------------------------------------------------- raw C entry points

def status_string(status: int) -> str:
    return lib.fa_status_string(int(status)).decode()


def fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, dtype, stream) -> int:
    """Mirror of the C ``fa_fwd``; pointers and stream are plain integers."""
    return lib.fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, int(causal), float(scale), int(dtype), stream)


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, dtype, workspace,
           workspace_bytes, stream) -> int:
    """Mirror of the C ``fa_bwd``."""
    return lib.fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, int(causal), float(scale),
                      int(dtype), workspace, int(workspace_bytes), stream)


def fa_bwd_deterministic(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, dtype, workspace,
                         workspace_bytes, stream) -> int:
    """Mirror of the C ``fa_bwd_deterministic``."""
    return lib.fa_bwd_deterministic(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, int(causal), float(scale),
                                    int(dtype), workspace, int(workspace_bytes), stream)


def fa_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, dtype, stream) -> int:
    """Mirror of the C ``fa_bwd_noalloc`` (fa_bwd on the library's own scratch array)."""
    return lib.fa_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, int(causal), float(scale),
                              int(dtype), stream)


def fa_bwd_workspace_size(B, Hq, Hkv, N, d) -> int:
    return int(lib.fa_bwd_workspace_size(B, Hq, Hkv, N, d))


def fa_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, used_q, used_k, B, Hq, Hkv, total_q, total_k, max_q, max_k, d,
                  causal, scale, dtype, stream) -> int:
    """Mirror of the C ``fa_fwd_varlen``."""
    return lib.fa_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, used_q, used_k, B, Hq, Hkv, total_q, total_k, max_q,
                             max_k, d, int(causal), float(scale), int(dtype), stream)


def fa_bwd_varlen_workspace_size(B, Hq, max_q, d) -> int:
    return int(lib.fa_bwd_varlen_workspace_size(B, Hq, max_q, d))


def fa_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_q, cu_k, used_q, used_k, B, Hq, Hkv, total_q, total_k,
                  max_q, max_k, d, causal, scale, dtype, workspace, workspace_bytes, stream) -> int:
    """Mirror of the C ``fa_bwd_varlen``."""
    return lib.fa_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_q, cu_k, used_q, used_k, B, Hq, Hkv, total_q,
                             total_k, max_q, max_k, d, int(causal), float(scale), int(dtype), workspace,
                             int(workspace_bytes), stream)


def fa_fwd_decode(q, k_cache, v_cache, cache_seqlens, o, lse, B, Hq, Hkv, Nq, Nmax, d, causal, scale, num_splits,
                  dtype, workspace, workspace_bytes, stream) -> int:
    """Mirror of the C ``fa_fwd_decode``."""
    return lib.fa_fwd_decode(q, k_cache, v_cache, cache_seqlens, o, lse, B, Hq, Hkv, Nq, Nmax, d, int(causal),
                             float(scale), int(num_splits), int(dtype), workspace, int(workspace_bytes), stream)


def fa_fwd_decode_paged(q, k_pages, v_pages, block_table, cache_seqlens, o, lse, B, Hq, Hkv, Nq, num_pages,
                        max_pages, d, causal, scale, num_splits, dtype, workspace, workspace_bytes, stream) -> int:
    """Mirror of the C ``fa_fwd_decode_paged``."""
    return lib.fa_fwd_decode_paged(q, k_pages, v_pages, block_table, cache_seqlens, o, lse, B, Hq, Hkv, Nq, num_pages,
                                   max_pages, d, int(causal), float(scale), int(num_splits), int(dtype), workspace,
                                   int(workspace_bytes), stream)


def fa_decode_workspace_size(B, Hq, Hkv, Nq, Nmax, d, num_splits=0) -> int:
    return int(lib.fa_decode_workspace_size(B, Hq, Hkv, Nq, Nmax, d, num_splits))


def fa_decode_num_splits(B, Hq, Hkv, Nq, Nmax, d, num_splits=0) -> int:
    return int(lib.fa_decode_num_splits(B, Hq, Hkv, Nq, Nmax, d, num_splits))


def fa_fwd_fp8(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, q_descale, k_descale, v_descale, workspace,
               workspace_bytes, stream) -> int:
    """Mirror of the C ``fa_fwd_fp8``."""
    return lib.fa_fwd_fp8(q, k, v, o, lse, B, Hq, Hkv, N, d, int(causal), float(scale), float(q_descale),
                          float(k_descale), float(v_descale), workspace, int(workspace_bytes), stream)


def fa_fwd_fp8_workspace_size(B, Hkv, N, d) -> int:
    return int(lib.fa_fwd_fp8_workspace_size(B, Hkv, N, d))


def fa_fwd_fp8_blockscaled(q, k, v, q_descale, k_descale, v_descale, o, lse, B, Hq, Hkv, N, d, causal, scale,
                           workspace, workspace_bytes, stream) -> int:
    """Mirror of the C ``fa_fwd_fp8_blockscaled``; the descales are device pointers."""
    return lib.fa_fwd_fp8_blockscaled(q, k, v, q_descale, k_descale, v_descale, o, lse, B, Hq, Hkv, N, d,
                                      int(causal), float(scale), workspace, int(workspace_bytes), stream)


def fa_selftest_wait_timeout(limit_us, stream) -> int:
    """Mirror of the C ``fa_selftest_wait_timeout``."""
    return lib.fa_selftest_wait_timeout(int(limit_us), stream)


def fa_check_device_error(stream) -> int:
    return lib.fa_check_device_error(stream)


# ------------------------------------------------------------------- conveniences

def _ptr(t):
    return t.data_ptr() if t is not None else None


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _shapes(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, N, H, d]")
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError("q, k, v must be contiguous CUDA tensors of one dtype")
    if q.dtype not in _DT:
        raise ValueError("dtype must be bf16 or fp16")
    return B, N, Hq, Hkv, d


def forward(q, k, v, causal=False, scale=None, out=None, lse=None, stream=None):
    """Returns (o [B,N,Hq,d], lse [B,Hq,N] fp32)."""
    B, N, Hq, Hkv, d = _shapes(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if lse is None else lse
    st = fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d, causal, scale, _DT[q.dtype],
                _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd")
    return o, lse


def backward(dout, q, k, v, o, lse, causal=False, scale=None, workspace=None, dq=None, dk=None, dv=None,
             stream=None, deterministic=False):
    """Returns (dq, dk, dv); allocates the workspace with torch if not given.  With
    ``deterministic`` the results are identical bit for bit from run to run."""
    B, N, Hq, Hkv, d = _shapes(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    ws_bytes = fa_bwd_workspace_size(B, Hq, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    fn = fa_bwd_deterministic if deterministic else fa_bwd
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), B, Hq,
            Hkv, N, d, causal, scale, _DT[q.dtype], _ptr(workspace), workspace.numel(), _stream(stream))
    if st != FA_OK:
        raise FaError(st, fn.__name__)
    return dq, dk, dv


def _varlen_shapes(q, k, v, cu_q, cu_k):
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3 or k.shape != v.shape:
        raise ValueError("varlen q must be [total_q, Hq, d], k and v [total_k, Hkv, d]")
    if q.shape[2] != k.shape[2] or q.dtype not in _DT or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share d and a 16-bit dtype")
    for t in (cu_q, cu_k):
        if t.dtype != torch.int32 or t.dim() != 1 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("cu_seqlens must be contiguous int32 CUDA vectors of B+1 offsets")
    if cu_q.numel() != cu_k.numel() or cu_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold B+1 >= 2 offsets")
    return cu_q.numel() - 1, q.shape[0], k.shape[0], q.shape[1], k.shape[1], q.shape[2]


def forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal=False, scale=None,
                   seqused_q=None, seqused_k=None, out=None, lse=None, stream=None):
    """Packed variable-length forward.  Returns (o [total_q,Hq,d], lse [Hq,total_q] fp32).

    Rows outside every sequence are left as allocated (uninitialised unless `out` /
    `lse` are passed in)."""
    B, tq, tk, Hq, Hkv, d = _varlen_shapes(q, k, v, cu_seqlens_q, cu_seqlens_k)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((Hq, tq), dtype=torch.float32, device=q.device) if lse is None else lse
    st = fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                       _ptr(seqused_q), _ptr(seqused_k), B, Hq, Hkv, tq, tk, int(max_seqlen_q), int(max_seqlen_k), d,
                       causal, scale, _DT[q.dtype], _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_varlen")
    return o, lse


def backward_varlen(dout, q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal=False,
                    scale=None, seqused_q=None, seqused_k=None, workspace=None, dq=None, dk=None, dv=None,
                    stream=None):
    """Packed variable-length backward.  Returns (dq, dk, dv); rows outside every
    sequence are left as allocated."""
    B, tq, tk, Hq, Hkv, d = _varlen_shapes(q, k, v, cu_seqlens_q, cu_seqlens_k)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    ws_bytes = fa_bwd_varlen_workspace_size(B, Hq, int(max_seqlen_q), d)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    st = fa_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                       _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(seqused_q), _ptr(seqused_k), B, Hq, Hkv, tq, tk,
                       int(max_seqlen_q), int(max_seqlen_k), d, causal, scale, _DT[q.dtype], _ptr(workspace),
                       workspace.numel(), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_bwd_varlen")
    return dq, dk, dv


def forward_decode(q, k_cache, v_cache, cache_seqlens, causal=False, scale=None, num_splits=0, out=None, lse=None,
                   workspace=None, stream=None):
    """Decode forward: q [B,Nq,Hq,d] against caches [B,Nmax,Hkv,d] with per-sequence
    lengths ``cache_seqlens`` (int32 CUDA [B]).  Returns (o [B,Nq,Hq,d], lse [B,Hq,Nq])."""
    if q.dim() != 4 or k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("q must be [B,Nq,Hq,d] and the caches [B,Nmax,Hkv,d]")
    B, Nq, Hq, d = q.shape
    Nmax, Hkv = k_cache.shape[1], k_cache.shape[2]
    if k_cache.shape[0] != B or k_cache.shape[3] != d or q.dtype not in _DT or k_cache.dtype != q.dtype:
        raise ValueError("q and the caches must share B, d and a 16-bit dtype")
    if cache_seqlens.dtype != torch.int32 or cache_seqlens.numel() != B or not cache_seqlens.is_cuda:
        raise ValueError("cache_seqlens must be an int32 CUDA vector of B lengths")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    ws_bytes = fa_decode_workspace_size(B, Hq, Hkv, Nq, Nmax, d, num_splits)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    st = fa_fwd_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_seqlens), _ptr(o), _ptr(lse), B, Hq, Hkv,
                       Nq, Nmax, d, causal, scale, num_splits, _DT[q.dtype], _ptr(workspace),
                       workspace.numel() if workspace is not None else 0, _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_decode")
    return o, lse


def forward_fp8(q, k, v, q_descale, k_descale, v_descale, causal=False, scale=None, out=None, lse=None,
                workspace=None, stream=None):
    """FP8 forward: q [B,N,Hq,128], k/v [B,N,Hkv,128] as torch.float8_e4m3fn (or uint8
    holding E4M3 bytes) with per-tensor descales.  Returns (o bf16, lse fp32)."""
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B,N,Hq,d], k and v [B,N,Hkv,d]")
    for t in (q, k, v):
        if t.element_size() != 1 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous 8-bit CUDA tensors")
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device) if out is None else out
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if lse is None else lse
    ws_bytes = fa_fwd_fp8_workspace_size(B, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    st = fa_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d, causal, scale, q_descale,
                    k_descale, v_descale, _ptr(workspace), workspace.numel(), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_fp8")
    return o, lse


def forward_fp8_blockscaled(q, k, v, q_descale, k_descale, v_descale, causal=False, scale=None, out=None, lse=None,
                            workspace=None, stream=None):
    """FP8 forward with one descale per 128-row block of each head: q [B,N,Hq,128], k/v
    [B,N,Hkv,128] 8-bit E4M3 CUDA tensors; q_descale [B,Hq,ceil(N/128)], k_descale and
    v_descale [B,Hkv,ceil(N/128)] fp32 CUDA tensors.  Returns (o bf16, lse fp32)."""
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B,N,Hq,d], k and v [B,N,Hkv,d]")
    for t in (q, k, v):
        if t.element_size() != 1 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous 8-bit CUDA tensors")
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    nb = (N + 127) // 128
    for t, hh in ((q_descale, Hq), (k_descale, Hkv), (v_descale, Hkv)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (B, hh, nb):
            raise ValueError("descales must be contiguous fp32 CUDA tensors [B, H, ceil(N/128)]")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device) if out is None else out
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if lse is None else lse
    ws_bytes = fa_fwd_fp8_workspace_size(B, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    st = fa_fwd_fp8_blockscaled(_ptr(q), _ptr(k), _ptr(v), _ptr(q_descale), _ptr(k_descale), _ptr(v_descale),
                                _ptr(o), _ptr(lse), B, Hq, Hkv, N, d, causal, scale, _ptr(workspace),
                                workspace.numel(), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_fp8_blockscaled")
    return o, lse


def forward_decode_paged(q, k_pages, v_pages, block_table, cache_seqlens, causal=False, scale=None, num_splits=0,
                         out=None, lse=None, workspace=None, stream=None):
    """Decode forward over a paged cache: k_pages / v_pages [num_pages, 128, Hkv, d],
    block_table int32 CUDA [B, max_pages].  Returns (o [B,Nq,Hq,d], lse [B,Hq,Nq])."""
    B, Nq, Hq, d = q.shape
    num_pages, page, Hkv = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    if page != 128 or v_pages.shape != k_pages.shape or k_pages.shape[3] != d:
        raise ValueError("pages must be [num_pages, 128, Hkv, d] for both caches")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be int32 [B, max_pages]")
    max_pages = block_table.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    ws_bytes = fa_decode_workspace_size(B, Hq, Hkv, Nq, max_pages * 128, d, num_splits)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    st = fa_fwd_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(cache_seqlens), _ptr(o),
                             _ptr(lse), B, Hq, Hkv, Nq, num_pages, max_pages, d, causal, scale, num_splits,
                             _DT[q.dtype], _ptr(workspace), workspace.numel() if workspace is not None else 0,
                             _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_decode_paged")
    return o, lse


def check_device_error(stream=None):
    st = fa_check_device_error(_stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_check_device_error")
