"""Paged KV-cache attention for GB300 (sm_103a): Python binding.

Thin ctypes layer over ``libpagedattn.so`` (``include/pagedattn.h``).  The
functions keep the C names and only marshal arguments (pointers, strides,
sizes, the current CUDA stream); every step of the computation runs in the
library's CUDA kernels.  PyTorch is used for device memory and streams: the
convenience arguments that are left as ``None`` (``out``, ``lse``,
``workspace``) are allocated with ``torch.empty`` on the tensors' device.

There is no CPU fallback: if the library has not been built (``python -m
paged_kv_cache_page_gb300.build``) or a tensor is not on a CUDA device, the
call raises.
"""

import ctypes
import math
import os

import torch

from .build import lib_path

PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_CUDA = -3
PA_ERR_WORKSPACE = -4
PA_F16 = 0
PA_BF16 = 1
PA_DEVERR_PAGE_OOB = 1
PA_DEVERR_LENGTH = 2
PA_DEVERR_TIMEOUT = 3
PAGE_SIZE = 16
PA_NOALLOC_SCRATCH_BYTES = 8 << 20  # fixed split scratch of pa_fwd_kvcache_noalloc

_DTYPE = {torch.float16: PA_F16, torch.bfloat16: PA_BF16}


class PagedAttnError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"pagedattn error {code}: {msg}")
        self.code = code


class pa_tensor4(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("stride_b", ctypes.c_int64),
                ("stride_t", ctypes.c_int64), ("stride_h", ctypes.c_int64)]


_lib = None
_vp, _i32, _i64, _f32, _sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                              ctypes.c_size_t)

_SIGNATURES = {
    "pa_append_kv": (_i32, [pa_tensor4, pa_tensor4, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32,
                            _i32, _i32, _i32, _i64, _i32, _vp, _vp]),
    "pa_fwd_kvcache": (_i32, [_vp, _i64, _i64, _i64, pa_tensor4, pa_tensor4, _vp, _vp, _i32,
                              _vp, _vp, _i64, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i64,
                              _i32, _f32, _i32, _i32, _vp, _vp, _vp, _sz, _vp, _i32, _vp]),
    "pa_fwd_kvcache_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32]),
    "pa_fwd_kvcache_rotary": (_i32, [_vp, _i64, _i64, _i64, pa_tensor4, pa_tensor4, _vp, _vp,
                                     _i32, _vp, _vp, _i64, _i32, _i32, _i32, _i32, _i32, _i32,
                                     _i32, _i64, _i32, _vp, _vp, _i32, _i32, _i32, _f32, _i32,
                                     _i32, _vp, _vp, _vp, _sz, _vp, _i32, _vp]),
    "pa_fwd_kvcache_rotary_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                                   _i32]),
    "pa_fwd_kvcache_noalloc": (_i32, [_vp, _i64, _i64, _i64, pa_tensor4, pa_tensor4, _vp, _vp,
                                      _i32, _vp, _vp, _i64, _i32, _i32, _i32, _i32, _i32, _i32,
                                      _i32, _i64, _i32, _f32, _i32, _i32, _vp, _vp, _vp, _i32,
                                      _vp]),
    "pa_fwd_varlen_unified": (_i32, [_vp, _i64, _i64, pa_tensor4, pa_tensor4, _vp, _vp, _vp,
                                     _i64, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                     _i64, _f32, _i32, _vp, _vp, _vp, _sz, _vp, _i32, _vp]),
    "pa_fwd_varlen_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32]),
    "pa_split_combine": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _i32,
                                _vp]),
    "pa_last_error_string": (ctypes.c_char_p, []),
    "pa_version": (_i32, []),
}


def load_library(path=None):
    """Load libpagedattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with python -m paged_kv_cache_page_gb300.build")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(rc):
    if rc != PA_OK:
        raise PagedAttnError(rc, _lib.pa_last_error_string().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("pagedattn tensors must be on a CUDA device")


def _page_size(k_cache, block_table):
    """Tokens per page of a paged cache ``[num_pages, page_size, Hkv, D]``
    (ignored by the library for a contiguous cache)."""
    return k_cache.shape[1] if block_table is not None else PAGE_SIZE


def _stream(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _t4(cache):
    if cache.stride(-1) != 1:
        raise ValueError("cache head_dim axis must be contiguous")
    return pa_tensor4(cache.data_ptr(), cache.stride(0), cache.stride(1), cache.stride(2))


def _dtype(t):
    if t.dtype not in _DTYPE:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return _DTYPE[t.dtype]


def new_err_word(device):
    """int32[4] device error word (zeroed) for the ``err`` argument."""
    return torch.zeros(4, dtype=torch.int32, device=device)


def pa_append_kv(k_cache, v_cache, k_new, v_new, cache_seqlens, block_table=None, err=None):
    """Write k_new/v_new ``[B, Lnew, Hkv, D]`` at positions cache_seqlens[b] + i."""
    lib = load_library()
    _cuda(k_cache, v_cache, k_new, v_new, cache_seqlens, block_table)
    B, lnew, hkv, d = k_new.shape
    k_new = k_new.contiguous()
    v_new = v_new.contiguous()
    if block_table is not None:
        extent, max_pages, bt_stride = k_cache.shape[0], block_table.shape[1], block_table.stride(0)
    else:
        extent, max_pages, bt_stride = k_cache.shape[1], 0, 0
    _check(lib.pa_append_kv(_t4(k_cache), _t4(v_cache), _ptr(k_new), _ptr(v_new),
                            _ptr(cache_seqlens), _ptr(block_table), bt_stride, max_pages,
                            _page_size(k_cache, block_table), B, lnew, hkv, d, extent,
                            _dtype(k_cache), _ptr(err), _stream(k_cache)))


def fwd_kvcache_workspace_size(B, Lq, Hq, Hkv, D, max_seqlen_k, num_splits=0):
    return load_library().pa_fwd_kvcache_workspace_size(B, Lq, Hq, Hkv, D, max_seqlen_k,
                                                        num_splits)


def pa_fwd_kvcache(q, k_cache, v_cache, cache_seqlens, block_table=None, k=None, v=None,
                   scale=None, causal=False, num_splits=0, out=None, lse=None, workspace=None,
                   err=None, max_seqlen_k=None, return_lse=True, rotary_cos=None,
                   rotary_sin=None, rotary_interleaved=False):
    """flash_attn_with_kvcache-style forward; returns ``(out, lse)``.

    q ``[B, Lq, Hq, D]``; caches paged ``[num_pages, 16, Hkv, D]`` with
    ``block_table [B, max_pages]`` (int32) or contiguous ``[B, capacity, Hkv, D]``;
    ``k``/``v`` ``[B, Lnew, Hkv, D]`` are appended in the same call.
    ``max_seqlen_k`` defaults to the capacity implied by the table/cache shape.
    ``rotary_cos``/``rotary_sin`` ``[rotary_len, rotary_dim / 2]`` (q's dtype):
    rotary embedding of the new tokens' q and k (pa_fwd_kvcache_rotary).
    """
    lib = load_library()
    _cuda(q, k_cache, v_cache, cache_seqlens, block_table, k, v)
    B, lq, hq, d = q.shape
    hkv = k_cache.shape[2]
    lnew = 0 if k is None else k.shape[1]
    if k is not None:
        k = k.contiguous()
        v = v.contiguous()
    if block_table is not None:
        extent, max_pages, bt_stride = k_cache.shape[0], block_table.shape[1], block_table.stride(0)
        cap = max_pages * k_cache.shape[1]
    else:
        extent, max_pages, bt_stride = k_cache.shape[1], 0, 0
        cap = extent
    if max_seqlen_k is None:
        max_seqlen_k = cap
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, lq, hq, d), dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, hq, lq), dtype=torch.float32, device=q.device)
    if rotary_cos is not None:
        _cuda(rotary_cos, rotary_sin)
        rotary_cos = rotary_cos.contiguous()
        rotary_sin = rotary_sin.contiguous()
        ws_bytes = lib.pa_fwd_kvcache_rotary_workspace_size(B, lq, hq, hkv, d, lnew, max_seqlen_k,
                                                            num_splits)
        if workspace is None:
            workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
        ws_len = workspace.numel() * workspace.element_size()
        _check(lib.pa_fwd_kvcache_rotary(
            _ptr(q), q.stride(0), q.stride(1), q.stride(2), _t4(k_cache), _t4(v_cache), _ptr(k),
            _ptr(v), lnew, _ptr(cache_seqlens), _ptr(block_table), bt_stride, max_pages,
            _page_size(k_cache, block_table), B, lq, hq, hkv, d, extent, max_seqlen_k,
            _ptr(rotary_cos), _ptr(rotary_sin),
            rotary_cos.shape[0], 2 * rotary_cos.shape[1], int(bool(rotary_interleaved)),
            float(scale), int(bool(causal)), int(num_splits), _ptr(out), _ptr(lse),
            _ptr(workspace), ws_len, _ptr(err), _dtype(q), _stream(q)))
        return out, lse
    ws_bytes = lib.pa_fwd_kvcache_workspace_size(B, lq, hq, hkv, d, max_seqlen_k, num_splits)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pa_fwd_kvcache(_ptr(q), q.stride(0), q.stride(1), q.stride(2), _t4(k_cache),
                              _t4(v_cache), _ptr(k), _ptr(v), lnew, _ptr(cache_seqlens),
                              _ptr(block_table), bt_stride, max_pages,
                              _page_size(k_cache, block_table), B, lq, hq, hkv, d, extent,
                              max_seqlen_k, float(scale), int(bool(causal)), int(num_splits),
                              _ptr(out), _ptr(lse), _ptr(workspace), ws_len, _ptr(err),
                              _dtype(q), _stream(q)))
    return out, lse


def pa_fwd_kvcache_noalloc(q, k_cache, v_cache, cache_seqlens, out, block_table=None, k=None,
                           v=None, lse=None, scale=None, causal=False, num_splits=0, err=None,
                           max_seqlen_k=None):
    """pa_fwd_kvcache for callers that cannot allocate device memory.

    The caller passes every tensor, including ``out`` (and optionally ``lse``);
    this wrapper allocates nothing and the library uses its own fixed split
    scratch (``PA_NOALLOC_SCRATCH_BYTES``).  Calls that could overlap on the GPU
    must be serialised by the caller because they share that scratch.
    """
    lib = load_library()
    _cuda(q, k_cache, v_cache, cache_seqlens, block_table, k, v, out, lse)
    B, lq, hq, d = q.shape
    hkv = k_cache.shape[2]
    lnew = 0 if k is None else k.shape[1]
    # the library reads k/v as contiguous [B, Lnew, Hkv, D]; a strided view
    # cannot be copied here (this call allocates nothing), so it is refused
    for name, t in (("k", k), ("v", v)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"pa_fwd_kvcache_noalloc: {name} must be contiguous")
    if block_table is not None:
        extent, max_pages, bt_stride = k_cache.shape[0], block_table.shape[1], block_table.stride(0)
        cap = max_pages * k_cache.shape[1]
    else:
        extent, max_pages, bt_stride = k_cache.shape[1], 0, 0
        cap = extent
    if max_seqlen_k is None:
        max_seqlen_k = cap
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(lib.pa_fwd_kvcache_noalloc(_ptr(q), q.stride(0), q.stride(1), q.stride(2),
                                      _t4(k_cache), _t4(v_cache), _ptr(k), _ptr(v), lnew,
                                      _ptr(cache_seqlens), _ptr(block_table), bt_stride,
                                      max_pages, _page_size(k_cache, block_table), B, lq, hq, hkv,
                                      d, extent, max_seqlen_k,
                                      float(scale), int(bool(causal)), int(num_splits),
                                      _ptr(out), _ptr(lse), _ptr(err), _dtype(q), _stream(q)))
    return out, lse


def pa_fwd_varlen_unified(q, k_cache, v_cache, cu_seqlens_q, seqlens_k, block_table,
                          max_seqlen_q, max_seqlen_k, scale=None, causal=True, out=None, lse=None,
                          workspace=None, err=None, return_lse=True):
    """One launch over a mixed prefill/decode batch; returns ``(out, lse)``.

    q ``[total_q, Hq, D]`` packed by ``cu_seqlens_q [B+1]``; ``seqlens_k [B]``
    counts each sequence's keys including its new chunk (already in the cache).
    """
    lib = load_library()
    _cuda(q, k_cache, v_cache, cu_seqlens_q, seqlens_k, block_table)
    total_q, hq, d = q.shape
    hkv = k_cache.shape[2]
    B = cu_seqlens_q.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((total_q, hq, d), dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((hq, total_q), dtype=torch.float32, device=q.device)
    ws_bytes = lib.pa_fwd_varlen_workspace_size(B, total_q, max_seqlen_q, hq, hkv, d,
                                                max_seqlen_k)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pa_fwd_varlen_unified(_ptr(q), q.stride(0), q.stride(1), _t4(k_cache),
                                     _t4(v_cache), _ptr(cu_seqlens_q), _ptr(seqlens_k),
                                     _ptr(block_table), block_table.stride(0),
                                     block_table.shape[1], k_cache.shape[1], B, total_q,
                                     max_seqlen_q, max_seqlen_k,
                                     hq, hkv, d, k_cache.shape[0], float(scale),
                                     int(bool(causal)), _ptr(out), _ptr(lse), _ptr(workspace),
                                     ws_len, _ptr(err), _dtype(q), _stream(q)))
    return out, lse


def pa_split_combine(o_partial, lse_partial, out, lse=None, splits_per_seq=None):
    """Merge split partials: o_partial fp32 ``[S, B, Lq, Hq, D]``, lse_partial
    fp32 ``[S, B, Lq, Hq]`` into out ``[B, Lq, Hq, D]`` and lse ``[B, Hq, Lq]``."""
    lib = load_library()
    _cuda(o_partial, lse_partial, out, lse, splits_per_seq)
    S, B, lq, hq, d = o_partial.shape
    _check(lib.pa_split_combine(_ptr(o_partial.contiguous()), _ptr(lse_partial.contiguous()),
                                _ptr(splits_per_seq), S, B, lq, hq, d, _ptr(out), _ptr(lse),
                                _dtype(out), _stream(out)))
    return out, lse
