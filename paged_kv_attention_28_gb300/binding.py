"""ctypes binding to ``libpkvattn.so``: the C ABI declared in ``include/pkv_attn.h``.

This layer only marshals arguments. It turns torch CUDA tensors into device
pointers, checks shapes and dtypes on the host, and passes the current CUDA
stream. Every step of the computation runs in the library's kernels. If the
library is missing, importing this module raises; nothing falls back to
another implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpkvattn.so")

PKV_F32 = 0
PKV_BF16 = 1
PKV_FP8_E4M3 = 2
PKV_OK = 0
PKV_ERR_INVALID_ARG = -1
PKV_ERR_UNSUPPORTED = -2
PKV_ERR_WORKSPACE = -3
PKV_ERR_LAUNCH = -4
PKV_ERR_DEVICE = -5
PKV_DEVERR_BAD_PAGE = 1
PKV_DEVERR_BAD_LEN = 2
PKV_DEVERR_TIMEOUT = 4

EXPORTS = [
    "attn_status_string", "attn_last_cuda_error_string", "attn_decode_num_splits", "attn_decode_workspace_size",
    "attn_decode_paged", "attn_decode_paged_unified_max", "attn_merge_states",
    "attn_prefill_causal", "attn_cascade_workspace_size", "attn_decode_cascade",
    "attn_decode_paged_noalloc", "attn_decode_paged_fp8", "attn_prefill_paged_chunk",
    "attn_flat_gemm", "attn_flat_gemm_num_splits", "attn_debug_decode_stall",
]


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = f"{what}: {status_string(status)} ({status})"
        if status == PKV_ERR_LAUNCH:
            msg += f": {lib.attn_last_cuda_error_string().decode()}"
        super().__init__(msg)
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m paged_kv_attention_28_gb300.build` "
            "(the CUDA path has no fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_status_string.argtypes = [i32]
    lib.attn_last_cuda_error_string.restype = ctypes.c_char_p
    lib.attn_last_cuda_error_string.argtypes = []
    lib.attn_decode_num_splits.restype = i32
    lib.attn_decode_num_splits.argtypes = [i32] * 8
    lib.attn_decode_workspace_size.restype = sz
    lib.attn_decode_workspace_size.argtypes = [i32] * 8
    lib.attn_decode_paged.restype = i32
    lib.attn_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp] + [i32] * 7 + [f32, i32, i32, vp, sz, vp, vp]
    lib.attn_decode_paged_unified_max.restype = i32
    lib.attn_decode_paged_unified_max.argtypes = ([vp, vp, vp, vp, vp, vp, vp] + [i32] * 7 +
                                                  [f32, i32, i32, f32, vp, vp, sz, vp, vp])
    lib.attn_decode_paged_noalloc.restype = i32
    lib.attn_decode_paged_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp] + [i32] * 7 + [f32, i32, i32, vp, vp]
    lib.attn_decode_paged_fp8.restype = i32
    lib.attn_decode_paged_fp8.argtypes = [vp] * 9 + [i32] * 7 + [f32, i32, vp, sz, vp, vp]
    lib.attn_merge_states.restype = i32
    lib.attn_merge_states.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, vp]
    lib.attn_prefill_causal.restype = i32
    lib.attn_prefill_causal.argtypes = [vp, vp, vp, vp, vp] + [i32] * 5 + [f32, i32, vp, vp]
    lib.attn_prefill_paged_chunk.restype = i32
    lib.attn_prefill_paged_chunk.argtypes = [vp] * 7 + [i32] * 8 + [f32, i32, vp, vp]
    lib.attn_cascade_workspace_size.restype = sz
    lib.attn_cascade_workspace_size.argtypes = [i32] * 7
    lib.attn_decode_cascade.restype = i32
    lib.attn_decode_cascade.argtypes = ([vp, vp, vp, vp, i32, vp, vp, vp, vp] + [i32] * 7 +
                                        [f32, i32, vp, sz, vp, vp])
    lib.attn_flat_gemm.restype = i32
    lib.attn_flat_gemm.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp]
    lib.attn_debug_decode_stall.restype = i32
    lib.attn_debug_decode_stall.argtypes = [i32, ctypes.c_ulonglong]
    lib.attn_flat_gemm_num_splits.restype = i32
    lib.attn_flat_gemm_num_splits.argtypes = [i32, i32, i32]
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.attn_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != PKV_OK:
        raise AttnError(status, what)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return PKV_F32
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


# --------------------------------------------------------------------------- decode

def decode_num_splits(batch, max_blocks, n_qo_heads, n_kv_heads, head_dim, page_size, num_splits=0,
                      dtype=PKV_BF16):
    r = lib.attn_decode_num_splits(batch, max_blocks, n_qo_heads, n_kv_heads, head_dim, page_size,
                                   num_splits, dtype)
    _check(min(r, 0), "attn_decode_num_splits")
    return r


def decode_workspace_size(batch, max_blocks, n_qo_heads, n_kv_heads, head_dim, page_size,
                          num_splits=0, dtype=PKV_BF16) -> int:
    n = lib.attn_decode_workspace_size(batch, max_blocks, n_qo_heads, n_kv_heads, head_dim,
                                       page_size, num_splits, dtype)
    if n == ctypes.c_size_t(-1).value:
        raise AttnError(PKV_ERR_INVALID_ARG, "attn_decode_workspace_size")
    return n


def alloc_workspace(nbytes: int, device) -> torch.Tensor | None:
    """A 256-byte aligned device buffer (torch's allocator aligns to at least 512 bytes)."""
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def decode_paged(q, k_pages, v_pages, block_table, kv_lens, scale, num_splits=0, out=None,
                 lse=None, workspace=None, err_flag=None, stream=None, unified_phi=None,
                 fallback_count=None):
    """Paged decode through ``attn_decode_paged`` (or the unified-max variant when
    ``unified_phi`` is given). Returns ``(out, lse)``."""
    B, Hq, D = q.shape
    num_pages, Hkv, P, D2 = k_pages.shape
    assert D2 == D
    max_blocks = block_table.shape[1]
    _need(q, "q")
    _need(k_pages, "k_pages", q.dtype)
    _need(v_pages, "v_pages", q.dtype, k_pages.shape)
    _need(block_table, "block_table", torch.int32, (B, max_blocks))
    _need(kv_lens, "kv_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    ws_bytes = decode_workspace_size(B, max_blocks, Hq, Hkv, D, P, num_splits, _dt(q))
    if workspace is None:
        workspace = alloc_workspace(ws_bytes, q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = [_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(kv_lens), _ptr(out),
            _ptr(lse), B, max_blocks, num_pages, Hq, Hkv, D, P, float(scale), int(num_splits), _dt(q)]
    if unified_phi is None:
        st = lib.attn_decode_paged(*args, _ptr(workspace), wsz, _ptr(err_flag), _stream(stream))
        _check(st, "attn_decode_paged")
    else:
        st = lib.attn_decode_paged_unified_max(*args, float(unified_phi), _ptr(fallback_count),
                                               _ptr(workspace), wsz, _ptr(err_flag), _stream(stream))
        _check(st, "attn_decode_paged_unified_max")
    return out, lse


def decode_paged_fp8(q, k_codes, v_codes, k_scale, v_scale, block_table, kv_lens, scale,
                     num_splits=0, out=None, lse=None, workspace=None, err_flag=None, stream=None):
    """Paged decode over FP8 E4M3 pools through ``attn_decode_paged_fp8``.

    ``q`` bf16 ``[B, Hq, D]``; ``k_codes``/``v_codes`` uint8 ``[num_pages, Hkv, P, D]``;
    ``k_scale``/``v_scale`` float32 ``[num_pages, Hkv]``. Returns ``(out, lse)``."""
    B, Hq, D = q.shape
    num_pages, Hkv, P, D2 = k_codes.shape
    assert D2 == D
    max_blocks = block_table.shape[1]
    _need(q, "q", torch.bfloat16)
    _need(k_codes, "k_codes", torch.uint8)
    _need(v_codes, "v_codes", torch.uint8, k_codes.shape)
    _need(k_scale, "k_scale", torch.float32, (num_pages, Hkv))
    _need(v_scale, "v_scale", torch.float32, (num_pages, Hkv))
    _need(block_table, "block_table", torch.int32, (B, max_blocks))
    _need(kv_lens, "kv_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    ws_bytes = decode_workspace_size(B, max_blocks, Hq, Hkv, D, P, num_splits, PKV_FP8_E4M3)
    if workspace is None:
        workspace = alloc_workspace(ws_bytes, q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.attn_decode_paged_fp8(_ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scale),
                                   _ptr(v_scale), _ptr(block_table), _ptr(kv_lens), _ptr(out),
                                   _ptr(lse), B, max_blocks, num_pages, Hq, Hkv, D, P, float(scale),
                                   int(num_splits), _ptr(workspace), wsz, _ptr(err_flag),
                                   _stream(stream))
    _check(st, "attn_decode_paged_fp8")
    return out, lse


def merge_states(out_a, lse_a, out_b, lse_b, out=None, lse=None, out_dtype=torch.float32,
                 stream=None):
    """Pairwise log-sum-exp merge through ``attn_merge_states``."""
    D = out_a.shape[-1]
    rows = out_a.numel() // D
    for t, n in ((out_a, "out_a"), (out_b, "out_b")):
        _need(t, n, torch.float32, out_a.shape)
    for t, n in ((lse_a, "lse_a"), (lse_b, "lse_b")):
        _need(t, n, torch.float32, out_a.shape[:-1])
    if out is None:
        out = torch.empty(out_a.shape, dtype=out_dtype, device=out_a.device)
    if lse is None:
        lse = torch.empty(lse_a.shape, dtype=torch.float32, device=out_a.device)
    st = lib.attn_merge_states(_ptr(out_a), _ptr(lse_a), _ptr(out_b), _ptr(lse_b), _ptr(out),
                               _ptr(lse), rows, D, _dt(out), _stream(stream))
    _check(st, "attn_merge_states")
    return out, lse


# --------------------------------------------------------------------------- prefill

def prefill_causal(q, k, v, scale, out=None, lse=None, err_flag=None, stream=None):
    """Causal prefill through ``attn_prefill_causal``. ``q, k, v`` are ``[B, T, H, D]``."""
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    _need(q, "q")
    _need(k, "k", q.dtype, (B, T, Hkv, D))
    _need(v, "v", q.dtype, (B, T, Hkv, D))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    st = lib.attn_prefill_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, T, Hq, Hkv, D,
                                 float(scale), _dt(q), _ptr(err_flag), _stream(stream))
    _check(st, "attn_prefill_causal")
    return out, lse


def prefill_paged_chunk(q, k_pages, v_pages, block_table, prefix_lens, scale, out=None, lse=None,
                        err_flag=None, stream=None):
    """Chunked prefill over the paged cache through ``attn_prefill_paged_chunk``.

    ``q`` ``[B, C, Hq, D]``; the new tokens' K/V are already in the pools. Returns
    ``(out, lse)`` with ``lse`` ``[B, Hq, C]``."""
    B, C, Hq, D = q.shape
    num_pages, Hkv, P, D2 = k_pages.shape
    assert D2 == D
    max_blocks = block_table.shape[1]
    _need(q, "q")
    _need(k_pages, "k_pages", q.dtype)
    _need(v_pages, "v_pages", q.dtype, k_pages.shape)
    _need(block_table, "block_table", torch.int32, (B, max_blocks))
    _need(prefix_lens, "prefix_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, C), dtype=torch.float32, device=q.device)
    st = lib.attn_prefill_paged_chunk(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                      _ptr(prefix_lens), _ptr(out), _ptr(lse), B, C, max_blocks,
                                      num_pages, Hq, Hkv, D, P, float(scale), _dt(q), _ptr(err_flag),
                                      _stream(stream))
    _check(st, "attn_prefill_paged_chunk")
    return out, lse


# --------------------------------------------------------------------------- cascade

def cascade_workspace_size(n_requests, prefix_len, max_suffix_blocks, n_qo_heads, n_kv_heads,
                           head_dim, page_size) -> int:
    n = lib.attn_cascade_workspace_size(n_requests, prefix_len, max_suffix_blocks, n_qo_heads,
                                        n_kv_heads, head_dim, page_size)
    if n == ctypes.c_size_t(-1).value:
        raise AttnError(PKV_ERR_INVALID_ARG, "attn_cascade_workspace_size")
    return n


def decode_cascade(q, k_pages, v_pages, prefix_table, prefix_len, suffix_table, suffix_lens, scale,
                   out=None, lse=None, workspace=None, err_flag=None, stream=None):
    """Shared-prefix decode through ``attn_decode_cascade``. Returns ``(out, lse)``."""
    R, Hq, D = q.shape
    num_pages, Hkv, P, _ = k_pages.shape
    ms = suffix_table.shape[1]
    _need(q, "q")
    _need(k_pages, "k_pages", q.dtype)
    _need(v_pages, "v_pages", q.dtype, k_pages.shape)
    _need(suffix_table, "suffix_table", torch.int32, (R, ms))
    _need(suffix_lens, "suffix_lens", torch.int32, (R,))
    if prefix_len > 0:
        _need(prefix_table, "prefix_table", torch.int32)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((R, Hq), dtype=torch.float32, device=q.device)
    nb = cascade_workspace_size(R, prefix_len, ms, Hq, Hkv, D, P)
    if workspace is None:
        workspace = alloc_workspace(nb, q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.attn_decode_cascade(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(prefix_table),
                                 int(prefix_len), _ptr(suffix_table), _ptr(suffix_lens), _ptr(out),
                                 _ptr(lse), R, ms, num_pages, Hq, Hkv, D, P, float(scale), _dt(q),
                                 _ptr(workspace), wsz, _ptr(err_flag), _stream(stream))
    _check(st, "attn_decode_cascade")
    return out, lse


# --------------------------------------------------------------------------- flat GEMM

def flat_gemm_num_splits(m, n, k) -> int:
    """CTAs that share K (one cluster) per 128-row tile of ``w`` for this shape."""
    r = lib.attn_flat_gemm_num_splits(int(m), int(n), int(k))
    if r < 0:
        raise AttnError(r, "attn_flat_gemm_num_splits")
    return r


def flat_gemm(x, w, out=None, err_flag=None, stream=None):
    """``y = x w^T`` through ``attn_flat_gemm``: ``x`` ``[m, k]``, ``w`` ``[n, k]``, bf16."""
    m, k = x.shape
    n = w.shape[0]
    _need(x, "x")
    _need(w, "w", x.dtype, (n, k))
    if out is None:
        out = torch.empty((m, n), dtype=x.dtype, device=x.device)
    _need(out, "out", x.dtype, (m, n))
    st = lib.attn_flat_gemm(_ptr(x), _ptr(w), _ptr(out), m, n, k, _dt(x), _ptr(err_flag), _stream(stream))
    _check(st, "attn_flat_gemm")
    return out


def debug_decode_stall(page: int, wait_limit_ns: int = 0) -> None:
    """Failure-handling hook for tests: ``attn_debug_decode_stall`` (``page = -1`` turns it off)."""
    _check(lib.attn_debug_decode_stall(int(page), int(wait_limit_ns)), "attn_debug_decode_stall")
