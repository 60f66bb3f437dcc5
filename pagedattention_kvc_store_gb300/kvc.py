"""Thin ctypes binding of libkvc (the C ABI in include/kvc.h).

Argument marshalling only: every step of the store and of the attention runs in the CUDA
kernels behind these calls.  Tensors are torch CUDA tensors; the functions pass their
device pointers and the current CUDA stream.  There is no CPU path: without the compiled
library or a GPU these functions raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

from . import build as _build

KVC_BF16 = 0
KVC_F32 = 1

STATUS = {0: "KVC_OK", 1: "KVC_ERR_INVALID_ARG", 2: "KVC_ERR_UNSUPPORTED",
          3: "KVC_ERR_WORKSPACE", 4: "KVC_ERR_CUDA", 5: "KVC_ERR_DEVICE",
          6: "KVC_ERR_OUT_OF_RANGE"}
KVC_ERR_OUT_OF_RANGE = 6

# Every entry point declared in include/kvc.h.
EXPORTS = ("kvc_status_string", "kvc_last_error", "kvc_slot_mapping", "kvc_store",
           "kvc_decode", "kvc_decode_plan", "kvc_merge", "kvc_append", "kvc_device_errors",
           "kvc_decode_noalloc", "kvc_decode_shared_prefix", "kvc_decode_shared_prefix_plan",
           "kvc_validate_workspace_size", "kvc_validate", "kvc_copy_pages", "kvc_store_int8",
           "kvc_decode_int8", "kvc_decode_int8_plan", "kvc_append_int8",
           "kvc_append_store", "kvc_shared_prefix_groups", "kvc_decode_store",
           "kvc_selftest_wait", "kvc_decode_int8_store", "kvc_set_error_word")

# Size of the library's own split-partials scratch used by kvc_decode_noalloc (bytes).
NOALLOC_SCRATCH_BYTES = 8 << 20


class KvcError(RuntimeError):
    def __init__(self, call: str, status: int, detail: str):
        super().__init__(f"{call}: {STATUS.get(status, status)}: {detail}")
        self.call = call
        self.status = status


KVC_NHD = 0
KVC_HND = 1
LAYOUTS = {"nhd": KVC_NHD, "hnd": KVC_HND}


class PoolDesc(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("layout", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libkvc.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libkvc.so not found at {path}")
            L = ctypes.CDLL(path)
            i32, p, sz = ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
            f = ctypes.c_float
            L.kvc_status_string.restype = ctypes.c_char_p
            L.kvc_status_string.argtypes = [ctypes.c_int]
            L.kvc_last_error.restype = ctypes.c_char_p
            L.kvc_last_error.argtypes = []
            L.kvc_slot_mapping.restype = ctypes.c_int
            L.kvc_slot_mapping.argtypes = [p, p, i32, p, p, i32, i32, i32, i32, p]
            L.kvc_store.restype = ctypes.c_int
            L.kvc_store.argtypes = [p, p, PoolDesc, p, p, p, i32, p]
            L.kvc_decode.restype = ctypes.c_int
            L.kvc_decode.argtypes = [p, i32, p, p, p, PoolDesc, p, i32, p, i32, i32, i32, f,
                                     i32, p, sz, p]
            L.kvc_decode_store.restype = ctypes.c_int
            L.kvc_decode_store.argtypes = [p, i32, p, p, p, p, p, PoolDesc, p, i32, p, i32, i32,
                                           i32, f, i32, p, sz, p]
            L.kvc_decode_plan.restype = ctypes.c_int
            L.kvc_decode_plan.argtypes = [i32, i32, PoolDesc, i32, i32,
                                          ctypes.POINTER(i32), ctypes.POINTER(i32),
                                          ctypes.POINTER(sz)]
            L.kvc_merge.restype = ctypes.c_int
            L.kvc_merge.argtypes = [p, i32, p, p, i32, i32, i32, p, p]
            L.kvc_append.restype = ctypes.c_int
            L.kvc_append.argtypes = [p, i32, p, p, p, PoolDesc, p, i32, p, p, i32, i32, i32,
                                     i32, i32, f, p]
            L.kvc_decode_noalloc.restype = ctypes.c_int
            L.kvc_decode_noalloc.argtypes = [p, i32, p, p, p, PoolDesc, p, i32, p, i32, i32,
                                             i32, f, i32, p]
            L.kvc_decode_shared_prefix.restype = ctypes.c_int
            L.kvc_decode_shared_prefix.argtypes = [p, i32, p, p, p, PoolDesc, p, i32, p, i32,
                                                   i32, i32, f, p, p, p, i32, i32, i32, p, sz, p]
            L.kvc_shared_prefix_groups.restype = ctypes.c_int
            L.kvc_shared_prefix_groups.argtypes = [p, i32, p, i32, i32, i32, p, p, p, p, p]
            L.kvc_decode_shared_prefix_plan.restype = ctypes.c_int
            L.kvc_decode_shared_prefix_plan.argtypes = [i32, i32, PoolDesc, i32, i32, i32,
                                                        ctypes.POINTER(sz)]
            L.kvc_selftest_wait.restype = ctypes.c_int
            L.kvc_selftest_wait.argtypes = [p]
            L.kvc_device_errors.restype = ctypes.c_int
            L.kvc_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
            L.kvc_set_error_word.restype = ctypes.c_int
            L.kvc_set_error_word.argtypes = [p]
            L.kvc_store_int8.restype = ctypes.c_int
            L.kvc_store_int8.argtypes = [p, p, p, p, PoolDesc, p, p, p, i32, p]
            L.kvc_decode_int8_plan.restype = ctypes.c_int
            L.kvc_decode_int8_plan.argtypes = [i32, i32, PoolDesc, i32, i32,
                                               ctypes.POINTER(i32), ctypes.POINTER(i32),
                                               ctypes.POINTER(sz)]
            L.kvc_decode_int8.restype = ctypes.c_int
            L.kvc_decode_int8.argtypes = [p, i32, p, p, p, p, p, PoolDesc, p, i32, p, i32, i32,
                                          i32, f, i32, p, sz, p]
            L.kvc_decode_int8_store.restype = ctypes.c_int
            L.kvc_decode_int8_store.argtypes = [p, i32, p, p, p, p, p, p, p, PoolDesc, p, i32, p,
                                                i32, i32, i32, f, i32, p, sz, p]
            L.kvc_append_int8.restype = ctypes.c_int
            L.kvc_append_int8.argtypes = [p, i32, p, p, p, p, p, PoolDesc, p, i32, p, p, i32,
                                          i32, i32, i32, i32, f, p]
            L.kvc_append_store.restype = ctypes.c_int
            L.kvc_append_store.argtypes = [p, i32, p, p, p, p, p, PoolDesc, p, i32, p, p, i32,
                                           i32, i32, i32, i32, f, p]
            L.kvc_copy_pages.restype = ctypes.c_int
            L.kvc_copy_pages.argtypes = [p, p, PoolDesc, p, p, i32, p]
            L.kvc_validate_workspace_size.restype = ctypes.c_int
            L.kvc_validate_workspace_size.argtypes = [PoolDesc, ctypes.POINTER(sz)]
            L.kvc_validate.restype = ctypes.c_int
            L.kvc_validate.argtypes = [PoolDesc, p, i32, p, i32, p, i32, p, sz,
                                       ctypes.POINTER(ctypes.c_int64), p]
            _lib = L
    return _lib


def _check(call: str, status: int) -> None:
    if status != 0:
        detail = lib().kvc_last_error().decode(errors="replace")
        raise KvcError(call, status, detail)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda(name: str, t: torch.Tensor, dtype=None, contiguous=True) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libkvc has no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _reachable(name: str, t: torch.Tensor, dtype=None) -> torch.Tensor:
    """An argument the kernels may reach in host memory: a CUDA tensor, or a pinned host
    tensor that they read or write across the host link directly."""
    if isinstance(t, torch.Tensor) and not t.is_cuda:
        if not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or a pinned host tensor")
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        return t
    return _cuda(name, t, dtype)


def _decode_out(t: torch.Tensor) -> torch.Tensor:
    """`out` of the decode calls (a CUDA tensor or a pinned host tensor)."""
    return _reachable("out", t)


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _out_dtype(out: torch.Tensor) -> int:
    if out.dtype == torch.bfloat16:
        return KVC_BF16
    if out.dtype == torch.float32:
        return KVC_F32
    raise TypeError(f"out must be bfloat16 or float32, got {out.dtype}")


def pool_desc(k_pool: torch.Tensor, layout: str = "nhd") -> PoolDesc:
    """Descriptor of a bf16 pool: [num_pages, page_size, kv_heads, head_dim] (layout "nhd")
    or [num_pages, kv_heads, page_size, head_dim] (layout "hnd")."""
    if k_pool.dim() != 4:
        raise ValueError("a pool is a 4-D tensor")
    if layout not in LAYOUTS:
        raise ValueError(f"layout {layout!r}: 'nhd' or 'hnd'")
    n, a, b, d = (int(x) for x in k_pool.shape)
    page_size, kv_heads = (a, b) if layout == "nhd" else (b, a)
    return PoolDesc(n, page_size, kv_heads, d, LAYOUTS[layout])


def kvc_slot_mapping(slot_mapping: torch.Tensor, block_table: torch.Tensor,
                     context_lens: torch.Tensor, q_indptr: Optional[torch.Tensor],
                     page_size: int, max_q_len: int = 1, stream=None) -> None:
    _cuda("slot_mapping", slot_mapping, torch.int32)
    _reachable("block_table", block_table, torch.int32)
    _reachable("context_lens", context_lens, torch.int32)
    if q_indptr is not None:
        _reachable("q_indptr", q_indptr, torch.int32)
    S = int(context_lens.shape[0])
    _check("kvc_slot_mapping", lib().kvc_slot_mapping(
        _ptr(slot_mapping), _ptr(block_table), int(block_table.shape[1]), _ptr(context_lens),
        _ptr(q_indptr), S, int(slot_mapping.shape[0]), int(max_q_len), int(page_size),
        _stream(stream)))


def kvc_store(k_pool: torch.Tensor, v_pool: torch.Tensor, k_new: torch.Tensor,
              v_new: torch.Tensor, slot_mapping: torch.Tensor, stream=None,
              layout: str = "nhd") -> None:
    _cuda("k_pool", k_pool, torch.bfloat16)
    _cuda("v_pool", v_pool, torch.bfloat16)
    _reachable("k_new", k_new, torch.bfloat16)
    _reachable("v_new", v_new, torch.bfloat16)
    _cuda("slot_mapping", slot_mapping, torch.int32)
    _check("kvc_store", lib().kvc_store(
        _ptr(k_pool), _ptr(v_pool), pool_desc(k_pool, layout), _ptr(k_new), _ptr(v_new),
        _ptr(slot_mapping), int(slot_mapping.shape[0]), _stream(stream)))


def int8_pool_desc(k_codes: torch.Tensor, layout: str = "nhd") -> PoolDesc:
    """Descriptor of an int8 code pool: [num_pages, page_size, kv_heads, head_dim] (layout
    "nhd") or [num_pages, kv_heads, page_size, head_dim] (layout "hnd")."""
    if k_codes.dim() != 4 or k_codes.dtype != torch.int8:
        raise ValueError("INT8 codes are an int8 4-D tensor")
    if layout not in LAYOUTS:
        raise ValueError(f"layout {layout!r}: 'nhd' or 'hnd'")
    n, a, b, d = (int(x) for x in k_codes.shape)
    p, h = (a, b) if layout == "nhd" else (b, a)
    return PoolDesc(n, p, h, d, LAYOUTS[layout])


def _int8_pools(k_codes, v_codes, k_scales, v_scales, layout="nhd"):
    pool = int8_pool_desc(k_codes, layout)
    for name, t, dt in (("k_codes", k_codes, torch.int8), ("v_codes", v_codes, torch.int8),
                        ("k_scales", k_scales, torch.float32),
                        ("v_scales", v_scales, torch.float32)):
        _cuda(name, t, dt)
    want = (pool.num_pages, pool.kv_heads, pool.page_size)
    if tuple(k_scales.shape) != want or tuple(v_scales.shape) != want:
        raise ValueError(f"scales are [num_pages, kv_heads, page_size] = {want}")
    return pool


def kvc_store_int8(k_codes: torch.Tensor, v_codes: torch.Tensor, k_scales: torch.Tensor,
                   v_scales: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                   slot_mapping: torch.Tensor, stream=None, layout: str = "nhd") -> None:
    pool = _int8_pools(k_codes, v_codes, k_scales, v_scales, layout)
    _cuda("k_new", k_new, torch.bfloat16)
    _cuda("v_new", v_new, torch.bfloat16)
    _cuda("slot_mapping", slot_mapping, torch.int32)
    _check("kvc_store_int8", lib().kvc_store_int8(
        _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), pool, _ptr(k_new),
        _ptr(v_new), _ptr(slot_mapping), int(slot_mapping.numel()), _stream(stream)))


def kvc_decode_int8_plan(num_seqs: int, q_heads: int, pool: PoolDesc, max_ctx: int,
                         num_splits: int = 0) -> Tuple[int, int, int]:
    """(CTAs, block, workspace_bytes) of kvc_decode_int8's plan: per kv head, the positions of
    all sequences in 64-position blocks are cut into runs of equal cost (num_splits 0: one
    wave of resident CTAs; 1: one CTA per (sequence, kv head), no workspace; n: n runs per
    sequence)."""
    splits, chunk, ws = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t()
    _check("kvc_decode_int8_plan", lib().kvc_decode_int8_plan(
        int(num_seqs), int(q_heads), pool, int(max_ctx), int(num_splits), ctypes.byref(splits),
        ctypes.byref(chunk), ctypes.byref(ws)))
    return splits.value, chunk.value, ws.value


def kvc_decode_int8(out: torch.Tensor, q: torch.Tensor, k_codes: torch.Tensor,
                    v_codes: torch.Tensor, k_scales: torch.Tensor, v_scales: torch.Tensor,
                    block_table: torch.Tensor, context_lens: torch.Tensor, max_ctx: int,
                    scale: float = 0.0, num_splits: int = 0,
                    workspace: Optional[torch.Tensor] = None, stream=None,
                    layout: str = "nhd") -> None:
    pool = _int8_pools(k_codes, v_codes, k_scales, v_scales, layout)
    _decode_out(out)
    _reachable("q", q, torch.bfloat16)
    _reachable("block_table", block_table, torch.int32)
    _reachable("context_lens", context_lens, torch.int32)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("kvc_decode_int8", lib().kvc_decode_int8(
        _ptr(out), _out_dtype(out), _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales),
        _ptr(v_scales), pool, _ptr(block_table), int(block_table.shape[1]), _ptr(context_lens),
        int(context_lens.shape[0]), int(max_ctx), int(q.shape[1]), float(scale),
        int(num_splits), _ptr(workspace), ws, _stream(stream)))


def kvc_decode_int8_store(out: torch.Tensor, q: torch.Tensor, k_new: torch.Tensor,
                          v_new: torch.Tensor, k_codes: torch.Tensor, v_codes: torch.Tensor,
                          k_scales: torch.Tensor, v_scales: torch.Tensor,
                          block_table: torch.Tensor, context_lens: torch.Tensor, max_ctx: int,
                          scale: float = 0.0, num_splits: int = 0,
                          workspace: Optional[torch.Tensor] = None, stream=None,
                          layout: str = "nhd") -> None:
    """Quantise and store each sequence's new token (k_new / v_new bf16 [S, Hkv, D]) into the
    INT8 pools and decode over them, in one call."""
    pool = _int8_pools(k_codes, v_codes, k_scales, v_scales, layout)
    _decode_out(out)
    _reachable("q", q, torch.bfloat16)
    _reachable("k_new", k_new, torch.bfloat16)
    _reachable("v_new", v_new, torch.bfloat16)
    _reachable("block_table", block_table, torch.int32)
    _reachable("context_lens", context_lens, torch.int32)
    ws = 0
    if workspace is not None:
        _cuda("workspace", workspace)
        ws = workspace.numel() * workspace.element_size()
    _check("kvc_decode_int8_store", lib().kvc_decode_int8_store(
        _ptr(out), _out_dtype(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_codes),
        _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), pool, _ptr(block_table),
        int(block_table.shape[1]), _ptr(context_lens), int(context_lens.shape[0]), int(max_ctx),
        int(q.shape[1]), float(scale), int(num_splits), _ptr(workspace), ws, _stream(stream)))


def kvc_append_int8(out: torch.Tensor, q: torch.Tensor, k_codes: torch.Tensor,
                    v_codes: torch.Tensor, k_scales: torch.Tensor, v_scales: torch.Tensor,
                    block_table: torch.Tensor, q_indptr: torch.Tensor,
                    context_lens: torch.Tensor, max_q_len: int, max_ctx: int,
                    scale: float = 0.0, stream=None, layout: str = "nhd") -> None:
    """kvc_append over INT8 pages (codes int8 [pages, P, Hkv, D], or [pages, Hkv, P, D] with
    layout "hnd"; scales fp32 [pages, Hkv, P])."""
    pool = _int8_pools(k_codes, v_codes, k_scales, v_scales, layout)
    _cuda("out", out)
    _cuda("q", q, torch.bfloat16)
    _cuda("block_table", block_table, torch.int32)
    _cuda("q_indptr", q_indptr, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    _check("kvc_append_int8", lib().kvc_append_int8(
        _ptr(out), _out_dtype(out), _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales),
        _ptr(v_scales), pool, _ptr(block_table), int(block_table.shape[1]), _ptr(q_indptr),
        _ptr(context_lens), int(context_lens.shape[0]), int(q.shape[0]), int(max_q_len),
        int(max_ctx), int(q.shape[1]), float(scale), _stream(stream)))


def kvc_copy_pages(k_pool: torch.Tensor, v_pool: torch.Tensor, src_pages: torch.Tensor,
                   dst_pages: torch.Tensor, stream=None,
                   layout: str = "nhd") -> None:
    """Copy-on-write: page dst_pages[i] of both pools receives page src_pages[i]."""
    _cuda("k_pool", k_pool, torch.bfloat16)
    _cuda("v_pool", v_pool, torch.bfloat16)
    _cuda("src_pages", src_pages, torch.int32)
    _cuda("dst_pages", dst_pages, torch.int32)
    if src_pages.numel() != dst_pages.numel():
        raise ValueError("src_pages and dst_pages differ in length")
    _check("kvc_copy_pages", lib().kvc_copy_pages(
        _ptr(k_pool), _ptr(v_pool), pool_desc(k_pool, layout), _ptr(src_pages),
        _ptr(dst_pages),
        int(src_pages.numel()), _stream(stream)))


def kvc_decode_plan(num_seqs: int, q_heads: int, pool: PoolDesc, max_ctx: int,
                    num_splits: int = 0) -> Tuple[int, int, int]:
    """(splits, chunk, workspace_bytes) that kvc_decode will use."""
    splits, chunk, ws = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t()
    _check("kvc_decode_plan", lib().kvc_decode_plan(
        int(num_seqs), int(q_heads), pool, int(max_ctx), int(num_splits),
        ctypes.byref(splits), ctypes.byref(chunk), ctypes.byref(ws)))
    return splits.value, chunk.value, ws.value


def kvc_decode(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
               block_table: torch.Tensor, context_lens: torch.Tensor, max_ctx: int,
               scale: float = 0.0, num_splits: int = 0,
               workspace: Optional[torch.Tensor] = None, stream=None,
               layout: str = "nhd") -> None:
    _decode_out(out)
    _reachable("q", q, torch.bfloat16)
    _cuda("k_pool", k_pool, torch.bfloat16)
    _cuda("v_pool", v_pool, torch.bfloat16)
    _reachable("block_table", block_table, torch.int32)
    _reachable("context_lens", context_lens, torch.int32)
    ws_bytes = 0
    if workspace is not None:
        _cuda("workspace", workspace)
        ws_bytes = workspace.numel() * workspace.element_size()
    _check("kvc_decode", lib().kvc_decode(
        _ptr(out), _out_dtype(out), _ptr(q), _ptr(k_pool), _ptr(v_pool),
        pool_desc(k_pool, layout),
        _ptr(block_table), int(block_table.shape[1]), _ptr(context_lens),
        int(context_lens.shape[0]), int(max_ctx), int(q.shape[1]), float(scale),
        int(num_splits), _ptr(workspace), ws_bytes, _stream(stream)))


def kvc_decode_store(out: torch.Tensor, q: torch.Tensor, k_new: torch.Tensor,
                     v_new: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                     block_table: torch.Tensor, context_lens: torch.Tensor, max_ctx: int,
                     scale: float = 0.0, num_splits: int = 0,
                     workspace: Optional[torch.Tensor] = None, stream=None,
                     layout: str = "nhd") -> None:
    """Store each sequence's new token (k_new / v_new [S, Hkv, D]) and decode, in one call."""
    _decode_out(out)
    _reachable("q", q, torch.bfloat16)
    _reachable("k_new", k_new, torch.bfloat16)
    _reachable("v_new", v_new, torch.bfloat16)
    _cuda("k_pool", k_pool, torch.bfloat16)
    _cuda("v_pool", v_pool, torch.bfloat16)
    _reachable("block_table", block_table, torch.int32)
    _reachable("context_lens", context_lens, torch.int32)
    ws_bytes = 0
    if workspace is not None:
        _cuda("workspace", workspace)
        ws_bytes = workspace.numel() * workspace.element_size()
    _check("kvc_decode_store", lib().kvc_decode_store(
        _ptr(out), _out_dtype(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool),
        _ptr(v_pool), pool_desc(k_pool, layout), _ptr(block_table), int(block_table.shape[1]),
        _ptr(context_lens), int(context_lens.shape[0]), int(max_ctx), int(q.shape[1]),
        float(scale), int(num_splits), _ptr(workspace), ws_bytes, _stream(stream)))


def kvc_merge(out: torch.Tensor, partial_o: torch.Tensor, partial_lse: torch.Tensor,
              lse_out: Optional[torch.Tensor] = None, stream=None) -> None:
    """partial_o [rows, splits, D] fp32, partial_lse [rows, splits] fp32 -> out [rows, D]."""
    _decode_out(out)
    _cuda("partial_o", partial_o, torch.float32)
    _cuda("partial_lse", partial_lse, torch.float32)
    if lse_out is not None:
        _cuda("lse_out", lse_out, torch.float32)
    rows, splits, d = (int(x) for x in partial_o.shape)
    _check("kvc_merge", lib().kvc_merge(
        _ptr(out), _out_dtype(out), _ptr(partial_o), _ptr(partial_lse), rows, splits, d,
        _ptr(lse_out), _stream(stream)))


def kvc_append(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
               block_table: torch.Tensor, q_indptr: torch.Tensor, context_lens: torch.Tensor,
               max_q_len: int, max_ctx: int, scale: float = 0.0, stream=None,
               layout: str = "nhd") -> None:
    _cuda("out", out)
    _cuda("q", q, torch.bfloat16)
    _cuda("k_pool", k_pool, torch.bfloat16)
    _cuda("v_pool", v_pool, torch.bfloat16)
    _cuda("block_table", block_table, torch.int32)
    _cuda("q_indptr", q_indptr, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    _check("kvc_append", lib().kvc_append(
        _ptr(out), _out_dtype(out), _ptr(q), _ptr(k_pool), _ptr(v_pool),
        pool_desc(k_pool, layout),
        _ptr(block_table), int(block_table.shape[1]), _ptr(q_indptr), _ptr(context_lens),
        int(context_lens.shape[0]), int(q.shape[0]), int(max_q_len), int(max_ctx),
        int(q.shape[1]), float(scale), _stream(stream)))


def kvc_append_store(out: torch.Tensor, q: torch.Tensor, k_new: torch.Tensor,
                     v_new: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                     block_table: torch.Tensor, q_indptr: torch.Tensor,
                     context_lens: torch.Tensor, max_q_len: int, max_ctx: int,
                     scale: float = 0.0, stream=None, layout: str = "nhd") -> None:
    """Store the chunk's K/V at their slots and attend (kvc_slot_mapping + kvc_store +
    kvc_append in one pass over the chunk)."""
    _cuda("out", out)
    _cuda("q", q, torch.bfloat16)
    _cuda("k_new", k_new, torch.bfloat16)
    _cuda("v_new", v_new, torch.bfloat16)
    _cuda("k_pool", k_pool, torch.bfloat16)
    _cuda("v_pool", v_pool, torch.bfloat16)
    _cuda("block_table", block_table, torch.int32)
    _cuda("q_indptr", q_indptr, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    _check("kvc_append_store", lib().kvc_append_store(
        _ptr(out), _out_dtype(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool),
        _ptr(v_pool), pool_desc(k_pool, layout), _ptr(block_table), int(block_table.shape[1]),
        _ptr(q_indptr), _ptr(context_lens), int(context_lens.shape[0]), int(q.shape[0]),
        int(max_q_len), int(max_ctx), int(q.shape[1]), float(scale), _stream(stream)))


def kvc_decode_noalloc(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor,
                       v_pool: torch.Tensor, block_table: torch.Tensor,
                       context_lens: torch.Tensor, max_ctx: int, scale: float = 0.0,
                       num_splits: int = 0, stream=None,
                       layout: str = "nhd") -> None:
    """kvc_decode without a workspace, for callers that may not allocate device memory:
    the split partials go to scratch memory the library owns (NOALLOC_SCRATCH_BYTES on
    every GPU that loads it).  Plans needing more scratch than that raise KvcError
    (KVC_ERR_WORKSPACE).  Calls share that scratch, so calls whose kernels could overlap
    on the GPU must be ordered by the caller; call it once on a device before any stream
    capture."""
    _decode_out(out)
    _cuda("q", q, torch.bfloat16)
    _cuda("k_pool", k_pool, torch.bfloat16)
    _cuda("v_pool", v_pool, torch.bfloat16)
    _cuda("block_table", block_table, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    _check("kvc_decode_noalloc", lib().kvc_decode_noalloc(
        _ptr(out), _out_dtype(out), _ptr(q), _ptr(k_pool), _ptr(v_pool),
        pool_desc(k_pool, layout),
        _ptr(block_table), int(block_table.shape[1]), _ptr(context_lens),
        int(context_lens.shape[0]), int(max_ctx), int(q.shape[1]), float(scale),
        int(num_splits), _stream(stream)))


def kvc_decode_shared_prefix_plan(num_seqs: int, q_heads: int, pool: PoolDesc, max_ctx: int,
                                  num_groups: int, max_prefix_len: int) -> int:
    """Workspace bytes kvc_decode_shared_prefix needs."""
    ws = ctypes.c_size_t()
    _check("kvc_decode_shared_prefix_plan", lib().kvc_decode_shared_prefix_plan(
        int(num_seqs), int(q_heads), pool, int(max_ctx), int(num_groups), int(max_prefix_len),
        ctypes.byref(ws)))
    return ws.value


def kvc_decode_shared_prefix(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor,
                             v_pool: torch.Tensor, block_table: torch.Tensor,
                             context_lens: torch.Tensor, max_ctx: int,
                             group_indptr: torch.Tensor, group_seqs: torch.Tensor,
                             prefix_len: torch.Tensor, max_group_size: int, max_prefix_len: int,
                             workspace: torch.Tensor, scale: float = 0.0, stream=None,
                             layout: str = "nhd") -> None:
    _cuda("out", out)
    _cuda("q", q, torch.bfloat16)
    _cuda("k_pool", k_pool, torch.bfloat16)
    _cuda("v_pool", v_pool, torch.bfloat16)
    _cuda("block_table", block_table, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    for name, t in (("group_indptr", group_indptr), ("group_seqs", group_seqs),
                    ("prefix_len", prefix_len)):
        _cuda(name, t, torch.int32)
    _cuda("workspace", workspace)
    _check("kvc_decode_shared_prefix", lib().kvc_decode_shared_prefix(
        _ptr(out), _out_dtype(out), _ptr(q), _ptr(k_pool), _ptr(v_pool),
        pool_desc(k_pool, layout),
        _ptr(block_table), int(block_table.shape[1]), _ptr(context_lens),
        int(context_lens.shape[0]), int(max_ctx), int(q.shape[1]), float(scale),
        _ptr(group_indptr), _ptr(group_seqs), _ptr(prefix_len), int(prefix_len.shape[0]),
        int(max_group_size), int(max_prefix_len), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def kvc_shared_prefix_groups(group_indptr: torch.Tensor, group_seqs: torch.Tensor,
                             prefix_len: torch.Tensor, num_groups: torch.Tensor,
                             block_table: torch.Tensor, context_lens: torch.Tensor,
                             page_size: int, max_members: int, stream=None) -> None:
    """Groups for kvc_decode_shared_prefix from the block tables (device prepass).  Outputs:
    group_indptr [S // 2 + 1], group_seqs [S], prefix_len [S // 2], num_groups [1], int32."""
    for name, t in (("group_indptr", group_indptr), ("group_seqs", group_seqs),
                    ("prefix_len", prefix_len), ("num_groups", num_groups),
                    ("block_table", block_table), ("context_lens", context_lens)):
        _cuda(name, t, torch.int32)
    S = int(context_lens.shape[0])
    if group_indptr.numel() < S // 2 + 1 or group_seqs.numel() < S or \
            prefix_len.numel() < S // 2 or num_groups.numel() < 1:
        raise ValueError("group outputs smaller than num_seqs / 2 groups need")
    _check("kvc_shared_prefix_groups", lib().kvc_shared_prefix_groups(
        _ptr(block_table), int(block_table.shape[1]), _ptr(context_lens), S, int(page_size),
        int(max_members), _ptr(group_indptr), _ptr(group_seqs), _ptr(prefix_len),
        _ptr(num_groups), _stream(stream)))


def kvc_selftest_wait(stream=None) -> None:
    """Enqueue the bounded-wait self-test (about a second); kvc_device_errors() then has bit
    1 << 12 set."""
    _check("kvc_selftest_wait", lib().kvc_selftest_wait(_stream(stream)))


def kvc_set_error_word(word) -> None:
    """Route the error bits of this thread's later calls into `word` (a 4-byte int32/uint32
    device tensor of one element, owned by the caller), or back to the library's own words with
    None."""
    if word is None:
        _check("kvc_set_error_word", lib().kvc_set_error_word(None))
        return
    if word.numel() != 1 or word.element_size() != 4 or not word.is_cuda:
        raise ValueError("the error word is one 4-byte element on the GPU")
    _check("kvc_set_error_word", lib().kvc_set_error_word(word.data_ptr()))


def kvc_device_errors() -> int:
    flags = ctypes.c_uint32(0)
    status = lib().kvc_device_errors(ctypes.byref(flags))
    if status not in (0, 5):
        _check("kvc_device_errors", status)
    return int(flags.value)


def kvc_validate_workspace_size(pool: PoolDesc) -> int:
    """Device bytes kvc_validate needs for this pool."""
    n = ctypes.c_size_t()
    _check("kvc_validate_workspace_size", lib().kvc_validate_workspace_size(pool, ctypes.byref(n)))
    return n.value


def kvc_validate(pool: PoolDesc, block_table: Optional[torch.Tensor] = None,
                 context_lens: Optional[torch.Tensor] = None,
                 slot_mapping: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None, stream=None) -> Tuple[int, str]:
    """Deep check of a step's tables (synchronises).  Returns (-1, "") when every check passes,
    else (smallest offending index of the first failing check, reason)."""
    num_seqs = 0
    bt_stride = 1
    if block_table is not None:
        _cuda("block_table", block_table, torch.int32)
        _cuda("context_lens", context_lens, torch.int32)
        num_seqs, bt_stride = int(block_table.shape[0]), int(block_table.shape[1])
    num_tokens = 0
    if slot_mapping is not None:
        _cuda("slot_mapping", slot_mapping, torch.int32)
        num_tokens = int(slot_mapping.numel())
    if workspace is None:
        workspace = torch.empty(kvc_validate_workspace_size(pool), dtype=torch.uint8,
                                device="cuda")
    _cuda("workspace", workspace)
    bad = ctypes.c_int64(-1)
    status = lib().kvc_validate(
        pool, _ptr(block_table), bt_stride, _ptr(context_lens), num_seqs, _ptr(slot_mapping),
        num_tokens, _ptr(workspace), workspace.numel() * workspace.element_size(),
        ctypes.byref(bad), _stream(stream))
    if status == KVC_ERR_OUT_OF_RANGE:
        return int(bad.value), lib().kvc_last_error().decode(errors="replace")
    _check("kvc_validate", status)
    return -1, ""
