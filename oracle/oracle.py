"""ctypes marshalling for the fp64 C oracle (``kvc_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the benchmark's
CPU-baseline leg, never by the product path.  This module does argument marshalling
only; every step of the arithmetic is in ``kvc_oracle.c``.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvc_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkvc_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, no fast-math) and return the library path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.kvo_slot_of_position.restype = i64
            lib.kvo_slot_of_position.argtypes = [p, i64, i64, i64, i64]
            lib.kvo_slot_mapping.restype = None
            lib.kvo_slot_mapping.argtypes = [p, i64, p, p, i64, i64, p]
            lib.kvo_store.restype = None
            lib.kvo_store.argtypes = [p, p, i64, i64, p, p, p, i64]
            lib.kvo_quantize_vector.restype = None
            lib.kvo_quantize_vector.argtypes = [p, i64, p, p]
            lib.kvo_store_int8.restype = None
            lib.kvo_store_int8.argtypes = [p, p, p, p, i64, i64, i64, p, p, p, i64]
            lib.kvo_attention_int8.restype = None
            lib.kvo_attention_int8.argtypes = [p, p, p, p, p, i64, i64, i64, p, i64, p, p,
                                               i64, i64, ctypes.c_double, p, p, p, p, i64]
            lib.kvo_copy_pages.restype = None
            lib.kvo_copy_pages.argtypes = [p, p, i64, p, p, i64, p, p]
            lib.kvo_attention.restype = None
            lib.kvo_attention.argtypes = [p, p, p, i64, i64, i64, p, i64, p, p, i64, i64,
                                          ctypes.c_double, p, p, p, p, i64]
            lib.kvo_merge.restype = None
            lib.kvo_merge.argtypes = [p, p, i64, i64, i64, p, p]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def slot_of_position(block_table, seq: int, position: int, page_size: int) -> int:
    bt = _c(np.atleast_2d(block_table), np.int32)
    return int(_load().kvo_slot_of_position(_ptr(bt), bt.shape[1], seq, position, page_size))


def slot_mapping(block_table, context_lens, q_indptr, page_size: int) -> np.ndarray:
    bt = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    ind = _c(q_indptr, np.int32)
    out = np.empty(int(ind[-1]), dtype=np.int64)
    _load().kvo_slot_mapping(_ptr(bt), bt.shape[1], _ptr(ctx), _ptr(ind), ctx.shape[0],
                             page_size, _ptr(out))
    return out


def hnd_to_nhd(pool):
    """A pool in the HND layout [pages, Hkv, P, D] (TileInfer.jl "KV cache", "Pages and block
    tables": its Julia (head_dim, page_size, kv_heads, num_pages) array, column-major) as the
    same values in the NHD layout [pages, P, Hkv, D].  Layout only: no value changes."""
    return np.ascontiguousarray(pool.transpose(0, 2, 1, 3))


def nhd_to_hnd(pool):
    return np.ascontiguousarray(pool.transpose(0, 2, 1, 3))


def store(k_pool, v_pool, k_new, v_new, slots, layout: str = "nhd") -> None:
    """In place on k_pool / v_pool (uint16 bf16 bit patterns, [pages, P, Hkv, D], or
    [pages, Hkv, P, D] with layout "hnd")."""
    assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous
    assert v_pool.dtype == np.uint16 and v_pool.flags.c_contiguous
    if layout == "hnd":
        kp, vp = hnd_to_nhd(k_pool), hnd_to_nhd(v_pool)
        store(kp, vp, k_new, v_new, slots)
        k_pool[...] = nhd_to_hnd(kp)
        v_pool[...] = nhd_to_hnd(vp)
        return
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    sl = _c(slots, np.int64)
    hkv, d = k_pool.shape[2], k_pool.shape[3]
    _load().kvo_store(_ptr(k_pool), _ptr(v_pool), hkv, d, _ptr(kn), _ptr(vn), _ptr(sl),
                      sl.shape[0])


def quantize_vector(x_bits):
    """INT8 codes and fp32 scale of one bf16 vector (uint16 bits): x ~ scale * code."""
    x = _c(x_bits, np.uint16)
    codes = np.empty(x.shape[0], dtype=np.int8)
    scale = np.zeros(1, dtype=np.float32)
    _load().kvo_quantize_vector(_ptr(x), x.shape[0], _ptr(codes), _ptr(scale))
    return codes, float(scale[0])


def store_int8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, slots) -> None:
    """In place: quantise every new token's K/V vectors into INT8 pages at their slots.
    codes int8 [pages, P, Hkv, D]; scales float32 [pages, Hkv, P]."""
    for a, t in ((k_codes, np.int8), (v_codes, np.int8), (k_scales, np.float32),
                 (v_scales, np.float32)):
        assert a.dtype == t and a.flags.c_contiguous
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    sl = _c(slots, np.int64)
    P, hkv, d = k_codes.shape[1], k_codes.shape[2], k_codes.shape[3]
    _load().kvo_store_int8(_ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), P,
                           hkv, d, _ptr(kn), _ptr(vn), _ptr(sl), sl.shape[0])


def attention_int8(q, k_codes, v_codes, k_scales, v_scales, block_table, context_lens,
                   q_indptr, scale=None, key_lo=None, key_hi=None, num_threads: int = 1):
    """fp64 paged attention over INT8 pages (x = scale * code); returns (out, lse)."""
    q = _c(q, np.uint16)
    kc = _c(k_codes, np.int8)
    vc = _c(v_codes, np.int8)
    ks = _c(k_scales, np.float32)
    vs = _c(v_scales, np.float32)
    bt = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    ind = _c(q_indptr, np.int32)
    lo = None if key_lo is None else _c(key_lo, np.int32)
    hi = None if key_hi is None else _c(key_hi, np.int32)
    t, hq, d = q.shape
    page_size, hkv = kc.shape[1], kc.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.empty((t, hq, d), dtype=np.float64)
    lse = np.empty((t, hq), dtype=np.float64)
    _load().kvo_attention_int8(_ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), page_size, hkv,
                               d, _ptr(bt), bt.shape[1], _ptr(ctx), _ptr(ind), ctx.shape[0],
                               hq, float(scale), _ptr(lo), _ptr(hi), _ptr(out), _ptr(lse),
                               int(num_threads))
    return out, lse


def copy_pages(k_pool, v_pool, src_pages, dst_pages) -> None:
    """In place: page dst[i] of both pools receives page src[i] (uint16 bit patterns)."""
    assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous
    assert v_pool.dtype == np.uint16 and v_pool.flags.c_contiguous
    src = _c(src_pages, np.int64)
    dst = _c(dst_pages, np.int64)
    assert src.shape == dst.shape
    page_elems = int(np.prod(k_pool.shape[1:]))
    sk = np.empty(max(src.shape[0], 1) * page_elems, dtype=np.uint16)
    sv = np.empty_like(sk)
    _load().kvo_copy_pages(_ptr(k_pool), _ptr(v_pool), page_elems, _ptr(src), _ptr(dst),
                           src.shape[0], _ptr(sk), _ptr(sv))


def attention(q, k_pool, v_pool, block_table, context_lens, q_indptr, scale=None,
              key_lo=None, key_hi=None, num_threads: int = 1, layout: str = "nhd"):
    """fp64 paged attention; returns (out [T, Hq, D] float64, lse [T, Hq] float64).  Pools
    are NHD [pages, P, Hkv, D], or HND [pages, Hkv, P, D] with layout "hnd"."""
    if layout == "hnd":
        k_pool, v_pool = hnd_to_nhd(k_pool), hnd_to_nhd(v_pool)
    q = _c(q, np.uint16)
    kp = _c(k_pool, np.uint16)
    vp = _c(v_pool, np.uint16)
    bt = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    ind = _c(q_indptr, np.int32)
    lo = None if key_lo is None else _c(key_lo, np.int32)
    hi = None if key_hi is None else _c(key_hi, np.int32)
    t, hq, d = q.shape
    page_size, hkv = kp.shape[1], kp.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.empty((t, hq, d), dtype=np.float64)
    lse = np.empty((t, hq), dtype=np.float64)
    _load().kvo_attention(_ptr(q), _ptr(kp), _ptr(vp), page_size, hkv, d, _ptr(bt),
                          bt.shape[1], _ptr(ctx), _ptr(ind), ctx.shape[0], hq, float(scale),
                          _ptr(lo), _ptr(hi), _ptr(out), _ptr(lse), int(num_threads))
    return out, lse


def merge(partial_o, partial_lse):
    """partial_o [rows, n_split, D], partial_lse [rows, n_split] -> (out, lse), fp64."""
    po = _c(partial_o, np.float64)
    pl = _c(partial_lse, np.float64)
    rows, n_split, d = po.shape
    out = np.empty((rows, d), dtype=np.float64)
    lse = np.empty(rows, dtype=np.float64)
    _load().kvo_merge(_ptr(po), _ptr(pl), rows, n_split, d, _ptr(out), _ptr(lse))
    return out, lse
