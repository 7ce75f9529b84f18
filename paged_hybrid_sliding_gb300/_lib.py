"""ctypes declarations of libphs.so (the C ABI in include/phs.h).

The library is loaded on first use.  There is no fallback: if the shared
object is missing or fails to load, every call raises."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

c_i32, c_i64, c_f32, c_size, c_vp = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                     ctypes.c_size_t, ctypes.c_void_p)
P_i32 = ctypes.POINTER(ctypes.c_int32)
P_i64 = ctypes.POINTER(ctypes.c_int64)


class PagedPoolC(ctypes.Structure):
    _fields_ = [("k", c_vp), ("v", c_vp), ("num_pages", c_i64), ("page_size", c_i32),
                ("num_kv_heads", c_i32), ("head_dim", c_i32)]


class RingPoolC(ctypes.Structure):
    _fields_ = [("k", c_vp), ("v", c_vp), ("num_rings", c_i64), ("window", c_i32),
                ("num_kv_heads", c_i32), ("head_dim", c_i32)]


class Int8PoolC(ctypes.Structure):
    _fields_ = [("k", c_vp), ("v", c_vp), ("k_scale", c_vp), ("v_scale", c_vp),
                ("num_qpages", c_i64), ("num_kv_heads", c_i32), ("head_dim", c_i32)]


class LayerC(ctypes.Structure):
    _fields_ = [("is_full", c_i32), ("q", c_vp), ("k_new", c_vp), ("v_new", c_vp), ("out", c_vp),
                ("paged", PagedPoolC), ("ring", RingPoolC)]


_P = ctypes.POINTER
_SIGS = {
    "phs_version": (c_i32, []),
    "phs_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "phs_kv_append_paged": (ctypes.c_int, [_P(PagedPoolC), c_vp, c_vp, c_vp, c_i32, c_vp, c_i32,
                                           c_vp, c_vp, c_vp]),
    "phs_kv_append_ring": (ctypes.c_int, [_P(RingPoolC), c_vp, c_vp, c_vp, c_vp, c_i32, c_vp,
                                          c_vp]),
    "phs_kv_quant_int8_block32": (ctypes.c_int, [_P(PagedPoolC), c_vp, c_i32, _P(Int8PoolC), c_vp,
                                                 c_i32, c_vp, c_vp, c_i32, c_i32, c_vp, c_vp]),
    "phs_decode_workspace_bytes": (c_size, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32]),
    "phs_decode_tokens_per_split": (c_i32, [c_i32, c_i32, c_i32, c_i32]),
    "phs_attn_decode_full_paged": (ctypes.c_int, [c_vp, c_i32, _P(PagedPoolC), c_vp, c_i32, c_vp,
                                                  c_i32, _P(Int8PoolC), c_vp, c_i32, c_vp, c_i32,
                                                  c_f32, c_i32, c_vp, c_i32, c_vp, c_size, c_vp,
                                                  c_vp, c_vp, c_vp, c_vp]),
    "phs_attn_decode_full_paged_split": (ctypes.c_int, [c_vp, c_i32, _P(PagedPoolC), c_vp, c_i32,
                                                        c_vp, c_i32, _P(Int8PoolC), c_vp, c_i32,
                                                        c_vp, c_i32, c_f32, c_i32, c_vp, c_i32,
                                                        c_vp, c_size, c_vp, c_vp, c_vp, c_vp,
                                                        c_vp]),
    "phs_attn_decode_full_paged_noalloc": (ctypes.c_int, [c_vp, c_i32, _P(PagedPoolC), c_vp,
                                                          c_i32, c_vp, c_i32, _P(Int8PoolC), c_vp,
                                                          c_i32, c_vp, c_i32, c_f32, c_i32, c_vp,
                                                          c_i32, c_vp, c_vp]),
    "phs_shared_prefix_workspace_bytes": (c_size, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32]),
    "phs_attn_decode_shared_prefix": (ctypes.c_int, [c_vp, c_i32, _P(PagedPoolC), c_vp, c_i32, c_vp,
                                                     c_i32, c_i32, c_i32, c_f32, c_vp, c_i32, c_vp,
                                                     c_size, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "phs_attn_merge_splits": (ctypes.c_int, [c_i32, c_i32, c_i32, c_i32, c_vp, c_i32, c_vp, c_i32,
                                             c_i32, c_vp, c_i32, c_vp, c_size, c_vp]),
    "phs_attn_decode_swa_ring": (ctypes.c_int, [c_vp, c_i32, _P(RingPoolC), c_vp, c_vp, c_vp,
                                                c_i32, c_f32, c_vp, c_i32, c_vp, c_vp]),
    "phs_attn_decode_hybrid_stack": (ctypes.c_int, [_P(LayerC), c_i32, c_i32, c_i32, c_vp, c_i32,
                                                    c_vp, c_vp, c_i32, c_vp, c_vp, c_f32, c_i32,
                                                    c_i32, c_vp, c_size, c_vp, c_vp]),
    "phs_hybrid_stack_workspace_bytes": (c_size, [c_i32, c_i32, c_i32, c_i32, c_i32]),
    "phs_attn_decode_hybrid_stack_fused": (ctypes.c_int, [_P(LayerC), c_i32, c_i32, c_i32, c_vp,
                                                          c_i32, c_vp, c_vp, c_i32, c_vp, c_vp,
                                                          c_f32, c_i32, c_vp, c_size, c_vp, c_vp]),
    "phs_hybrid_stack_fused_workspace_bytes": (c_size, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32]),
    "phs_hybrid_kv_tokens": (ctypes.c_int, [c_vp, c_i32, c_vp, c_i32, c_i32, P_i64, P_i64]),
    "phs_copy_d2d": (ctypes.c_int, [c_vp, c_vp, c_size, c_vp]),
    "phs_read_checksum": (ctypes.c_int, [c_vp, c_size, c_vp, c_vp]),
    "phs_copy_pages": (ctypes.c_int, [_P(PagedPoolC), c_vp, c_vp, c_i32, c_vp, c_vp]),
    "phs_page_allocator_create": (c_vp, [c_i64]),
    "phs_page_allocator_destroy": (None, [c_vp]),
    "phs_page_alloc": (ctypes.c_int, [c_vp, c_i32, c_vp]),
    "phs_page_incref": (ctypes.c_int, [c_vp, c_vp, c_i32]),
    "phs_page_decref": (ctypes.c_int, [c_vp, c_vp, c_i32]),
    "phs_page_free_count": (c_i64, [c_vp]),
    "phs_page_refcounts": (ctypes.c_int, [c_vp, c_vp]),
    "phs_page_cow": (ctypes.c_int, [c_vp, c_i32, P_i32]),
    "phs_radix_create": (c_vp, [c_vp, c_vp, c_i32]),
    "phs_radix_destroy": (None, [c_vp]),
    "phs_radix_match": (ctypes.c_int, [c_vp, c_vp, c_i64, c_vp, c_i32, P_i32]),
    "phs_radix_match_window_safe": (ctypes.c_int, [c_vp, c_vp, c_i64, c_i32, c_vp, c_i32, P_i32,
                                                   c_vp, c_i32, P_i32]),
    "phs_radix_insert": (ctypes.c_int, [c_vp, c_vp, c_i64, c_vp, c_vp]),
    "phs_radix_evict": (ctypes.c_int, [c_vp, c_i64, P_i64]),
    "phs_radix_cached_pages": (c_i64, [c_vp]),
    "phs_window_safe_len": (c_i64, [c_vp, c_i64, c_i32, c_i32]),
    "phs_swa_ring_save": (ctypes.c_int, [_P(RingPoolC), _P(PagedPoolC), c_i32, c_vp, c_vp, c_vp,
                                         c_vp, c_vp, c_i32, c_vp, c_vp]),
    "phs_swa_ring_seed": (ctypes.c_int, [_P(RingPoolC), _P(PagedPoolC), c_i32, c_vp, c_vp, c_vp,
                                         c_vp, c_i32, c_i32, c_vp, c_vp]),
}

# every symbol include/phs.h declares
EXPORTED = tuple(_SIGS)


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libphs.so (building it first if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(f"libphs.so not built ({path})")
                _build.build()
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
