"""ctypes loader and signatures of libpagedattn.so.

The library is the only compute path: if it is missing or cannot be loaded the
import fails loudly; there is no fallback."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedattn.so")

c_int = ctypes.c_int
c_i32p = ctypes.c_void_p
c_void_p = ctypes.c_void_p
c_size_t = ctypes.c_size_t
c_int64 = ctypes.c_int64
c_float = ctypes.c_float

# name -> (restype, argtypes); mirrors include/pagedattn.h
SIGNATURES = {
    "pa_status_string": (ctypes.c_char_p, [c_int]),
    "pa_version": (c_int, []),
    "pa_decode_workspace_bytes": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "pa_decode_workspace_bytes_for": (c_size_t, [c_int, c_int, c_int, c_int, c_int, c_int,
                                                 c_int, c_int, c_int, c_int]),
    "pa_decode": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                          c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                          c_float, c_int, c_int, c_void_p, c_size_t, c_void_p, c_void_p]),
    "pa_decode_append": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int,
                                 c_int, c_int, c_float, c_int, c_int, c_void_p, c_size_t,
                                 c_void_p, c_void_p]),
    "pa_decode_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                  c_float, c_int, c_int, c_void_p, c_void_p]),
    "pa_reshape_and_cache": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                     c_int64, c_int, c_int, c_int, c_int, c_int, c_void_p,
                                     c_void_p]),
    "pa_copy_blocks": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                               c_int, c_void_p, c_void_p]),
    "pa_set_decode_path": (c_int, [c_int]),
    "pa_decode_kernel_for": (c_int, [c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                     c_int, c_int]),
    "pa_set_prefill_path": (c_int, [c_int]),
    "pa_prefill": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                           c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                           ctypes.c_float, c_int, c_void_p, c_void_p]),
    "pa_copy_blocks_multi": (c_int, [c_void_p, c_int, c_void_p, c_int, c_int64, c_int, c_void_p,
                                     c_void_p]),
    "pa_swap_blocks": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int64, c_int, c_int,
                               c_void_p, c_void_p]),
    "pa_append_tokens": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_void_p, c_int, c_int64, c_int, c_int, c_int, c_int, c_int,
                                 c_int, c_void_p, c_void_p]),
    "pa_stream_read": (c_int, [c_void_p, c_size_t, c_void_p, c_void_p]),
    "pa_decode_slots": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                c_void_p, c_void_p]),
    "pa_bm_create": (c_int, [c_int, c_int, c_void_p, ctypes.POINTER(c_void_p)]),
    "pa_bm_destroy": (None, [c_void_p]),
    "pa_sim_run": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p]),
    "pa_bm_num_free": (c_int, [c_void_p]),
    "pa_bm_num_evictable": (c_int, [c_void_p]),
    "pa_bm_seq_create_cached": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(c_int),
                                        ctypes.POINTER(c_int)]),
    "pa_bm_refcount": (c_int, [c_void_p, c_int]),
    "pa_bm_allocate": (c_int, [c_void_p, c_int, c_void_p]),
    "pa_bm_free": (c_int, [c_void_p, c_void_p, c_int]),
    "pa_bm_fork": (c_int, [c_void_p, c_void_p, c_int]),
    "pa_bm_seq_create": (c_int, [c_void_p, c_int, ctypes.POINTER(c_int)]),
    "pa_bm_seq_fork": (c_int, [c_void_p, c_int, ctypes.POINTER(c_int)]),
    "pa_bm_seq_release": (c_int, [c_void_p, c_int]),
    "pa_bm_seq_append": (c_int, [c_void_p, c_int, ctypes.POINTER(ctypes.c_int32),
                                 ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
    "pa_bm_seq_len": (c_int, [c_void_p, c_int]),
    "pa_bm_seq_num_blocks": (c_int, [c_void_p, c_int]),
    "pa_bm_export": (c_int, [c_void_p, c_void_p, c_int, c_int, ctypes.c_int32, c_void_p,
                             c_void_p]),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load libpagedattn.so (build it first with paged_kv_cache_301_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"libpagedattn.so not found at {LIB_PATH}; build it with "
                "`python -m paged_kv_cache_301_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib
