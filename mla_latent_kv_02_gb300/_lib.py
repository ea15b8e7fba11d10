"""ctypes loader for the in-tree ``libmla.so`` (the C ABI of include/mla.h).

There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

from . import _build

_lock = threading.Lock()
_lib = None


class mla_config(C.Structure):
    _fields_ = [("num_heads", C.c_int32), ("head_dim_c", C.c_int32), ("latent_dim", C.c_int32),
                ("rope_dim", C.c_int32), ("page_size", C.c_int32), ("scale", C.c_float)]


class mla_plan_info(C.Structure):
    _fields_ = [("magic", C.c_uint32), ("T", C.c_int32), ("B", C.c_int32), ("num_clusters", C.c_int32),
                ("num_segments", C.c_int32), ("num_partials", C.c_int32), ("num_split_rows", C.c_int32),
                ("max_pages_needed", C.c_int32), ("total_tiles", C.c_int64), ("plan_bytes", C.c_size_t)]


P = C.c_void_p
I32 = C.c_int32
I64 = C.c_int64
PI32 = C.POINTER(C.c_int32)
PI64 = C.POINTER(C.c_int64)
SZ = C.c_size_t

SIGNATURES = {
    "mla_last_error": (C.c_char_p, []),
    "mla_status_string": (C.c_char_p, [C.c_int]),
    "mla_version": (I32, []),
    "mla_config_default": (mla_config, []),
    "mla_config_validate": (C.c_int, [C.POINTER(mla_config)]),
    "mla_kv_bytes": (C.c_int, [I64, I64, I64, I64, I64, I64, C.POINTER(C.c_uint64)]),
    "mla_pool_create": (C.c_int, [I32, C.POINTER(P)]),
    "mla_pool_alloc": (C.c_int, [P, I32, PI32]),
    "mla_pool_free": (C.c_int, [P, PI32, I32]),
    "mla_pool_available": (C.c_int, [P, PI32]),
    "mla_pool_destroy": (None, [P]),
    "mla_slot_mapping": (C.c_int, [PI32, I32, I32, PI32, PI32, I32, PI64]),
    "mla_cache_init": (C.c_int, [P, I64, P]),
    "mla_kv_append": (C.c_int, [P, P, P, I32, P, I64, P, P]),
    "mla_gather_paged": (C.c_int, [P, I64, P, I32, I32, I32, P, P, P]),
    "mla_kv_append_fp8": (C.c_int, [P, P, P, I32, P, P, I64, P, P]),
    "mla_gather_paged_fp8": (C.c_int, [P, P, I64, P, I32, I32, I32, P, P, P]),
    "mla_kv_append_nvfp4": (C.c_int, [P, P, P, I32, C.c_float, P, I64, P, P]),
    "mla_gather_paged_nvfp4": (C.c_int, [P, C.c_float, I64, P, I32, I32, I32, P, P, P]),
    "mla_gather_paged_nvfp4_batch": (C.c_int, [P, C.c_float, I64, P, I32, I32, P, P, I32, I64, P, P, P]),
    "mla_prefill_threshold": (I32, []),
    "mla_branch_for": (I32, [I32]),
    "mla_expand_kv": (C.c_int, [P, I32, P, P, P, P, P, P]),
    "mla_prefill_attention": (C.c_int, [P, P, I32, P, P, P, I32, C.c_float, P, P, P]),
    "mla_prefill_workspace_size": (C.c_int, [I32, C.POINTER(SZ)]),
    "mla_prefill_batch_workspace_size": (C.c_int, [PI32, I32, C.POINTER(SZ)]),
    "mla_prefill_decompress_batch": (C.c_int, [P, P, PI32, PI32, PI32, PI32, I32, P, I64, P, I32, I32, P, P, C.c_float,
                                               P, SZ, P, P, P]),
    "mla_prefill_decompress": (C.c_int, [P, P, I32, P, I64, P, I32, I32, I32, P, P, C.c_float, P, SZ, P, P, P]),
    "mla_rope_table": (C.c_int, [I32, C.c_float, P, P]),
    "mla_kv_append_rope": (C.c_int, [P, P, P, P, I32, P, I32, P, I64, P, P]),
    "mla_rope_q": (C.c_int, [P, P, P, I32, P, I32, P, P]),
    "mla_absorb_q": (C.c_int, [P, P, P, I32, P, P]),
    "mla_up_v": (C.c_int, [P, P, P, I32, P, P]),
    "mla_decode_max_clusters": (C.c_int, [PI32]),
    "mla_decode_plan_bytes": (C.c_int, [I32, I32, C.POINTER(SZ)]),
    "mla_decode_workspace_size": (C.c_int, [I32, C.POINTER(SZ)]),
    "mla_decode_plan_host": (C.c_int, [PI32, PI32, I32, I32, P, SZ, C.POINTER(mla_plan_info)]),
    "mla_decode_plan": (C.c_int, [PI32, PI32, I32, I32, P, SZ, C.POINTER(mla_plan_info), P]),
    "mla_decode_paged": (C.c_int, [P, P, P, I64, P, I32, P, C.POINTER(mla_plan_info), C.c_float, P, SZ, P, P, P, P]),
    "mla_decode_paged_fp8": (C.c_int, [P, P, P, P, I64, P, I32, P, C.POINTER(mla_plan_info), C.c_float, P, SZ, P, P,
                                       P, P]),
    "mla_check": (C.c_int, [P, P, PI32]),
    "mla_debug_set_decode_wait_limit": (C.c_int, [C.c_uint64]),
    "mla_decode_paged_noalloc": (C.c_int, [P, P, P, I64, P, I32, PI32, PI32, I32, C.c_float, P, P, P, P]),
    "mla_debug_noalloc_last_plan": (C.c_int, [C.POINTER(mla_plan_info)]),
}


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError(
                    f"{_build.LIB} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
            h = C.CDLL(_build.LIB)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(h, name)
                f.restype = res
                f.argtypes = args
            _lib = h
    return _lib


def path() -> str:
    return _build.LIB
