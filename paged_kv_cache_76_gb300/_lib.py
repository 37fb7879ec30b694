"""ctypes loader for ``libpa.so`` with the prototypes of ``include/pa.h``.

There is no fallback: if the library is missing or cannot be loaded, every
call raises :class:`LibraryMissing`.  Build it with
``python -m paged_kv_cache_76_gb300.build``.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpa.so")

PA_OK = 0
PA_ERR_INVALID = -1
PA_ERR_NO_FREE_BLOCKS = -2
PA_ERR_DTYPE = -3
PA_ERR_CUDA = -4
PA_ERR_DEVICE_CHECK = -5
PA_ERR_SHARED_BLOCK = -6
PA_ERR_WORKSPACE = -7
PA_ERR_HOST_MEMORY = -8

PA_FP16 = 0
PA_BF16 = 1

PA_DEVERR_NONE = 0
PA_DEVERR_BLOCK_ID = 1
PA_DEVERR_CONTEXT_LEN = 2
PA_DEVERR_SLOT = 3
PA_DEVERR_TIMEOUT = 4
PA_DEVERR_QUERY_RANGE = 5


class LibraryMissing(RuntimeError):
    pass


class PAError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class PAHostMemoryError(PAError, MemoryError):
    """PA_ERR_HOST_MEMORY: a host allocation inside the library failed (the
    call changed nothing)."""


class AllocStats(C.Structure):
    _fields_ = [(n, C.c_int64) for n in (
        "num_blocks", "num_free", "num_used", "num_shared", "num_seqs", "cow_copies", "alloc_failures",
        "waste_slots")]


class PrefixCacheStats(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("lookup_blocks", "hit_blocks", "evictions", "cached_blocks")]


class VkvStats(C.Structure):
    _fields_ = [(n, C.c_int64) for n in (
        "page_bytes", "slot_pages", "pages_mapped", "pages_pooled", "pages_created", "map_calls", "unmap_calls",
        "bytes_reserved", "bytes_committed", "last_step_map_ns", "total_map_ns", "active_slots",
        "step_failures", "bytes_used")]


PA_VKV_DRY_RUN = 1

_P = C.c_void_p
_I = C.c_int
_I32P = C.POINTER(C.c_int32)
_F = C.c_float
_SZ = C.c_size_t

PROTOTYPES = {
    "pa_status_string": (C.c_char_p, [_I]),
    "pa_version": (_I, []),
    "pa_launch_count": (C.c_uint64, []),
    "pa_reshape_and_cache": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P]),
    "pa_copy_blocks": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "pa_swap_blocks": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
    "pa_decode_split_tokens": (_I, [_I, _I, _I]),
    "pa_decode_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "pa_decode": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P, _I, _P]),
    "pa_decode_partial": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P, _I, _P]),
    "pa_lse_merge": (_I, [_P, _SZ, _P, _I, _I, _I, _I, _I, _I, _P, _I, _P]),
    "pa_verify_split_tokens": (_I, [_I, _I, _I, _I]),
    "pa_selftest_wait_timeout": (_I, [_I, _P]),
    "pa_verify_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "pa_verify_decode": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P, _I, _P]),
    "pa_verify_decode_tc": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _I, _P]),
    "pa_decode_noalloc": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _I, _P]),
    "pa_chunked_prefill": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P, _I, _P]),
    "pa_decode_shared_prefix_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "pa_decode_shared_prefix_split_tokens": (_I, [_I, _I, _I, _I]),
    "pa_decode_shared_prefix": (_I, [_P, _P, _P, _P, _I, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P, _I,
                                     _P, _P]),
    "pa_get_device_error": (_I, [_I32P, _P]),
    "pa_alloc_create": (_I, [_I, _I, _I32P, C.POINTER(_P)]),
    "pa_alloc_destroy": (None, [_P]),
    "pa_alloc_add_seq": (_I, [_P, _I]),
    "pa_alloc_append_slots": (_I, [_P, _I, _I, _I32P]),
    "pa_alloc_share": (_I, [_P, _I, _I, _I]),
    "pa_alloc_cow": (_I, [_P, _I, _I, _I32P]),
    "pa_alloc_free_seq": (_I, [_P, _I]),
    "pa_alloc_block_table": (_I, [_P, _I, _I32P, _I, C.POINTER(_I)]),
    "pa_alloc_build_tables": (_I, [_P, C.POINTER(_I), _I, _I32P, _I, _I32P]),
    "pa_alloc_common_prefix": (_I, [_P, C.POINTER(_I), _I, C.POINTER(_I)]),
    "pa_alloc_seq_len": (_I, [_P, _I, C.POINTER(C.c_int64)]),
    "pa_alloc_num_free": (_I, [_P]),
    "pa_alloc_ref": (_I, [_P, _I]),
    "pa_alloc_free_list": (_I, [_P, _I32P, _I]),
    "pa_alloc_get_stats": (_I, [_P, C.POINTER(AllocStats)]),
    "pa_block_hash": (C.c_uint64, [C.c_uint64, _I32P, _I]),
    "pa_alloc_enable_prefix_caching": (_I, [_P]),
    "pa_alloc_add_seq_cached": (_I, [_P, _I, _I32P, _I, C.c_uint64, C.POINTER(_I)]),
    "pa_alloc_append_tokens": (_I, [_P, _I, _I32P, _I, _I32P]),
    "pa_alloc_block_hash": (_I, [_P, _I, C.POINTER(C.c_uint64), C.POINTER(_I)]),
    "pa_alloc_get_prefix_cache_stats": (_I, [_P, C.POINTER(PrefixCacheStats)]),
    "pa_vkv_granularity": (_I, [C.POINTER(_SZ)]),
    "pa_vkv_create": (_I, [_I, _I, _I, _I, _I, _I, _SZ, C.c_int64, _I, C.POINTER(_P)]),
    "pa_vkv_destroy": (None, [_P]),
    "pa_vkv_alloc_slot": (_I, [_P, C.POINTER(_I)]),
    "pa_vkv_free_slot": (_I, [_P, _I]),
    "pa_vkv_step": (_I, [_P, _I32P, _P]),
    "pa_vkv_tensor": (_I, [_P, _I, _I, C.POINTER(_P)]),
    "pa_vkv_slot_tokens": (_I, [_P, _I32P, C.POINTER(_P)]),
    "pa_vkv_slot_pages": (_I, [_P, _I]),
    "pa_vkv_get_stats": (_I, [_P, C.POINTER(VkvStats)]),
    "pa_decode_contiguous": (_I, [_P, _P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _SZ, _P, _I, _P]),
    "pa_reshape_and_cache_slots": (_I, [_P, _P, _P, _P, _I, _P, _P, _I, _I, _P, _I, _I, _I, _P]),
    "pa_vkv_decode": (_I, [_P, _I, _P, _P, _P, _I, _I, _F, _I, _P, _SZ, _P, _P]),
    "pa_vkv_reshape_and_cache": (_I, [_P, _I, _P, _P, _P, _P, _I, _P]),
    "pa_alloc_enable_swap": (_I, [_P, _I]),
    "pa_alloc_export": (_I, [_P, _P, C.c_int64, C.POINTER(C.c_int64)]),
    "pa_alloc_import": (_I, [_P, C.c_int64, C.POINTER(_P)]),
    "pa_alloc_num_free_cpu": (_I, [_P]),
    "pa_alloc_is_swapped": (_I, [_P, _I]),
    "pa_alloc_swap_out": (_I, [_P, _I, _I32P, _I, C.POINTER(_I)]),
    "pa_alloc_swap_in": (_I, [_P, _I, _I32P, _I, C.POINTER(_I)]),
}

_lock = threading.Lock()
_lib = None


def lib():
    """The loaded library (raises LibraryMissing if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise LibraryMissing(
                    f"{LIB_PATH} is not built; run `python -m paged_kv_cache_76_gb300.build` "
                    "(there is no CPU fallback)")
            try:
                h = C.CDLL(LIB_PATH)
            except OSError as e:
                raise LibraryMissing(f"cannot load {LIB_PATH}: {e}") from e
            for name, (res, args) in PROTOTYPES.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().pa_status_string(status).decode()
    except LibraryMissing:
        return str(status)


def check(status: int, what: str = ""):
    if status == PA_ERR_HOST_MEMORY:
        raise PAHostMemoryError(status, what)
    if status < 0:
        raise PAError(status, what)
    return status
