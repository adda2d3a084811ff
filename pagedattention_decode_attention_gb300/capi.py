"""ctypes declarations of ``libpagedattn.so`` (the C ABI in ``include/pagedattn.h``).

Every ``pa_*`` attribute of the loaded library keeps the C name.  Loading fails
loudly if the library has not been built; there is no fallback path.
"""

from __future__ import annotations

import ctypes as C
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libpagedattn.so")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_NO_BLOCKS = 3
PA_ERR_CUDA = 4
PA_ERR_DEVICE_BOUNDS = 5
PA_ERR_DEVICE_TIMEOUT = 6
PA_ERR_NOT_FOUND = 7

STATUS_NAMES = {
    PA_OK: "PA_OK", PA_ERR_INVALID_ARG: "PA_ERR_INVALID_ARG",
    PA_ERR_UNSUPPORTED: "PA_ERR_UNSUPPORTED", PA_ERR_NO_BLOCKS: "PA_ERR_NO_BLOCKS",
    PA_ERR_CUDA: "PA_ERR_CUDA", PA_ERR_DEVICE_BOUNDS: "PA_ERR_DEVICE_BOUNDS",
    PA_ERR_DEVICE_TIMEOUT: "PA_ERR_DEVICE_TIMEOUT", PA_ERR_NOT_FOUND: "PA_ERR_NOT_FOUND",
}

PA_F32, PA_F16, PA_BF16 = 0, 1, 2
BLOCK_SIZE = 16


PA_SWAP_OUT, PA_SWAP_IN = 0, 1


class PoolStats(C.Structure):
    _fields_ = [(name, C.c_int64) for name in (
        "num_blocks", "free_blocks", "used_blocks", "pinned_blocks", "shared_blocks",
        "cow_copies", "live_seqs", "tokens", "internal_frag_slots", "host_blocks",
        "host_free_blocks", "swapped_seqs", "cached_blocks", "evictable_blocks",
        "prefix_hit_tokens", "evictions")]


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_vp, _i, _i64p, _i32p, _sz = C.c_void_p, C.c_int, C.POINTER(C.c_int64), C.POINTER(C.c_int32), C.c_size_t

SIGNATURES = {
    "pa_last_error": (C.c_char_p, []),
    "pa_version": (_i, []),
    "pa_kv_append": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "pa_paged_attention_decode_workspace_size": (_i, [_i, _i, _i, _i, _i, C.POINTER(_sz)]),
    "pa_paged_attention_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                                       C.c_float, _i, _vp, _vp, _sz, _vp]),
    "pa_paged_attention_decode_plan": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _sz, _vp]),
    "pa_paged_attention_decode_run": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                                           C.c_float, _i, _vp, _vp, _sz, _vp]),
    "pa_paged_attention_decode_append_run": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i,
                                                  _i, _i, _i, _i, C.c_float, _i, _vp, _vp, _sz,
                                                  _vp]),
    "pa_paged_attention_decode_shared_prefix_workspace_size": (_i, [_i, _i, _i, _i, _i,
                                                                    C.POINTER(_sz)]),
    "pa_paged_attention_decode_shared_prefix": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                                     _i, _i, C.c_float, _i, _vp, _vp, _sz, _vp]),
    "pa_paged_attention_decode_shared_prefix_plan": (_i, [_vp, _i, _i, _i, _i, _i, _i, C.c_float,
                                                          _i, _vp, _sz, _vp]),
    "pa_paged_attention_decode_shared_prefix_run": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i,
                                                         _i, _i, _i, C.c_float, _i, _vp, _vp, _sz,
                                                         _vp]),
    "pa_paged_attention_decode_grouped_prefix_workspace_size": (_i, [_i, _i, _i, _i, _i,
                                                                     C.POINTER(_sz)]),
    "pa_paged_attention_decode_grouped_prefix": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i,
                                                      _i, _i, _i, _i, _i, C.c_float, _i, _vp,
                                                      _vp, _sz, _vp]),
    "pa_paged_attention_decode_grouped_prefix_plan": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i,
                                                           _i, _i, C.c_float, _i, _vp, _sz, _vp]),
    "pa_paged_attention_decode_grouped_prefix_run": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i,
                                                          _i, _i, _i, _i, _i, C.c_float, _i, _vp,
                                                          _vp, _sz, _vp]),
    "pa_paged_attention_decode_shared_prefix_append_run": (_i, [_vp, _vp, _vp, _vp, _vp, _vp,
                                                                _vp, _vp, _i, _i, _i, _i, _i,
                                                                _i, _i, C.c_float, _i, _vp,
                                                                _vp, _sz, _vp]),
    "pa_paged_attention_decode_grouped_prefix_append_run": (_i, [_vp, _vp, _vp, _vp, _vp, _vp,
                                                                 _vp, _vp, _vp, _i, _i, _i, _i,
                                                                 _i, _i, _i, C.c_float, _i, _vp,
                                                                 _vp, _sz, _vp]),
    "pa_paged_attention_prefill_workspace_size": (_i, [_i, _i, _i, _i, _i, C.POINTER(_sz)]),
    "pa_paged_attention_prefill": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                        C.c_float, _i, _vp, _vp, _sz, _vp]),
    "pa_paged_attention_prefill_plan": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, C.c_float, _i,
                                             _vp, _sz, _vp]),
    "pa_paged_attention_prefill_run": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                                            _i, C.c_float, _i, _vp, _vp, _sz, _vp]),
    "pa_paged_attention_decode_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                                               C.c_float, _i, _vp, _vp]),
    "pa_block_copy": (_i, [C.POINTER(_vp), C.POINTER(_vp), _i, _vp, _i, _i, _i, _i, _i, _vp]),
    "pa_block_swap": (_i, [C.POINTER(_vp), C.POINTER(_vp), C.POINTER(_vp), C.POINTER(_vp), _i,
                           _vp, _i, _i, _i, _i, _i, _i, _i, _vp]),
    "pa_check_status": (_i, [_vp]),
    "pa_pool_create": (_i, [_i, _i, _i32p, C.POINTER(_vp)]),
    "pa_pool_destroy": (_i, [_vp]),
    "pa_pool_new_seq": (_i, [_vp, C.POINTER(_i)]),
    "pa_pool_append_slot": (_i, [_vp, _i, _i64p, _i64p, _i64p]),
    "pa_pool_append_slots": (_i, [_vp, _i32p, _i, _i64p, _i64p, _i, C.POINTER(_i), C.POINTER(_i)]),
    "pa_pool_append_tokens": (_i, [_vp, _i32p, _i32p, _i, _i64p, _i64p, _i, C.POINTER(_i),
                                   C.POINTER(_i)]),
    "pa_pool_fork": (_i, [_vp, _i, C.POINTER(_i)]),
    "pa_pool_share_prefix": (_i, [_vp, _i, _i, _i]),
    "pa_pool_pin": (_i, [_vp, _i, _i]),
    "pa_pool_unpin": (_i, [_vp, _i]),
    "pa_pool_free_seq": (_i, [_vp, _i]),
    "pa_pool_block_table": (_i, [_vp, _i, _i32p, _i, C.POINTER(_i), C.POINTER(_i)]),
    "pa_pool_refcount": (_i, [_vp, _i, C.POINTER(_i)]),
    "pa_pool_stats": (_i, [_vp, C.POINTER(PoolStats)]),
    "pa_pool_set_host_blocks": (_i, [_vp, _i, _i32p]),
    "pa_pool_swap_out": (_i, [_vp, _i, _i64p, _i, C.POINTER(_i)]),
    "pa_pool_swap_in": (_i, [_vp, _i, _i64p, _i, C.POINTER(_i)]),
    "pa_pool_is_swapped": (_i, [_vp, _i, C.POINTER(_i)]),
    "pa_pool_enable_prefix_cache": (_i, [_vp, _i]),
    "pa_pool_new_seq_with_prompt": (_i, [_vp, _i32p, _i, C.POINTER(_i), C.POINTER(_i)]),
    "pa_pool_append_token": (_i, [_vp, _i, C.c_int32, _i64p, _i64p, _i64p]),
}

_lib = None
_lock = threading.Lock()


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with "
                        "`python -m pagedattention_decode_attention_gb300.build` "
                        "(there is no CPU fallback)")
                handle = C.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def check(status: int) -> None:
    if status != PA_OK:
        raise PagedAttnError(status, lib().pa_last_error().decode(errors="replace"))
