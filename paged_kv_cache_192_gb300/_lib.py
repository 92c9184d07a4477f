"""ctypes loader of libpa_gb300.so with the C ABI declared in include/pa.h.

There is no fallback: if the shared library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa_gb300.so")

PA_OK, PA_ERR_INVALID, PA_ERR_OOM, PA_ERR_CUDA, PA_ERR_UNSUPPORTED, PA_ERR_DEVICE = range(6)
PA_BF16, PA_F32 = 0, 1
PA_DEVERR_BAD_BLOCK, PA_DEVERR_TIMEOUT = 1, 2
PA_DECODE_PERSISTENT, PA_DECODE_GRID = 1, 2
PA_DECODE_TILE_CUDA_CORE, PA_DECODE_TILE_TENSOR_CORE = 1, 2
PA_PREFILL_PERSISTENT_GRID, PA_PREFILL_ITEM_GRID, PA_PREFILL_SIMPLE = 1, 2, 3

_c_int, _c_i64, _c_sz, _c_vp, _c_f = (ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                      ctypes.c_void_p, ctypes.c_float)
_p_i64 = ctypes.POINTER(ctypes.c_int64)
_p_i32 = ctypes.POINTER(ctypes.c_int32)

# name -> (restype, argtypes); mirrors include/pa.h one to one
SIGNATURES = {
    "pa_last_error_string": (ctypes.c_char_p, []),
    "pa_version": (_c_int, []),
    "pa_set_validate": (_c_int, [_c_int]),
    "pa_device_error": (_c_int, [ctypes.POINTER(_c_int), _c_int, _c_vp]),
    "pa_check_wait_timeout": (_c_int, [_c_vp]),
    "pa_reshape_and_cache": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_int,
                                      _c_int, _c_int, _c_int, _c_vp]),
    "pa_copy_blocks": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_int, _c_int, _c_int,
                                _c_int, _c_vp]),
    "pa_swap_blocks": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64,
                                _c_int, _c_int, _c_int, _c_int, _c_vp]),
    "pa_decode_workspace_size": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                          ctypes.POINTER(_c_sz)]),
    "pa_decode_kernel_for": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int,
                                      ctypes.POINTER(_c_int)]),
    "pa_decode_tile_for": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_i64, _c_int,
                                    ctypes.POINTER(_c_int)]),
    "pa_decode": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_vp, _c_int, _c_int,
                           _c_int, _c_int, _c_int, _c_i64, _c_f, _c_int, _c_vp, _c_sz, _c_int,
                           _c_vp]),
    "pa_decode_contiguous_workspace_size": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int,
                                                     ctypes.POINTER(_c_sz)]),
    "pa_decode_contiguous": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int,
                                      _c_int, _c_int, _c_f, _c_int, _c_vp, _c_sz, _c_int, _c_vp]),
    "pa_decode_shared_workspace_size": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                                 _c_int, ctypes.POINTER(_c_sz)]),
    "pa_decode_shared": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_vp, _c_int,
                                  _c_int, _c_int, _c_int, _c_int, _c_i64, _c_f, _c_int, _c_vp,
                                  _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_int, _c_vp, _c_sz,
                                  _c_int, _c_vp]),
    "pa_decode_shared_forks_workspace_size": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int,
                                                       _c_int, _c_int, ctypes.POINTER(_c_sz)]),
    "pa_decode_shared_forks": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_vp,
                                        _c_int, _c_int, _c_int, _c_int, _c_int, _c_i64, _c_f,
                                        _c_int, _c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int,
                                        _c_int, _c_vp, _c_vp, _c_vp, _c_sz, _c_int, _c_vp]),
    "pa_decode_noalloc_capacity": (_c_sz, []),
    "pa_decode_noalloc": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_vp, _c_int, _c_int,
                                   _c_int, _c_int, _c_int, _c_i64, _c_f, _c_int, _c_int, _c_vp]),
    "pa_prefill_chunk": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_vp, _c_vp, _c_int,
                                  _c_int, _c_int, _c_int, _c_int, _c_int, _c_i64, _c_f, _c_int,
                                  _c_vp]),
    "pa_prefill_kernel_for": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_i64,
                                       _c_int, ctypes.POINTER(_c_int)]),
    "pa_bm_create": (_c_int, [_c_i64, _c_int, ctypes.c_uint64, ctypes.POINTER(_c_vp)]),
    "pa_bm_destroy": (None, [_c_vp]),
    "pa_bm_add_seq": (_c_int, [_c_vp, _c_i64, _c_i64, _p_i64]),
    "pa_bm_fork": (_c_int, [_c_vp, _c_i64, _c_i64]),
    "pa_bm_append": (_c_int, [_c_vp, _c_i64, _p_i64, _p_i64, _p_i64]),
    "pa_bm_append_n": (_c_int, [_c_vp, _c_i64, _c_i64, _p_i64, _p_i64, _p_i64]),
    "pa_bm_free_seq": (_c_int, [_c_vp, _c_i64]),
    "pa_bm_block_table": (_c_int, [_c_vp, _p_i64, _c_int, _p_i32, _c_int]),
    "pa_bm_seq_len": (_c_int, [_c_vp, _c_i64, _p_i64]),
    "pa_bm_seq_blocks": (_c_int, [_c_vp, _c_i64, _p_i32, _c_i64, _p_i64]),
    "pa_bm_refcount": (_c_int, [_c_vp, _c_i64, ctypes.POINTER(_c_int)]),
    "pa_bm_num_free": (_c_i64, [_c_vp]),
    "pa_bm_inject_alloc_failure": (None, [_c_i64]),
}


class PAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[pa error {code}] {msg}")
        self.code = code


class OutOfBlocks(PAError):
    pass


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with paged_kv_cache_192_gb300.build.build() "
                "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def check(rc: int):
    if rc != PA_OK:
        msg = lib().pa_last_error_string().decode(errors="replace")
        if rc == PA_ERR_OOM:
            raise OutOfBlocks(rc, msg)
        raise PAError(rc, msg)
