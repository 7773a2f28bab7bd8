"""Loads libpa.so and declares the C signatures of include/pa.h (ctypes).

This module only marshals arguments; every step of the compute path runs in
the library's CUDA kernels.  Loading fails loudly when the library is
missing: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

PA_OK, PA_ERR_INVALID, PA_ERR_OOM, PA_ERR_CUDA, PA_ERR_UNSUPPORTED = range(5)
PA_DECODE_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024  # include/pa.h
PA_KV_BF16, PA_KV_FP8_E4M3 = 0, 1


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class DecodeOpts(ctypes.Structure):
    _fields_ = [("partition_tokens", ctypes.c_int32), ("kernel", ctypes.c_int32)]


class PaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class PaOOM(PaError):
    pass


STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID", 2: "PA_ERR_OOM", 3: "PA_ERR_CUDA",
                4: "PA_ERR_UNSUPPORTED"}

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I32 = ctypes.c_int32
PI32 = ctypes.POINTER(ctypes.c_int32)
SIZE = ctypes.c_size_t

SIGNATURES = {
    "pa_reshape_and_cache": (I32, [P, P, P, P, CacheDesc, P, I32, P, P, P]),
    "pa_decode_workspace_size": (SIZE, [I32, I32, I32, I32, I32]),
    "pa_decode_workspace_size_ex": (SIZE, [I32, I32, I32, I32, I32, I32]),
    "pa_decode": (I32, [P, P, P, P, CacheDesc, P, I32, P, I32, I32, ctypes.c_float, P, P, P,
                        SIZE, P]),
    "pa_decode_ex": (I32, [P, P, P, P, CacheDesc, P, I32, P, I32, I32, ctypes.c_float, P, P,
                           P, SIZE, ctypes.POINTER(DecodeOpts), P]),
    "pa_decode_noalloc": (I32, [P, P, P, P, CacheDesc, P, I32, P, I32, I32, ctypes.c_float, P,
                                P, P]),
    "pa_decode_noalloc_error": (I32, [P, P]),
    "pa_write_and_decode": (I32, [P, P, P, I32, P, P, P, P, CacheDesc, P, I32, P, I32, I32,
                                  ctypes.c_float, P, P, P, SIZE, P]),
    "pa_copy_blocks": (I32, [P, P, CacheDesc, P, I32, P]),
    "pa_step_prepare": (I32, [P, I32, I32, I32, P, P, I32, I32, P, P]),
    "pa_swap_blocks": (I32, [P, P, I32, P, P, I32, CacheDesc, P, I32, P]),
    "pa_varlen_workspace_size": (ctypes.c_size_t, [I32, I32, I32, I32, I32]),
    "pa_decode_multi_workspace_size": (ctypes.c_size_t, [I32, I32, I32, I32, I32, I32]),
    "pa_decode_shared_prefix_workspace_size": (ctypes.c_size_t, [I32, I32, I32, I32, I32, I32]),
    "pa_decode_shared_prefix": (I32, [P, P, P, P, CacheDesc, P, I32, P, I32, I32, I32,
                                      ctypes.c_float, P, P, P, ctypes.c_size_t, P]),
    "pa_decode_multi": (I32, [P, P, P, P, CacheDesc, P, I32, P, I32, I32, I32, ctypes.c_float,
                              P, P, P, ctypes.c_size_t, P]),
    "pa_varlen_attention": (I32, [P, P, P, P, CacheDesc, P, I32, P, P, I32, I32, I32, ctypes.c_float, P, P,
                                  P, ctypes.c_size_t, P]),
    "pa_varlen_attention_ex": (I32, [P, P, P, P, CacheDesc, P, I32, P, P, I32, I32, I32,
                                     ctypes.c_float, P, P, I32, P, ctypes.c_size_t, P]),
    "pa_slot_mapping": (I32, [PI32, I32, I32, I32, PI32, PI32, I32, PI32]),
    "pa_pool_create": (P, [I32]),
    "pa_pool_create_ordered": (P, [I32, PI32]),
    "pa_pool_destroy": (None, [P]),
    "pa_pool_num_blocks": (I32, [P]),
    "pa_pool_num_free": (I32, [P]),
    "pa_pool_refcount": (I32, [P, I32]),
    "pa_pool_free_order": (I32, [P, PI32, I32]),
    "pa_pool_alloc": (I32, [P, I32, PI32]),
    "pa_pool_incref": (I32, [P, PI32, I32]),
    "pa_pool_free": (I32, [P, PI32, I32]),
    "pa_pool_cow": (I32, [P, I32, PI32]),
    "pa_pool_enable_prefix_cache": (I32, [P, I32]),
    "pa_pool_alloc_prefix": (I32, [P, PI32, I32, PI32, PI32]),
    "pa_pool_register_block": (I32, [P, I32, I32, PI32]),
    "pa_pool_num_cached": (I32, [P]),
    "pa_status_string": (ctypes.c_char_p, [I32]),
    "pa_last_error": (ctypes.c_char_p, []),
    "pa_version": (ctypes.c_char_p, []),
}


def lib():
    """The loaded library (built on first use if the CUDA toolkit is here)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                from . import build as _build
                _build.build()
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libpa.so not found at {LIB_PATH}; run build()")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def check(status: int) -> None:
    if status != PA_OK:
        msg = lib().pa_last_error().decode()
        if status == PA_ERR_OOM:
            raise PaOOM(status, msg)
        raise PaError(status, msg)
