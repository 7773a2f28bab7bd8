"""ctypes wrapper of the C oracle (``pa_oracle.c``) -- TEST INFRASTRUCTURE.

The C file holds all the arithmetic; this module only builds it with gcc,
marshals numpy arrays, and checks return codes.  Definitions followed:

* cache write  -- "Paged KV cache" (ai-infra-handbooks), ``PagedKVCache.write``:
  the pool viewed flat as [num_blocks*block_size, H_kv, d] is indexed by the
  slot.
* block copy   -- "4.6 PagedAttention & KV-Cache Memory Management"
  (llm-stack-book), section "Copy-on-write for shared prefixes".
* decode       -- "Paged KV cache", ``PagedKVCache.gather`` + ``paged_attention``
  restricted to one query token per sequence: gather through the block table,
  then softmax(scale * q K^T) V with the GQA map h -> h // G.
* varlen       -- ``orc_varlen``, wrapped by ``oracle/varlen.py``: "Paged KV
  cache", section "Paged attention" (several new tokens per request, each
  seeing the context up to its own position).
* E4M3         -- the OCP 8-bit floating point specification (E4M3, bias 7,
  max 448, NaN S.1111.111), round-to-nearest-even, saturating.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

KV_BF16 = 0
KV_FP8_E4M3 = 1


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into liboracle.so with plain gcc (no fast-math,
    no FMA contraction, so x86 and Arm give the same bits)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(
            _LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f32, f64 = (ctypes.c_int32, ctypes.c_int64,
                                  ctypes.c_float, ctypes.c_double)
            lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_double.restype = f64
            lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_to_double.restype = f64
            lib.orc_e4m3_encode.argtypes = [f32]
            lib.orc_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_e4m3_encode_array.argtypes = [P, P, i64]
            lib.orc_e4m3_encode_array.restype = None
            lib.orc_e4m3_decode_array.argtypes = [P, P, i64]
            lib.orc_e4m3_decode_array.restype = None
            lib.orc_reshape_and_cache.argtypes = [P, P, i32, i32, i32, P, P,
                                                  i32, i32, i32, P, f32, f32]
            lib.orc_reshape_and_cache.restype = ctypes.c_int
            lib.orc_copy_blocks.argtypes = [P, P, i32, i64, P, i32]
            lib.orc_copy_blocks.restype = ctypes.c_int
            lib.orc_decode.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P,
                                       i32, P, i32, i32, f64, f64, f64, P, i32,
                                       i32]
            lib.orc_decode.restype = ctypes.c_int
            lib.orc_varlen.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P,
                                       i32, P, P, i32, i32, f64, f64, f64, i32]
            lib.orc_varlen.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _kv_dtype_of(cache: np.ndarray) -> int:
    if cache.dtype == np.uint16:
        return KV_BF16
    if cache.dtype == np.uint8:
        return KV_FP8_E4M3
    raise TypeError(f"cache must hold bf16 (uint16) or e4m3 (uint8) bits, got {cache.dtype}")


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    u = bits.astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """E4M3 codes (uint8) of float32 values: RNE, saturating to +-448."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().orc_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """float64 values of E4M3 codes (uint8)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    _load().orc_e4m3_decode_array(_ptr(codes), _ptr(out), codes.size)
    return out


def reshape_and_cache(key: np.ndarray, value: np.ndarray, k_cache: np.ndarray,
                      v_cache: np.ndarray, slot_mapping: np.ndarray,
                      k_scale: float = 1.0, v_scale: float = 1.0) -> None:
    """Write key/value [N, H_kv, d] (bf16 bits) into the caches in place.

    Caches are [num_blocks, block_size, H_kv, d]: uint16 for bf16, uint8 for
    E4M3.  ``slot_mapping`` [N] int32; a negative slot skips that token."""
    key = np.ascontiguousarray(key, dtype=np.uint16)
    value = np.ascontiguousarray(value, dtype=np.uint16)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    nb, B, hkv, d = k_cache.shape
    assert v_cache.shape == k_cache.shape and v_cache.dtype == k_cache.dtype
    assert key.shape == value.shape == (slots.shape[0], hkv, d)
    st = _load().orc_reshape_and_cache(
        _ptr(key), _ptr(value), slots.shape[0], hkv, d, _ptr(k_cache),
        _ptr(v_cache), nb, B, _kv_dtype_of(k_cache), _ptr(slots),
        float(k_scale), float(v_scale))
    if st != 0:
        raise ValueError("oracle reshape_and_cache: slot outside the pool")


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray,
                pairs: np.ndarray) -> None:
    """For each (src, dst) row of ``pairs``: cache[dst] = cache[src], K and V."""
    pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    nb = k_cache.shape[0]
    block_bytes = k_cache[0].nbytes
    st = _load().orc_copy_blocks(_ptr(k_cache), _ptr(v_cache), nb,
                                 block_bytes, _ptr(pairs), pairs.shape[0])
    if st != 0:
        raise ValueError("oracle copy_blocks: block id outside the pool")


def decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
           block_tables: np.ndarray, context_lens: np.ndarray, scale: float,
           k_scale: float = 1.0, v_scale: float = 1.0, units=None,
           nthreads: int = 1, out: np.ndarray | None = None) -> np.ndarray:
    """fp64 decode attention, one query token per sequence.

    q [B_s, H_q, d] bf16 bits; caches [num_blocks, B, H_kv, d];
    block_tables [B_s, max_blocks] int32; context_lens [B_s] int32 (tokens
    valid after this step's write).  ``units`` optionally restricts the work
    to a list of (seq, kv_head) pairs; other output rows are left as given in
    ``out`` (zeros by default).  Returns out [B_s, H_q, d] float64."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    nb, B, hkv, d = k_cache.shape
    bs, hq, dq = q.shape
    assert dq == d and bt.shape[0] == bs and cl.shape == (bs,)
    if out is None:
        out = np.zeros((bs, hq, d), dtype=np.float64)
    u_ptr, n_units = None, 0
    if units is not None:
        u = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
        u_ptr, n_units = _ptr(u), u.shape[0]
    st = _load().orc_decode(
        _ptr(out), _ptr(q), _ptr(np.ascontiguousarray(k_cache)),
        _ptr(np.ascontiguousarray(v_cache)), nb, B, hkv, d,
        _kv_dtype_of(k_cache), _ptr(bt), bt.shape[1], _ptr(cl), bs, hq,
        float(scale), float(k_scale), float(v_scale), u_ptr, n_units,
        int(nthreads))
    if st == -2:
        raise MemoryError("oracle decode: host allocation failed")
    if st != 0:
        raise ValueError("oracle decode: block id or context length out of range")
    return out
