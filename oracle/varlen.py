"""fp64 variable-length causal paged attention -- TEST INFRASTRUCTURE.

Definition followed: "Paged KV cache" (ai-infra-handbooks), section "Paged
attention" and its input table.  A step holds the new tokens of several
requests laid end to end; request r's are queries qsl[r] .. qsl[r+1]-1, the
last num_new of its seq_len context tokens (seq_len counts them).  New token
j of the request sits at position seq_len - num_new + j and attends to
positions 0 .. seq_len - num_new + j of its own context; query head h reads
KV head h // (H / H_kv).  Each output row is softmax(scale q K^T) V over
those positions, computed the textbook way (max, exp, sum, divide) in fp64
with every cache element widened exactly (E4M3 codes times their per-tensor
scale).  A request with more new tokens than context has no valid position
for its first tokens: all its rows are zero (a reading; the pages are
silent).  The arithmetic is ``orc_varlen`` in ``pa_oracle.c``; this module
only marshals arrays.
"""
from __future__ import annotations

import numpy as np

from . import core


def varlen_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, block_tables,
                     seq_lens, query_start_loc, scale: float, k_scale: float = 1.0,
                     v_scale: float = 1.0, nthreads: int | None = None) -> np.ndarray:
    """q [N, H, d] bf16 bits; caches [num_blocks, B, H_kv, d] (uint16 bf16
    bits or uint8 e4m3 codes with per-tensor scales); block_tables
    [R, max_blocks]; seq_lens [R]; query_start_loc [R + 1].  Returns
    out [N, H, d] float64.  ``nthreads`` spreads the (request, KV head)
    units over host threads (default: every core); it does not change the
    result."""
    import os

    qb = np.ascontiguousarray(q, dtype=np.uint16)
    kc = np.ascontiguousarray(k_cache)
    vc = np.ascontiguousarray(v_cache)
    assert kc.shape == vc.shape and kc.dtype == vc.dtype
    nb, B, hkv, d = kc.shape
    N, H, dq = qb.shape
    assert dq == d
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int64).astype(np.int32))
    qsl = np.ascontiguousarray(np.asarray(query_start_loc, dtype=np.int64).astype(np.int32))
    R = sl.shape[0]
    assert qsl.shape == (R + 1,) and int(qsl[-1]) <= N
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32).reshape(R, -1))
    out = np.zeros((N, H, d), dtype=np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    st = core._load().orc_varlen(
        core._ptr(out), core._ptr(qb), core._ptr(kc), core._ptr(vc), nb, B, hkv, d,
        core._kv_dtype_of(kc), core._ptr(bt), bt.shape[1], core._ptr(sl), core._ptr(qsl),
        R, H, float(scale), float(np.float32(k_scale)), float(np.float32(v_scale)),
        int(nthreads))
    if st == -2:
        raise MemoryError("oracle varlen: host allocation failed")
    if st != 0:
        raise ValueError("oracle varlen: block id, length or head count out of range")
    return out
