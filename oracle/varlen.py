"""fp64 variable-length paged attention -- TEST INFRASTRUCTURE.

Definition followed: "Paged KV cache" (ai-infra-handbooks), ``paged_attention``
and the section "Paged attention".  A step holds N new tokens from B
requests laid end to end; request i's new tokens are q[qsl[i]:qsl[i+1]]
and are the last num_new = qsl[i+1] - qsl[i] tokens of its context of
seq_lens[i] tokens.  Its K/V are gathered through the block table into
contiguous [seq_len, H_kv, d] arrays; new token j sits at position
seq_len - num_new + j and sees positions 0..seq_len - num_new + j (the
lower-triangular mask with diagonal seq_len - num_new); query head h reads KV
head h // (H / H_kv); out = softmax(scale q K^T over the visible keys) V.
Everything is widened exactly and computed in float64 with numpy, one
request at a time, no blocking or reordering.
"""
from __future__ import annotations

import numpy as np

from .core import bf16_to_f64, e4m3_decode


def _widen(cache: np.ndarray, scale: float) -> np.ndarray:
    if cache.dtype == np.uint16:
        return bf16_to_f64(cache)
    return e4m3_decode(cache) * float(np.float32(scale))


def gather(cache: np.ndarray, table, seq_len: int) -> np.ndarray:
    """The first seq_len token rows of one sequence, [seq_len, H_kv, d]."""
    B = cache.shape[1]
    nblk = -(-seq_len // B)
    rows = cache[np.asarray(table[:nblk], dtype=np.int64)]
    return rows.reshape(nblk * B, *cache.shape[2:])[:seq_len]


def varlen_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, block_tables,
                     seq_lens, query_start_loc, scale: float, k_scale: float = 1.0,
                     v_scale: float = 1.0) -> np.ndarray:
    """q [N, H, d] bf16 bits; caches [num_blocks, B, H_kv, d] (bf16 bits or
    e4m3 codes with per-tensor scales).  Returns out [N, H, d] float64."""
    qf = bf16_to_f64(np.asarray(q, dtype=np.uint16))
    kf = _widen(k_cache, k_scale)
    vf = _widen(v_cache, v_scale)
    N, H, d = qf.shape
    Hkv = k_cache.shape[2]
    rep = H // Hkv
    out = np.zeros((N, H, d), dtype=np.float64)
    for i, seq_len in enumerate(seq_lens):
        start, end = int(query_start_loc[i]), int(query_start_loc[i + 1])
        num_new = end - start
        if num_new == 0:
            continue
        k = gather(kf, block_tables[i], int(seq_len))         # [S, Hkv, d]
        v = gather(vf, block_tables[i], int(seq_len))
        k = np.repeat(k, rep, axis=1)                          # head h reads KV head h // rep
        v = np.repeat(v, rep, axis=1)
        scores = np.einsum("thd,shd->hts", qf[start:end], k) * scale      # [H, T, S]
        visible = np.tril(np.ones((num_new, int(seq_len)), dtype=bool),
                          k=int(seq_len) - num_new)
        scores = np.where(visible[None], scores, -np.inf)
        scores -= scores.max(axis=-1, keepdims=True)
        p = np.exp(scores)
        p /= p.sum(axis=-1, keepdims=True)
        out[start:end] = np.einsum("hts,shd->thd", p, v)
    return out
