"""Runs one decode step of a synthetic workload on both sides.

``product_step`` drives the product path only (native slot mapping, the
library's cache-write and decode kernels through the Python binding);
``oracle_step`` drives the oracle only (its own slot formula, its own cache
write and fp64 decode).  The two share the seeded workload and nothing else.
"""
from __future__ import annotations

import os

import numpy as np
import torch

from oracle import core as ocore
from oracle import pool_model
from paged_kv_cache_108_gb300 import ops, pool, synth

BF16_ATOL, BF16_RTOL = 1e-2, 2e-2
FP8_ATOL, FP8_RTOL = 6e-2, 6e-2


def ctx_positions(w: synth.Workload):
    """(sequence index, position) of every context token, in sequence order."""
    seqs, poss = [], []
    for i, n in enumerate(w.context_lens):
        if n > 1:
            seqs.append(np.full(n - 1, i, dtype=np.int32))
            poss.append(np.arange(n - 1, dtype=np.int32))
    if not seqs:
        return np.zeros(0, np.int32), np.zeros(0, np.int32)
    return np.concatenate(seqs), np.concatenate(poss)


def new_positions(w: synth.Workload):
    return np.maximum(w.context_lens - 1, 0).astype(np.int32)


def to_dev_bits(a: np.ndarray, kv_dtype: str, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return t.view(torch.bfloat16) if kv_dtype == "bf16" else t


def bits_from_dev(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def product_step(w: synth.Workload, device="cuda", partition_tokens=0, kernel=0,
                 skip_new=None):
    """Cache writes (context, then the step's new token) and decode on the GPU.

    ``skip_new``: optional boolean mask of sequences whose new-token slot is
    replaced by -1 (padding)."""
    B = w.block_size
    kc = to_dev_bits(w.junk_k, w.kv_dtype, device)
    vc = to_dev_bits(w.junk_v, w.kv_dtype, device)
    ks = vs = None
    if w.kv_dtype == "fp8":
        ks = torch.tensor([w.k_scale], dtype=torch.float32, device=device)
        vs = torch.tensor([w.v_scale], dtype=torch.float32, device=device)
    seq_idx, pos = ctx_positions(w)
    slots_ctx = pool.slot_mapping(w.block_tables, B, pos, seq_idx) if pos.size else np.zeros(0, np.int32)
    if pos.size:
        ops.reshape_and_cache(to_dev_bits(w.ctx_k, "bf16", device), to_dev_bits(w.ctx_v, "bf16", device),
                              kc, vc, torch.from_numpy(slots_ctx).to(device), ks, vs)
    has_new = w.context_lens > 0
    slots_new = np.full(w.num_seqs, -1, dtype=np.int32)
    idx = np.nonzero(has_new)[0].astype(np.int32)
    if idx.size:
        slots_new[idx] = pool.slot_mapping(w.block_tables, B, new_positions(w)[idx], idx)
    if skip_new is not None:
        slots_new[skip_new] = -1
    ops.reshape_and_cache(to_dev_bits(w.k_new, "bf16", device), to_dev_bits(w.v_new, "bf16", device),
                          kc, vc, torch.from_numpy(slots_new).to(device), ks, vs)
    q = to_dev_bits(w.q, "bf16", device)
    bt = torch.from_numpy(w.block_tables).to(device)
    cl = torch.from_numpy(w.context_lens).to(device)
    ws = ops.alloc_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_blocks, B,
                             partition_tokens, device=device)
    # arbitrary bytes: the workspace needs no initialisation; word 0 is zeroed
    # because the tensor-core kernel reports expired waits / bad ids there
    ws.random_(0, 256)
    ws[:4] = 0
    out = torch.empty_like(q)
    ops.decode(out, q, kc, vc, bt, cl, w.scale, ks, vs, ws, partition_tokens, kernel)
    torch.cuda.synchronize()
    err = int(ws[:4].view(torch.int32).item()) if ws.numel() >= 4 else 0
    return {"out": out.float().cpu().numpy().astype(np.float64), "k_cache": bits_from_dev(kc),
            "v_cache": bits_from_dev(vc), "slots_ctx": slots_ctx, "slots_new": slots_new,
            "err": err,
            "dev": {"k_cache": kc, "v_cache": vc, "q": q, "bt": bt, "cl": cl, "ks": ks, "vs": vs,
                    "ws": ws}}


def oracle_step(w: synth.Workload, skip_new=None, decode=True, units=None):
    B = w.block_size
    kc, vc = w.junk_k.copy(), w.junk_v.copy()
    seq_idx, pos = ctx_positions(w)
    tables = w.block_tables
    slots_ctx = np.array([pool_model.slot_of(tables[s], int(p), B) for s, p in zip(seq_idx, pos)],
                         dtype=np.int32)
    if pos.size:
        ocore.reshape_and_cache(w.ctx_k, w.ctx_v, kc, vc, slots_ctx, w.k_scale, w.v_scale)
    slots_new = np.array([pool_model.slot_of(tables[i], int(n) - 1, B) if n > 0 else -1
                          for i, n in enumerate(w.context_lens)], dtype=np.int32)
    if skip_new is not None:
        slots_new[skip_new] = -1
    ocore.reshape_and_cache(w.k_new, w.v_new, kc, vc, slots_new, w.k_scale, w.v_scale)
    res = {"k_cache": kc, "v_cache": vc, "slots_ctx": slots_ctx, "slots_new": slots_new}
    if decode:
        res["out"] = ocore.decode(w.q, kc, vc, tables, w.context_lens, w.scale, w.k_scale,
                                  w.v_scale, units=units, nthreads=os.cpu_count() or 1)
    return res


def assert_close(got: np.ndarray, ref: np.ndarray, fp8: bool, mask=None):
    atol, rtol = (FP8_ATOL, FP8_RTOL) if fp8 else (BF16_ATOL, BF16_RTOL)
    g, r = got, ref
    if mask is not None:
        g, r = got[mask], ref[mask]
    err = np.abs(g - r)
    bad = ~(err <= atol + rtol * np.abs(r))
    if bad.any():
        i = np.argmax(err - (atol + rtol * np.abs(r)))
        raise AssertionError(
            f"{int(bad.sum())} of {bad.size} outputs outside |g-r| <= {atol} + {rtol}|r|; "
            f"worst flat index {i}: got {g.ravel()[i]}, oracle {r.ravel()[i]}")
    return float(err.max()) if err.size else 0.0
