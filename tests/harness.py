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


# ---------------------------------------------------------------- serving mix

def serving_pool_size(mix: synth.ServingMix) -> int:
    """Blocks for the serving mix with 20 % headroom (prefix blocks shared per
    group, private suffix blocks, one copy-on-write block per sequence)."""
    B = mix.block_size
    shared = mix.num_groups * -(-mix.prefix_len // B)
    private = sum(-(-(mix.prefix_len + int(s)) // B) - mix.prefix_len // B + 1
                  for s in mix.suffix_lens)
    return int(1.2 * (shared + private)) + 8


def _serving_tables(mix: synth.ServingMix, tables, num_blocks):
    """Build the serving state with `tables` (native or model bookkeeping):
    per group a parent allocates the prefix and forks the rest of the group;
    every sequence then takes its first divergent write at position
    prefix_len (copy-on-write if that block is shared) and grows to its
    context length.  Returns the (src, dst) copy pairs in order and each
    group's prefix table as it was when the prefix was written (before any
    copy-on-write remapped the parent's last shared block)."""
    G, P, B = mix.group_size, mix.prefix_len, mix.block_size
    pairs, prefix_tables = [], []
    for grp in range(mix.num_groups):
        parent = grp * G
        tables.allocate(parent, P)
        prefix_tables.append(list(tables.tables[parent]))
        for c in range(1, G):
            tables.fork(parent, parent + c)
    for i in range(mix.num_seqs):
        n = P + int(mix.suffix_lens[i])
        tables.append_token(i, P)
        src, dst = tables.cow_for_write(i, P)
        if src != dst:
            pairs.append((src, dst))
        for pos in range(P + 1, n):
            tables.append_token(i, pos)
    return pairs, prefix_tables


def serving_lengths(mix):
    return (mix.prefix_len + mix.suffix_lens).astype(np.int32)


def _serving_writes(mix, table_arr, prefix_tables, slot_fn):
    """(slots of prefix tokens, slots of suffix context tokens, slots of the
    step's new tokens) in the order the context rows are consumed: each
    group's prefix through its table at prefix time, then each sequence's
    suffix positions prefix..n-2, then position n-1 of every sequence."""
    P = mix.prefix_len
    n = serving_lengths(mix)
    pre = [slot_fn(prefix_tables[g], p) for g in range(mix.num_groups) for p in range(P)]
    suf = [slot_fn(table_arr[i], p) for i in range(mix.num_seqs) for p in range(P, int(n[i]) - 1)]
    new = [slot_fn(table_arr[i], int(n[i]) - 1) for i in range(mix.num_seqs)]
    return (np.array(pre, np.int32), np.array(suf, np.int32), np.array(new, np.int32))


def serving_unique_tokens(mix):
    n = serving_lengths(mix)
    return mix.num_groups * mix.prefix_len + int(np.sum(n - 1 - mix.prefix_len))


def serving_product(mix, data, num_blocks, device="cuda", kernel=0, shared_prefix_group=0):
    """Product path: native pool and tables, cache writes, copy-on-write copies
    and decode on the GPU.  The prefix is written before the copies (it was
    computed before the fork); the suffix and the new token after them."""
    npool = pool.BlockPool(num_blocks, free_order=mix.free_order(num_blocks))
    tabs = pool.SequenceTables(npool, mix.block_size)
    pairs, prefix_tables = _serving_tables(mix, tabs, num_blocks)
    bt = tabs.block_table_array(list(range(mix.num_seqs)))
    B = mix.block_size
    # one native slot-mapping call per kind of write
    n = serving_lengths(mix)
    P = mix.prefix_len
    pt = np.array(prefix_tables, dtype=np.int32)
    pre_seq = np.repeat(np.arange(mix.num_groups), P).astype(np.int32)
    pre_pos = np.tile(np.arange(P), mix.num_groups).astype(np.int32)
    suf_seq = np.concatenate([np.full(int(n[i]) - 1 - P, i, np.int32) for i in range(mix.num_seqs)])
    suf_pos = np.concatenate([np.arange(P, int(n[i]) - 1, dtype=np.int32) for i in range(mix.num_seqs)])
    s_pre = pool.slot_mapping(pt, B, pre_pos, pre_seq)
    s_suf = pool.slot_mapping(bt, B, suf_pos, suf_seq)
    s_new = pool.slot_mapping(bt, B, n - 1, np.arange(mix.num_seqs, dtype=np.int32))
    kc = to_dev_bits(data["junk_k"], "bf16", device)
    vc = to_dev_bits(data["junk_v"], "bf16", device)
    npre = s_pre.size
    ck, cv = data["ctx_k"], data["ctx_v"]
    ops.reshape_and_cache(to_dev_bits(ck[:npre], "bf16", device), to_dev_bits(cv[:npre], "bf16", device),
                          kc, vc, torch.from_numpy(s_pre).to(device))
    pr = np.array(pairs, dtype=np.int32).reshape(-1, 2)
    ops.copy_blocks(kc, vc, torch.from_numpy(pr).to(device))
    ops.reshape_and_cache(to_dev_bits(ck[npre:], "bf16", device), to_dev_bits(cv[npre:], "bf16", device),
                          kc, vc, torch.from_numpy(s_suf).to(device))
    ops.reshape_and_cache(to_dev_bits(data["k_new"], "bf16", device),
                          to_dev_bits(data["v_new"], "bf16", device), kc, vc,
                          torch.from_numpy(s_new).to(device))
    q = to_dev_bits(data["q"], "bf16", device)
    bt_d = torch.from_numpy(bt).to(device)
    cl = torch.from_numpy(n).to(device)
    ws = ops.alloc_workspace(mix.num_seqs, mix.num_heads, mix.head_dim, bt.shape[1], B, device=device)
    ws.random_(0, 256)
    ws[:4] = 0
    out = torch.empty_like(q)
    if shared_prefix_group:
        ops.decode_shared_prefix(out, q, kc, vc, bt_d, cl, shared_prefix_group,
                                 mix.head_dim ** -0.5)
    else:
        ops.decode(out, q, kc, vc, bt_d, cl, mix.head_dim ** -0.5, workspace=ws, kernel=kernel)
    torch.cuda.synchronize()
    return {"tables": bt, "pairs": pr, "slots": (s_pre, s_suf, s_new),
            "k_cache": bits_from_dev(kc), "v_cache": bits_from_dev(vc),
            "out": out.float().cpu().numpy().astype(np.float64),
            "err": int(ws[:4].view(torch.int32).item())}


def serving_oracle(mix, data, num_blocks, decode=True):
    mpool = pool_model.BlockPoolModel(num_blocks, free_order=list(mix.free_order(num_blocks)))
    tabs = pool_model.SequenceTablesModel(mpool, mix.block_size)
    pairs, prefix_tables = _serving_tables(mix, tabs, num_blocks)
    width = max(len(t) for t in tabs.tables.values())
    bt = np.zeros((mix.num_seqs, width), dtype=np.int32)
    for i in range(mix.num_seqs):
        bt[i, :len(tabs.tables[i])] = tabs.tables[i]
    s_pre, s_suf, s_new = _serving_writes(
        mix, bt, prefix_tables, lambda row, p: pool_model.slot_of(row, p, mix.block_size))
    kc, vc = data["junk_k"].copy(), data["junk_v"].copy()
    npre = s_pre.size
    ocore.reshape_and_cache(data["ctx_k"][:npre], data["ctx_v"][:npre], kc, vc, s_pre)
    pr = np.array(pairs, dtype=np.int32).reshape(-1, 2)
    ocore.copy_blocks(kc, vc, pr)
    ocore.reshape_and_cache(data["ctx_k"][npre:], data["ctx_v"][npre:], kc, vc, s_suf)
    ocore.reshape_and_cache(data["k_new"], data["v_new"], kc, vc, s_new)
    res = {"tables": bt, "pairs": pr, "slots": (s_pre, s_suf, s_new), "k_cache": kc,
           "v_cache": vc}
    if decode:
        res["out"] = ocore.decode(data["q"], kc, vc, bt, serving_lengths(mix),
                                  mix.head_dim ** -0.5, nthreads=os.cpu_count() or 1)
    return res
