"""Seeded synthetic inputs for the paged decode path.

This module is the one piece shared by the product side (benchmark) and the
oracle side (tests).  It draws numbers and shapes only: it holds none of the
method's arithmetic (no slot mapping, no attention, no quantisation) and
imports nothing from the rest of the package.

Workloads (all K/V/q i.i.d. N(0,1), rounded to bf16):

* ``tiny``      -- 4 sequences, context lengths {5, 16, 17, 40}, 4 query heads,
                   2 KV heads, d=64, block size 16, a 32-block pool assigned by
                   a seeded permutation, scale 1/8.
* ``llama8b``   -- Llama-3-8B layer shape: 32 query / 8 KV heads, d=128, block
                   size 16, batch 64.  Context length = prompt + output of the
                   first 64 requests of the seeded request mix of "Paged KV
                   cache" (ai-infra-handbooks), section "Why paging":
                   ``random.seed(0)``, prompt ``randint(100, 2000)``, output
                   ``randint(20, 1500)``.  Pool = ceil(1.2 x blocks used),
                   blocks placed by a seeded permutation.
* ``longctx``   -- same heads, batch 8, lengths {4K, 8K, 16K, 32K, 32K, 64K,
                   64K, 128K}; K multiplied by 3 on a seeded 1% of tokens.
* ``sweep``     -- ``llama8b`` lengths with block size in {1, 16, 64, 256},
                   bf16 or fp8-e4m3 cache.
* ``serving``   -- MHA 32/32 heads, d=128, block size 16, 256 sequences in 32
                   groups of 8 sharing a prefix (1024 tokens, or 1000 for the
                   copy-on-write variant), private suffix U[16, 2048].
"""
from __future__ import annotations

import math
import random
from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 1000


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits.

    Used only to turn drawn normals into bf16 inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def request_mix(count: int = 200):
    """(prompt, output) lengths of the seeded mix in "Paged KV cache"."""
    r = random.Random(0)
    return [(r.randint(100, 2000), r.randint(20, 1500)) for _ in range(count)]


@dataclass
class Workload:
    """A decode step's inputs, before any slot mapping or cache write.

    ``context_lens`` count tokens after this step's write, so the new token of
    sequence i sits at position ``context_lens[i] - 1``.  ``ctx_k``/``ctx_v``
    hold the K/V of positions 0..n_i-2 of every sequence, concatenated in
    sequence order ([sum(n_i - 1), H_kv, d] bf16 bits); ``k_new``/``v_new``
    hold the new token's K/V ([B_s, H_kv, d]).  ``block_tables`` is right-padded
    with 0.  ``junk_k``/``junk_v`` fill the whole pool before any write, so
    slots that are never written hold arbitrary bits (including NaN/Inf
    patterns) that must never reach an output."""
    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: str  # "bf16" or "fp8"
    num_blocks: int
    context_lens: np.ndarray
    block_tables: np.ndarray
    scale: float
    seed: int
    q: np.ndarray = field(repr=False, default=None)
    k_new: np.ndarray = field(repr=False, default=None)
    v_new: np.ndarray = field(repr=False, default=None)
    ctx_k: np.ndarray = field(repr=False, default=None)
    ctx_v: np.ndarray = field(repr=False, default=None)
    junk_k: np.ndarray = field(repr=False, default=None)
    junk_v: np.ndarray = field(repr=False, default=None)
    k_scale: float = 1.0
    v_scale: float = 1.0

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def elem_bytes(self) -> int:
        return 2 if self.kv_dtype == "bf16" else 1


def _place_blocks(rng, lengths, block_size, num_blocks):
    """Assign ceil(n/B) physical blocks per sequence from a seeded permutation."""
    counts = [max(1, math.ceil(n / block_size)) for n in lengths]
    assert sum(counts) <= num_blocks
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = np.zeros((len(lengths), max(counts)), dtype=np.int32)
    at = 0
    for i, c in enumerate(counts):
        tables[i, :c] = perm[at:at + c]
        at += c
    return tables


def per_tensor_scale(x_bits: np.ndarray) -> float:
    """fp32 amax(|x|)/448 of a bf16 tensor: the caller-chosen e4m3 scale."""
    u = (x_bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    amax = np.float32(np.max(np.abs(u))) if u.size else np.float32(1.0)
    return float(np.float32(amax) / np.float32(448.0))


def make(name: str, lengths, num_heads, num_kv_heads, head_dim, block_size,
         kv_dtype="bf16", pool_factor=1.2, num_blocks=None, seed=None,
         heavy_frac=0.0, heavy_mult=1.0, with_data=True) -> Workload:
    seed = SEED_BASE if seed is None else seed
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int32)
    used = int(sum(max(1, math.ceil(n / block_size)) for n in lengths))
    if num_blocks is None:
        num_blocks = int(math.ceil(pool_factor * used))
    tables = _place_blocks(rng, lengths, block_size, num_blocks)
    w = Workload(name, num_heads, num_kv_heads, head_dim, block_size, kv_dtype,
                 num_blocks, lengths, tables, 1.0 / math.sqrt(head_dim), seed)
    if not with_data:
        return w
    bs = len(lengths)
    n_ctx = int(np.sum(np.maximum(lengths - 1, 0)))
    w.q = normal_bf16(rng, (bs, num_heads, head_dim))
    w.k_new = normal_bf16(rng, (bs, num_kv_heads, head_dim))
    w.v_new = normal_bf16(rng, (bs, num_kv_heads, head_dim))
    kf = rng.standard_normal(size=(n_ctx, num_kv_heads, head_dim), dtype=np.float32)
    if heavy_frac > 0 and n_ctx > 0:
        heavy = rng.random(n_ctx) < heavy_frac
        kf[heavy] *= np.float32(heavy_mult)
    w.ctx_k = bf16_bits(kf)
    del kf
    w.ctx_v = normal_bf16(rng, (n_ctx, num_kv_heads, head_dim))
    shape = (num_blocks, block_size, num_kv_heads, head_dim)
    if kv_dtype == "bf16":
        w.junk_k = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)
        w.junk_v = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)
    else:
        w.junk_k = rng.integers(0, 256, size=shape, dtype=np.uint8)
        w.junk_v = rng.integers(0, 256, size=shape, dtype=np.uint8)
        w.k_scale = per_tensor_scale(np.concatenate([w.ctx_k.ravel(), w.k_new.ravel()]))
        w.v_scale = per_tensor_scale(np.concatenate([w.ctx_v.ravel(), w.v_new.ravel()]))
    return w


# ---- the named workloads ----------------------------------------------------

LONG_CTX_LENS = [4096, 8192, 16384, 32768, 32768, 65536, 65536, 131072]


def llama8b_lengths(batch: int = 64):
    return [p + o for p, o in request_mix(200)[:batch]]


def tiny(**kw) -> Workload:
    return make("tiny", [5, 16, 17, 40], 4, 2, 64, 16, num_blocks=32,
                seed=SEED_BASE + 1, **kw)


def llama8b(batch: int = 64, block_size: int = 16, kv_dtype: str = "bf16",
            **kw) -> Workload:
    return make(f"llama8b-b{batch}-bs{block_size}-{kv_dtype}",
                llama8b_lengths(batch), 32, 8, 128, block_size, kv_dtype,
                seed=SEED_BASE + 2, **kw)


def longctx(lengths=None, **kw) -> Workload:
    return make("longctx", LONG_CTX_LENS if lengths is None else lengths,
                32, 8, 128, 16, seed=SEED_BASE + 3, heavy_frac=0.01,
                heavy_mult=3.0, **kw)


def sweep(block_size: int, kv_dtype: str, **kw) -> Workload:
    w = make(f"sweep-bs{block_size}-{kv_dtype}", llama8b_lengths(64), 32, 8,
             128, block_size, kv_dtype, seed=SEED_BASE + 4, **kw)
    return w


@dataclass
class ServingMix:
    """Shape of the copy-on-write serving step (no pool decisions here)."""
    num_groups: int
    group_size: int
    prefix_len: int
    suffix_lens: np.ndarray  # [num_groups * group_size]
    num_heads: int = 32
    num_kv_heads: int = 32
    head_dim: int = 128
    block_size: int = 16
    seed: int = SEED_BASE + 5

    @property
    def num_seqs(self) -> int:
        return self.num_groups * self.group_size

    def free_order(self, num_blocks: int) -> np.ndarray:
        """Seeded initial order of the pool's free queue (scatters blocks)."""
        return np.random.default_rng(self.seed + 7).permutation(num_blocks).astype(np.int32)


def serving(num_groups=32, group_size=8, prefix_len=1024, max_suffix=2048,
            min_suffix=16) -> ServingMix:
    rng = np.random.default_rng(SEED_BASE + 5)
    suffix = rng.integers(min_suffix, max_suffix + 1,
                          size=num_groups * group_size).astype(np.int32)
    return ServingMix(num_groups, group_size, prefix_len, suffix)


def serving_data(mix: ServingMix, num_blocks: int, unique_tokens: int):
    """K/V/q draws for the serving mix: pool junk, ``unique_tokens`` context
    rows (consumed in order by whoever fills the pool), and the step's new
    token K/V and q.  Returns a dict of bf16 bit arrays."""
    rng = np.random.default_rng(mix.seed + 1)
    H, Hkv, d, B = mix.num_heads, mix.num_kv_heads, mix.head_dim, mix.block_size
    shape = (num_blocks, B, Hkv, d)
    return {
        "junk_k": rng.integers(0, 1 << 16, size=shape, dtype=np.uint16),
        "junk_v": rng.integers(0, 1 << 16, size=shape, dtype=np.uint16),
        "ctx_k": normal_bf16(rng, (unique_tokens, Hkv, d)),
        "ctx_v": normal_bf16(rng, (unique_tokens, Hkv, d)),
        "q": normal_bf16(rng, (mix.num_seqs, H, d)),
        "k_new": normal_bf16(rng, (mix.num_seqs, Hkv, d)),
        "v_new": normal_bf16(rng, (mix.num_seqs, Hkv, d)),
    }
