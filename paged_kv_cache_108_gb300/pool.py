"""Host-side block pool (native, libpa.so) and per-sequence block tables.

``BlockPool`` wraps the C pool: FIFO free queue, ref counts, all-or-nothing
allocation, fork (incref), release and the copy-on-write decision.
``SequenceTables`` keeps each sequence's block table on the host and turns
it into the int32 step tensors the kernels consume: ``block_tables``
(right-padded with 0), ``slot_mapping`` (computed by the library's
``pa_slot_mapping``) and ``context_lens`` -- "4.6 PagedAttention & KV-Cache
Memory Management" (llm-stack-book), sections "Block Tables, the Allocator &
Copy-on-Write" and "From Python bookkeeping to the tensors the kernel
actually takes".
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _lib
from ._lib import PaOOM


def load():
    return _lib.lib()


def _i32_array(values):
    a = np.ascontiguousarray(np.asarray(values, dtype=np.int32))
    return a, a.ctypes.data_as(_lib.PI32)


class BlockPool:
    def __init__(self, num_blocks: int, free_order=None):
        L = _lib.lib()
        if free_order is None:
            h = L.pa_pool_create(int(num_blocks))
        else:
            arr, ptr = _i32_array(free_order)
            if arr.size != num_blocks:
                raise ValueError("free_order must list every block once")
            h = L.pa_pool_create_ordered(int(num_blocks), ptr)
        if not h:
            raise ValueError(L.pa_last_error().decode())
        self._h = ctypes.c_void_p(h)
        self._lib = L

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._lib.pa_pool_destroy(h)
            self._h = None

    @property
    def num_blocks(self) -> int:
        return self._lib.pa_pool_num_blocks(self._h)

    def num_free(self) -> int:
        return self._lib.pa_pool_num_free(self._h)

    def refcount(self, block: int) -> int:
        return self._lib.pa_pool_refcount(self._h, int(block))

    def free_order(self):
        n = self.num_free()
        out = np.zeros(max(n, 1), dtype=np.int32)
        self._lib.pa_pool_free_order(self._h, out.ctypes.data_as(_lib.PI32), n)
        return out[:n].tolist()

    def allocate(self, n: int):
        """n blocks from the head of the free queue, or None if fewer are free."""
        out = np.zeros(max(int(n), 1), dtype=np.int32)
        st = self._lib.pa_pool_alloc(self._h, int(n), out.ctypes.data_as(_lib.PI32))
        if st == _lib.PA_ERR_OOM:
            return None
        _lib.check(st)
        return out[:n].tolist()

    def incref(self, blocks) -> None:
        arr, ptr = _i32_array(blocks)
        _lib.check(self._lib.pa_pool_incref(self._h, ptr, arr.size))

    def free(self, blocks) -> None:
        arr, ptr = _i32_array(blocks)
        _lib.check(self._lib.pa_pool_free(self._h, ptr, arr.size))

    def cow(self, block: int):
        """(src, dst) for a write into ``block``; dst == src when it is private."""
        dst = ctypes.c_int32(0)
        _lib.check(self._lib.pa_pool_cow(self._h, int(block), ctypes.byref(dst)))
        return int(block), int(dst.value)


    # ---- prefix caching across requests (full blocks) ----
    def enable_prefix_cache(self, block_size: int) -> None:
        _lib.check(self._lib.pa_pool_enable_prefix_cache(self._h, int(block_size)))
        self.prefix_block_size = int(block_size)

    def allocate_prefix(self, tokens):
        """Blocks for a new sequence with prompt ``tokens``: (blocks,
        cached_tokens), or None if the pool is short; the leading
        ``cached_tokens`` tokens' K/V are already in the shared blocks."""
        arr, ptr = _i32_array(tokens)
        bs = self.prefix_block_size
        out = np.zeros(max(-(-arr.size // bs), 1), dtype=np.int32)
        cached = ctypes.c_int32(0)
        st = self._lib.pa_pool_alloc_prefix(self._h, ptr, arr.size,
                                            out.ctypes.data_as(_lib.PI32), ctypes.byref(cached))
        if st == _lib.PA_ERR_OOM:
            return None
        _lib.check(st)
        return out[:-(-arr.size // bs)].tolist(), int(cached.value)

    def register_block(self, block: int, parent: int, tokens) -> None:
        arr, ptr = _i32_array(tokens)
        if arr.size != self.prefix_block_size:
            raise ValueError("a registered block holds exactly block_size tokens")
        _lib.check(self._lib.pa_pool_register_block(self._h, int(block), int(parent), ptr))

    def num_cached(self) -> int:
        return self._lib.pa_pool_num_cached(self._h)


def slot_mapping(block_tables: np.ndarray, block_size: int, positions, token_seq=None):
    """Slots of tokens at ``positions`` (sequence ``token_seq[i]``, default i)."""
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int32))
    out = np.zeros(max(pos.size, 1), dtype=np.int32)
    seq_ptr = None
    if token_seq is not None:
        seq = np.ascontiguousarray(np.asarray(token_seq, dtype=np.int32))
        seq_ptr = seq.ctypes.data_as(_lib.PI32)
    _lib.check(_lib.lib().pa_slot_mapping(
        bt.ctypes.data_as(_lib.PI32), bt.shape[0], bt.shape[1], int(block_size), seq_ptr,
        pos.ctypes.data_as(_lib.PI32), pos.size, out.ctypes.data_as(_lib.PI32)))
    return out[:pos.size]


class SequenceTables:
    """Per-sequence block tables over a ``BlockPool``."""

    def __init__(self, pool: BlockPool, block_size: int):
        self.pool = pool
        self.block_size = int(block_size)
        self.tables = {}

    def allocate(self, seq, num_tokens: int) -> None:
        n = -(-int(num_tokens) // self.block_size)
        blocks = self.pool.allocate(n)
        if blocks is None:
            raise PaOOM(_lib.PA_ERR_OOM, f"need {n} blocks, {self.pool.num_free()} free")
        self.tables[seq] = blocks

    def append_token(self, seq, cur_len: int) -> None:
        """Grow the table before position ``cur_len`` is written, if that
        position opens a new block."""
        if cur_len % self.block_size == 0:
            blocks = self.pool.allocate(1)
            if blocks is None:
                raise PaOOM(_lib.PA_ERR_OOM, "no free block to grow the sequence")
            self.tables[seq].append(blocks[0])

    def fork(self, parent, child) -> None:
        self.pool.incref(self.tables[parent])
        self.tables[child] = list(self.tables[parent])

    def cow_for_write(self, seq, pos: int):
        """Make the block holding ``pos`` private; (src, dst) to copy if they differ."""
        lb = pos // self.block_size
        src, dst = self.pool.cow(self.tables[seq][lb])
        self.tables[seq][lb] = dst
        return src, dst

    def slot_index(self, seq, pos: int) -> int:
        return int(slot_mapping(np.asarray([self.tables[seq]], dtype=np.int32),
                                self.block_size, [pos])[0])

    def free_seq(self, seq) -> None:
        self.pool.free(self.tables.pop(seq))

    def block_table_array(self, seqs, max_blocks=None) -> np.ndarray:
        tabs = [self.tables[s] for s in seqs]
        width = max_blocks or max(1, max(len(t) for t in tabs))
        bt = np.zeros((len(tabs), width), dtype=np.int32)
        for i, t in enumerate(tabs):
            bt[i, :len(t)] = t
        return bt

    def build_step_tensors(self, seqs, cur_lens, max_blocks=None):
        """(block_tables, slot_mapping, context_lens) for one decode step in
        which sequence ``seqs[i]`` writes position ``cur_lens[i]``; the tables
        must already hold that position (``append_token`` first)."""
        bt = self.block_table_array(seqs, max_blocks)
        slots = slot_mapping(bt, self.block_size, cur_lens)
        ctx = np.asarray(cur_lens, dtype=np.int32) + 1
        return bt, slots, ctx
