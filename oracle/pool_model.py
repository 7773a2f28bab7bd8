"""Pure-Python model of the block pool and block tables -- TEST INFRASTRUCTURE.

Followed definitions:

* Free queue and ref counts: "Paged KV cache" (ai-infra-handbooks), class
  ``BlockPool`` -- a FIFO queue of free ids initialised 0..n-1, allocation
  takes from the head and is all-or-nothing (returns None when short), a free
  decrements each ref count and appends blocks that reach zero to the tail.
* Per-sequence tables, growth and slots: "4.6 PagedAttention & KV-Cache
  Memory Management" (llm-stack-book), class ``BlockManager`` -- allocate
  ceil(n/B) blocks for a prompt, grow by one block exactly when the position
  about to be written is a multiple of B, slot = table[p // B] * B + p % B.
* Fork and copy-on-write: same page, section "Copy-on-write for shared
  prefixes" -- fork copies the table and increments every ref count; before a
  write into a block with ref count > 1 a fresh block is taken, the old ref
  count is decremented, the table entry is remapped, and (src, dst) is
  reported for a device copy; with ref count 1 the write goes in place.

* Prefix caching across requests (``PrefixCachePoolModel``): "Paged KV
  cache" (ai-infra-handbooks), copy-on-write exercise -- vLLM V1 shares only
  full blocks and every answer starts writing in its own block; "4.6
  PagedAttention & KV-Cache Memory Management", section "Copy-on-write for
  shared prefixes" -- the same machinery generalises to reuse across
  requests.  The pages do not say how a block is recognised; the reading
  taken: a full block is the content (parent block, parent generation, its
  B tokens), a generation advances whenever a block is handed out fresh (its
  entry dies with it), freed cached blocks wait in the free queue and leave it
  when matched.  Kept as plain dictionaries keyed by that tuple.

Readings where the pages differ: FIFO (the handbook's deque and its printed
``[5, 6, 7, 0]`` example) rather than the llm-stack-book's ``pop()`` from the
end; all-or-nothing allocation instead of raising after a partial pop.
"""
from __future__ import annotations

from collections import deque


class PoolExhausted(Exception):
    pass


class BlockPoolModel:
    def __init__(self, num_blocks: int, free_order=None):
        self.num_blocks = num_blocks
        self.ref_cnt = [0] * num_blocks
        order = range(num_blocks) if free_order is None else free_order
        self.free_queue = deque(order)

    def num_free(self) -> int:
        return len(self.free_queue)

    def refcount(self, blk: int) -> int:
        return self.ref_cnt[blk]

    def allocate(self, n: int):
        if n > len(self.free_queue):
            return None
        blocks = [self.free_queue.popleft() for _ in range(n)]
        for b in blocks:
            self.ref_cnt[b] = 1
        return blocks

    def incref(self, blocks) -> None:
        for b in blocks:
            self.ref_cnt[b] += 1

    def free(self, blocks) -> None:
        for b in blocks:
            self.ref_cnt[b] -= 1
            if self.ref_cnt[b] == 0:
                self.free_queue.append(b)

    def cow(self, blk: int):
        """(src, dst) for a write into ``blk``; dst == src when private."""
        if self.ref_cnt[blk] == 1:
            return blk, blk
        new = self.allocate(1)
        if new is None:
            raise PoolExhausted("no free block for copy-on-write")
        self.ref_cnt[blk] -= 1
        return blk, new[0]


def slot_of(table, pos: int, block_size: int) -> int:
    """Flat pool slot of logical position ``pos``."""
    return table[pos // block_size] * block_size + pos % block_size


class SequenceTablesModel:
    """Sequence-level bookkeeping on top of ``BlockPoolModel``."""

    def __init__(self, pool: BlockPoolModel, block_size: int):
        self.pool = pool
        self.block_size = block_size
        self.tables = {}

    def allocate(self, seq, num_tokens: int) -> None:
        n = -(-num_tokens // self.block_size)
        blocks = self.pool.allocate(n)
        if blocks is None:
            raise PoolExhausted(f"need {n} blocks, {self.pool.num_free()} free")
        self.tables[seq] = blocks

    def append_token(self, seq, cur_len: int) -> None:
        """Grow before writing position ``cur_len`` if it opens a new block."""
        if cur_len % self.block_size == 0:
            blocks = self.pool.allocate(1)
            if blocks is None:
                raise PoolExhausted("no free block to grow the sequence")
            self.tables[seq].append(blocks[0])

    def fork(self, parent, child) -> None:
        self.tables[child] = list(self.tables[parent])
        self.pool.incref(self.tables[parent])

    def cow_for_write(self, seq, pos: int):
        """Make the block holding ``pos`` private; return (src, dst)."""
        lb = pos // self.block_size
        src, dst = self.pool.cow(self.tables[seq][lb])
        self.tables[seq][lb] = dst
        return src, dst

    def slot_index(self, seq, pos: int) -> int:
        return slot_of(self.tables[seq], pos, self.block_size)

    def free_seq(self, seq) -> None:
        self.pool.free(self.tables.pop(seq))


class PrefixCachePoolModel(BlockPoolModel):
    """``BlockPoolModel`` plus full-block prefix caching (see module notes)."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        super().__init__(num_blocks, free_order)
        self.block_size = block_size
        self.gen = [0] * num_blocks
        self.entry_of = {}   # (parent, parent_gen, tokens) -> block
        self.key_of = {}     # block -> its key

    def num_cached(self) -> int:
        return len(self.key_of)

    def _drop_entry(self, b: int) -> None:
        key = self.key_of.pop(b, None)
        if key is not None and self.entry_of.get(key) == b:
            del self.entry_of[key]

    def _fresh(self) -> int:
        b = self.free_queue.popleft()
        self._drop_entry(b)
        self.gen[b] += 1
        self.ref_cnt[b] = 1
        return b

    def allocate(self, n: int):
        if n > len(self.free_queue):
            return None
        return [self._fresh() for _ in range(n)]

    def cow(self, blk: int):
        if self.ref_cnt[blk] == 1:
            return blk, blk
        if not self.free_queue:
            raise PoolExhausted("no free block for copy-on-write")
        self.ref_cnt[blk] -= 1
        return blk, self._fresh()

    def _key(self, parent: int, tokens) -> tuple:
        return (parent, self.gen[parent] if parent >= 0 else 0, tuple(int(t) for t in tokens))

    def register(self, b: int, parent: int, tokens) -> None:
        self._drop_entry(b)
        key = self._key(parent, tokens)
        if key in self.entry_of:
            return
        self.entry_of[key] = b
        self.key_of[b] = key

    def allocate_prefix(self, tokens):
        """(blocks, cached_tokens) for a new sequence, or None when short."""
        B = self.block_size
        n = len(tokens)
        nblk, nfull = -(-n // B), n // B
        hits, parent = [], -1
        for k in range(nfull):
            b = self.entry_of.get(self._key(parent, tokens[k * B:(k + 1) * B]))
            if b is None:
                break
            hits.append(b)
            parent = b
        free_hits = sum(1 for b in hits if self.ref_cnt[b] == 0)
        if nblk - len(hits) > len(self.free_queue) - free_hits:
            return None
        for b in hits:
            if self.ref_cnt[b] == 0:
                self.free_queue.remove(b)
            self.ref_cnt[b] += 1
        blocks = list(hits)
        parent = hits[-1] if hits else -1
        for k in range(len(hits), nblk):
            b = self._fresh()
            blocks.append(b)
            if k < nfull:
                self.register(b, parent, tokens[k * B:(k + 1) * B])
            parent = b
        return blocks, len(hits) * B
