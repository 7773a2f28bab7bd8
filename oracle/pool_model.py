"""Pure-Python model of the block pool and block tables -- TEST INFRASTRUCTURE.

Only tests, the smoke check and the benchmark's CPU legs use this module.

The rules it states, and where the pages give them:

* Pool ("Paged KV cache" (ai-infra-handbooks), section "Implementation",
  the block pool; its doctest under "Block tables and slot mapping"):
  R1  every block id starts free; the free ids wait in one queue, in the
      order 0..n-1 unless a start order is given;
  R2  a request for n blocks is granted only whole: with fewer than n free it
      is refused and nothing changes; otherwise the n ids at the front of the
      queue leave it, in queue order, each with exactly one holder;
  R3  a release takes one holder from each listed block; a block left with no
      holder joins the back of the queue.
* Tables and growth ("4.6 PagedAttention & KV-Cache Memory Management"
  (llm-stack-book), section "Block Tables, the Allocator & Copy-on-Write"):
  a prompt of n tokens takes ceil(n / B) blocks; a sequence takes one more
  block exactly when the position about to be written is a multiple of B;
  position p lives at slot table[p // B] * B + p % B.
* Fork and copy-on-write (same page, section "Copy-on-write for shared
  prefixes"): a fork shares every block (one more holder each); a write
  into a block that has other holders first moves the writer to a fresh
  block (R2 with n = 1), drops the writer's hold on the old one, and reports
  (old, new) so the device copies the contents; a block with one holder is
  written where it is.
* Prefix caching across requests (``PrefixCachePoolModel``): "Paged KV
  cache", Exercises (the copy-on-write answer: vLLM V1 shares only full
  blocks, so every request writes in a block of its own); "4.6 ...",
  section "Copy-on-write for shared prefixes" (the same sharing serves
  requests that repeat a prompt).  The pages do not say how a full block is
  recognised.  Reading taken: a full block's identity is (its parent block,
  the parent's generation, its B token ids), with parent -1 for a prompt's
  first block; a block's generation grows each time it is handed out fresh,
  which also forgets its identity; a cached block whose holders are all gone
  stays in the free queue, keeps its identity, and leaves the queue from
  wherever it sits when a later prompt matches it.

Readings where the pages disagree: the queue is first-in first-out (the
handbook's printed ``[5, 6, 7, 0]``), not the llm-stack-book's take from the
end; a short pool refuses the whole request instead of raising after a
partial hand-out.
"""
from __future__ import annotations


class PoolExhausted(Exception):
    pass


class BlockPoolModel:
    """Rules R1-R3 plus fork (``incref``) and copy-on-write (``cow``)."""

    def __init__(self, num_blocks: int, free_order=None):
        self.num_blocks = num_blocks
        start = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(start) != list(range(num_blocks)):
            raise ValueError("the start order must list every block once")
        self._waiting = start                   # R1: front of the queue first
        self._holders = [0] * num_blocks

    # -- queries
    def num_free(self) -> int:
        return len(self._waiting)

    def refcount(self, blk: int) -> int:
        return self._holders[blk]

    def free_order(self):
        return list(self._waiting)

    # -- R2
    def _take_front(self, n: int):
        granted, self._waiting = self._waiting[:n], self._waiting[n:]
        for b in granted:
            self._holders[b] = 1
        return granted

    def allocate(self, n: int):
        """n blocks from the front of the queue, or None (and no change)."""
        return self._take_front(n) if n <= len(self._waiting) else None

    # -- R3 and fork
    def free(self, blocks) -> None:
        for b in blocks:
            self._holders[b] -= 1
            if not self._holders[b]:
                self._waiting.append(b)

    def incref(self, blocks) -> None:
        for b in blocks:
            self._holders[b] += 1

    def cow(self, blk: int):
        """(src, dst) for a write into ``blk``; dst == src when unshared."""
        if self._holders[blk] == 1:
            return blk, blk
        fresh = self.allocate(1)
        if fresh is None:
            raise PoolExhausted("no free block for copy-on-write")
        self._holders[blk] -= 1
        return blk, fresh[0]


def slot_of(table, pos: int, block_size: int) -> int:
    """Flat pool slot of logical position ``pos``."""
    return table[pos // block_size] * block_size + pos % block_size


class SequenceTablesModel:
    """Per-sequence block tables kept on top of a ``BlockPoolModel``."""

    def __init__(self, pool: BlockPoolModel, block_size: int):
        self.pool = pool
        self.block_size = block_size
        self.tables = {}

    def allocate(self, seq, num_tokens: int) -> None:
        need = -(-num_tokens // self.block_size)
        got = self.pool.allocate(need)
        if got is None:
            raise PoolExhausted(f"need {need} blocks, {self.pool.num_free()} free")
        self.tables[seq] = got

    def append_token(self, seq, cur_len: int) -> None:
        """Before position ``cur_len`` is written: a new block if it opens one."""
        if cur_len % self.block_size:
            return
        got = self.pool.allocate(1)
        if got is None:
            raise PoolExhausted("no free block to grow the sequence")
        self.tables[seq] += got

    def fork(self, parent, child) -> None:
        self.tables[child] = self.tables[parent][:]
        self.pool.incref(self.tables[child])

    def cow_for_write(self, seq, pos: int):
        """Make the block holding ``pos`` the writer's own; return (src, dst)."""
        table = self.tables[seq]
        src, dst = self.pool.cow(table[pos // self.block_size])
        table[pos // self.block_size] = dst
        return src, dst

    def slot_index(self, seq, pos: int) -> int:
        return slot_of(self.tables[seq], pos, self.block_size)

    def free_seq(self, seq) -> None:
        self.pool.free(self.tables.pop(seq))


class PrefixCachePoolModel(BlockPoolModel):
    """``BlockPoolModel`` with full-block prefix caching (module notes)."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        super().__init__(num_blocks, free_order)
        self.block_size = block_size
        self._generation = [0] * num_blocks
        self._by_identity = {}   # identity -> the block holding it
        self._identity = {}      # block -> its identity, while it has one

    def num_cached(self) -> int:
        return len(self._identity)

    def _forget(self, b: int) -> None:
        ident = self._identity.pop(b, None)
        if ident is not None and self._by_identity.get(ident) == b:
            del self._by_identity[ident]

    def _take_front(self, n: int):
        granted = super()._take_front(n)
        for b in granted:                     # handed out fresh: a new generation
            self._forget(b)
            self._generation[b] += 1
        return granted

    def _identity_of(self, parent: int, tokens) -> tuple:
        gen = self._generation[parent] if parent >= 0 else 0
        return parent, gen, tuple(int(t) for t in tokens)

    def register_block(self, b: int, parent: int, tokens) -> None:
        """Give block ``b`` the identity (parent, parent's generation, tokens);
        the first block registered under an identity keeps it."""
        if len(tokens) != self.block_size:
            raise ValueError("a registered block holds exactly block_size tokens")
        self._forget(b)
        ident = self._identity_of(parent, tokens)
        if ident not in self._by_identity:
            self._by_identity[ident] = b
            self._identity[b] = ident

    def allocate_prefix(self, tokens):
        """(blocks, cached_tokens) for a new sequence with prompt ``tokens``,
        or None (and no change) when the pool is short."""
        B = self.block_size
        tokens = list(tokens)
        full, total = len(tokens) // B, -(-len(tokens) // B)
        # 1. the longest chain of full blocks already cached for this prompt
        matched, parent = [], -1
        while len(matched) < full:
            k = len(matched)
            b = self._by_identity.get(self._identity_of(parent, tokens[k * B:(k + 1) * B]))
            if b is None:
                break
            matched.append(b)
            parent = b
        # 2. all or nothing: matched blocks that sit in the queue are not
        #    available to serve the fresh part
        idle = [b for b in matched if self._holders[b] == 0]
        if total - len(matched) > len(self._waiting) - len(idle):
            return None
        for b in idle:
            self._waiting.remove(b)
        self.incref(matched)
        # 3. fresh blocks for the rest; each new full block gets its identity
        blocks = matched + self._take_front(total - len(matched))
        for k in range(len(matched), full):
            self.register_block(blocks[k], blocks[k - 1] if k else -1,
                                tokens[k * B:(k + 1) * B])
        return blocks, len(matched) * B
