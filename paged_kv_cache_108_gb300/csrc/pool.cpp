// Host-side block pool: FIFO free queue + per-block reference counts.
//
// Semantics follow "Paged KV cache" (ai-infra-handbooks), class BlockPool
// (free queue initialised 0..n-1, take from the head, return to the tail,
// allocation refused without side effects when short) and "4.6 PagedAttention
// & KV-Cache Memory Management" (llm-stack-book), BlockManager.fork and
// cow_append (copy-on-write decided per block from its reference count).
//
//
// Prefix caching (optional, pa_pool_enable_prefix_cache): a full block can
// be found again by its content, so a later request whose prompt starts the
// same way shares the block instead of recomputing it.  The pages make
// full-block sharing the unit ("Paged KV cache", copy-on-write exercise:
// vLLM V1 shares only full blocks, each answer writes into its own block;
// "4.6 PagedAttention & KV-Cache Memory Management", section "Copy-on-write
// for shared prefixes": the same machinery generalizes to prefix caching
// across requests).  A block's identity is (parent block, the parent's
// generation, its B token ids); a block's generation advances whenever it
// is handed out fresh, which also drops its own entry, so an entry never
// outlives the content it names.  Freed cached blocks wait in the free
// queue (least recently freed at the head, evicted first) and leave it when
// a later prompt matches them.
//
// The free queue is a doubly linked list over block ids (O(1) removal of a
// matched free block); every block is either in the queue (ref count 0) or
// referenced (ref count >= 1).  Nothing allocates after creation except the
// prefix index.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"
#include "pa_host.h"

struct pa_pool {
  int32_t n = 0;
  std::vector<int32_t> ref;            // ref count per block
  std::vector<int32_t> prv, nxt;       // free-queue links (-1: none)
  int32_t head = -1, tail = -1;        // free queue ends
  int32_t count = 0;                   // number of free blocks
  // prefix cache
  int32_t bs = 0;                      // tokens per block; 0 while caching is off
  std::vector<uint32_t> gen;           // generation per block
  std::vector<char> cached;            // block holds a registered entry
  std::vector<uint64_t> key_hash;
  std::vector<int32_t> key_parent;
  std::vector<uint32_t> key_pgen;
  std::vector<int32_t> key_tokens;     // n * bs
  std::unordered_map<uint64_t, int32_t> index;
  int32_t ncached = 0;

  void push_tail(int32_t b) {
    prv[b] = tail;
    nxt[b] = -1;
    if (tail >= 0) nxt[tail] = b; else head = b;
    tail = b;
    ++count;
  }
  void unlink(int32_t b) {
    if (prv[b] >= 0) nxt[prv[b]] = nxt[b]; else head = nxt[b];
    if (nxt[b] >= 0) prv[nxt[b]] = prv[b]; else tail = prv[b];
    prv[b] = nxt[b] = -1;
    --count;
  }
  void evict(int32_t b) {
    if (!cached[b]) return;
    auto it = index.find(key_hash[b]);
    if (it != index.end() && it->second == b) index.erase(it);
    cached[b] = 0;
    --ncached;
  }
  // the queue head, handed out with new content
  int32_t take_fresh() {
    const int32_t b = head;
    unlink(b);
    evict(b);
    ++gen[b];
    ref[b] = 1;
    return b;
  }
  static uint64_t hash_key(int32_t parent, uint32_t pgen, const int32_t* tok, int32_t m) {
    uint64_t h = 1469598103934665603ull;  // FNV-1a, 64-bit
    auto mix = [&h](uint32_t v) {
      for (int i = 0; i < 4; ++i) {
        h ^= (v >> (8 * i)) & 0xffu;
        h *= 1099511628211ull;
      }
    };
    mix((uint32_t)parent);
    mix(pgen);
    for (int32_t i = 0; i < m; ++i) mix((uint32_t)tok[i]);
    return h;
  }
  int32_t lookup(int32_t parent, uint32_t pgen, const int32_t* tok) const {
    auto it = index.find(hash_key(parent, pgen, tok, bs));
    if (it == index.end()) return -1;
    const int32_t b = it->second;
    if (key_parent[b] != parent || key_pgen[b] != pgen ||
        std::memcmp(&key_tokens[(size_t)b * bs], tok, sizeof(int32_t) * bs) != 0)
      return -1;  // a different content with the same hash
    return b;
  }
  void enter(int32_t b, int32_t parent, const int32_t* tok) {
    evict(b);
    const uint32_t pgen = parent >= 0 ? gen[parent] : 0u;
    const uint64_t h = hash_key(parent, pgen, tok, bs);
    if (index.count(h)) return;  // that content (or a colliding one) is cached already
    index[h] = b;
    key_hash[b] = h;
    key_parent[b] = parent;
    key_pgen[b] = pgen;
    std::memcpy(&key_tokens[(size_t)b * bs], tok, sizeof(int32_t) * bs);
    cached[b] = 1;
    ++ncached;
  }
};

static pa_pool* make_pool(int32_t num_blocks, const int32_t* order) {
  if (num_blocks <= 0) {
    pa_set_error("pa_pool_create: num_blocks must be positive");
    return nullptr;
  }
  pa_pool* p = new (std::nothrow) pa_pool;
  if (!p) return nullptr;
  try {
    p->n = num_blocks;
    p->ref.assign(num_blocks, 0);
    p->prv.assign(num_blocks, -1);
    p->nxt.assign(num_blocks, -1);
    p->gen.assign(num_blocks, 0);
    p->cached.assign(num_blocks, 0);
  } catch (...) {
    delete p;
    return nullptr;
  }
  if (order) {
    std::vector<char> seen(num_blocks, 0);
    for (int32_t i = 0; i < num_blocks; ++i) {
      int32_t b = order[i];
      if (b < 0 || b >= num_blocks || seen[b]) {
        pa_set_error("pa_pool_create_ordered: order is not a permutation");
        delete p;
        return nullptr;
      }
      seen[b] = 1;
    }
  }
  for (int32_t i = 0; i < num_blocks; ++i) p->push_tail(order ? order[i] : i);
  return p;
}

extern "C" {

pa_pool* pa_pool_create(int32_t num_blocks) { return make_pool(num_blocks, nullptr); }

pa_pool* pa_pool_create_ordered(int32_t num_blocks, const int32_t* order) {
  if (!order) {
    pa_set_error("pa_pool_create_ordered: order is NULL");
    return nullptr;
  }
  return make_pool(num_blocks, order);
}

void pa_pool_destroy(pa_pool* pool) { delete pool; }

int32_t pa_pool_num_blocks(const pa_pool* pool) { return pool ? pool->n : 0; }

int32_t pa_pool_num_free(const pa_pool* pool) { return pool ? pool->count : 0; }

int32_t pa_pool_refcount(const pa_pool* pool, int32_t block) {
  if (!pool || block < 0 || block >= pool->n) return -1;
  return pool->ref[block];
}

int32_t pa_pool_free_order(const pa_pool* pool, int32_t* out, int32_t cap) {
  if (!pool) return 0;
  int32_t i = 0;
  for (int32_t b = pool->head; b >= 0; b = pool->nxt[b], ++i)
    if (i < cap) out[i] = b;
  return pool->count;
}

pa_status pa_pool_alloc(pa_pool* pool, int32_t n, int32_t* out_blocks) {
  if (!pool || n < 0 || (n > 0 && !out_blocks))
    return pa_fail(PA_ERR_INVALID, "pa_pool_alloc: bad arguments");
  if (n > pool->count)
    return pa_fail(PA_ERR_OOM, "pa_pool_alloc: not enough free blocks");
  for (int32_t i = 0; i < n; ++i) out_blocks[i] = pool->take_fresh();
  return PA_OK;
}

pa_status pa_pool_incref(pa_pool* pool, const int32_t* blocks, int32_t n) {
  if (!pool || n < 0 || (n > 0 && !blocks))
    return pa_fail(PA_ERR_INVALID, "pa_pool_incref: bad arguments");
  for (int32_t i = 0; i < n; ++i) {
    int32_t b = blocks[i];
    if (b < 0 || b >= pool->n || pool->ref[b] <= 0)
      return pa_fail(PA_ERR_INVALID, "pa_pool_incref: block outside the pool or free");
  }
  for (int32_t i = 0; i < n; ++i) ++pool->ref[blocks[i]];
  return PA_OK;
}

pa_status pa_pool_free(pa_pool* pool, const int32_t* blocks, int32_t n) {
  if (!pool || n < 0 || (n > 0 && !blocks))
    return pa_fail(PA_ERR_INVALID, "pa_pool_free: bad arguments");
  // validate first (counting repeats) so a bad list leaves the pool unchanged
  std::vector<int32_t> dec;
  try {
    dec.assign(pool->n, 0);
  } catch (...) {
    return pa_fail(PA_ERR_OOM, "pa_pool_free: host allocation failed");
  }
  for (int32_t i = 0; i < n; ++i) {
    int32_t b = blocks[i];
    if (b < 0 || b >= pool->n || ++dec[b] > pool->ref[b])
      return pa_fail(PA_ERR_INVALID, "pa_pool_free: block outside the pool or released too often");
  }
  for (int32_t i = 0; i < n; ++i) {
    int32_t b = blocks[i];
    if (--pool->ref[b] == 0) pool->push_tail(b);
  }
  return PA_OK;
}

pa_status pa_pool_cow(pa_pool* pool, int32_t block, int32_t* out_dst) {
  if (!pool || !out_dst || block < 0 || block >= pool->n || pool->ref[block] <= 0)
    return pa_fail(PA_ERR_INVALID, "pa_pool_cow: block outside the pool or free");
  if (pool->ref[block] == 1) {
    *out_dst = block;
    return PA_OK;
  }
  if (pool->count == 0) return pa_fail(PA_ERR_OOM, "pa_pool_cow: no free block");
  const int32_t fresh = pool->take_fresh();
  --pool->ref[block];
  *out_dst = fresh;
  return PA_OK;
}

pa_status pa_pool_enable_prefix_cache(pa_pool* pool, int32_t block_size) {
  if (!pool || block_size <= 0)
    return pa_fail(PA_ERR_INVALID, "pa_pool_enable_prefix_cache: bad arguments");
  if (pool->bs == block_size) return PA_OK;
  if (pool->bs != 0)
    return pa_fail(PA_ERR_INVALID, "pa_pool_enable_prefix_cache: already on with another block size");
  try {
    pool->key_hash.assign(pool->n, 0);
    pool->key_parent.assign(pool->n, -1);
    pool->key_pgen.assign(pool->n, 0);
    pool->key_tokens.assign((size_t)pool->n * block_size, 0);
    pool->index.reserve((size_t)pool->n);
  } catch (...) {
    return pa_fail(PA_ERR_OOM, "pa_pool_enable_prefix_cache: host allocation failed");
  }
  pool->bs = block_size;
  return PA_OK;
}

int32_t pa_pool_num_cached(const pa_pool* pool) { return pool ? pool->ncached : 0; }

pa_status pa_pool_alloc_prefix(pa_pool* pool, const int32_t* tokens, int32_t num_tokens,
                               int32_t* out_blocks, int32_t* num_cached_tokens) {
  if (!pool || num_tokens < 0 || (num_tokens > 0 && (!tokens || !out_blocks)) ||
      !num_cached_tokens)
    return pa_fail(PA_ERR_INVALID, "pa_pool_alloc_prefix: bad arguments");
  if (pool->bs == 0)
    return pa_fail(PA_ERR_INVALID, "pa_pool_alloc_prefix: prefix caching is off");
  const int32_t B = pool->bs;
  const int32_t nblk = (num_tokens + B - 1) / B, nfull = num_tokens / B;
  // leading full blocks already cached, each keyed by its parent's identity
  int32_t hits = 0, free_hits = 0, parent = -1;
  uint32_t pgen = 0;
  for (int32_t k = 0; k < nfull; ++k) {
    const int32_t b = pool->lookup(parent, pgen, tokens + (size_t)k * B);
    if (b < 0) break;
    out_blocks[k] = b;
    if (pool->ref[b] == 0) ++free_hits;
    parent = b;
    pgen = pool->gen[b];
    ++hits;
  }
  if (nblk - hits > pool->count - free_hits)
    return pa_fail(PA_ERR_OOM, "pa_pool_alloc_prefix: not enough free blocks");
  for (int32_t k = 0; k < hits; ++k) {
    const int32_t b = out_blocks[k];
    if (pool->ref[b] == 0) pool->unlink(b);
    ++pool->ref[b];
  }
  parent = hits > 0 ? out_blocks[hits - 1] : -1;
  for (int32_t k = hits; k < nblk; ++k) {
    const int32_t b = pool->take_fresh();
    out_blocks[k] = b;
    if (k < nfull) pool->enter(b, parent, tokens + (size_t)k * B);
    parent = b;
  }
  *num_cached_tokens = hits * B;
  return PA_OK;
}

pa_status pa_pool_register_block(pa_pool* pool, int32_t block, int32_t parent,
                                 const int32_t* tokens) {
  if (!pool || !tokens || block < 0 || block >= pool->n || pool->ref[block] <= 0 ||
      parent < -1 || parent >= pool->n || parent == block)
    return pa_fail(PA_ERR_INVALID, "pa_pool_register_block: bad arguments");
  if (pool->bs == 0)
    return pa_fail(PA_ERR_INVALID, "pa_pool_register_block: prefix caching is off");
  pool->enter(block, parent, tokens);
  return PA_OK;
}

pa_status pa_slot_mapping(const int32_t* block_tables, int32_t num_seqs,
                          int32_t max_blocks_per_seq, int32_t block_size,
                          const int32_t* token_seq, const int32_t* token_pos,
                          int32_t num_tokens, int32_t* slot_mapping) {
  if (num_tokens < 0 || block_size <= 0 || max_blocks_per_seq < 0 || num_seqs < 0)
    return pa_fail(PA_ERR_INVALID, "pa_slot_mapping: bad sizes");
  if (num_tokens == 0) return PA_OK;
  if (!block_tables || !token_pos || !slot_mapping)
    return pa_fail(PA_ERR_INVALID, "pa_slot_mapping: NULL array");
  for (int32_t i = 0; i < num_tokens; ++i) {
    int32_t s = token_seq ? token_seq[i] : i;
    int32_t pos = token_pos[i];
    if (s < 0 || s >= num_seqs || pos < 0 || pos / block_size >= max_blocks_per_seq)
      return pa_fail(PA_ERR_INVALID, "pa_slot_mapping: sequence or position out of range");
    int64_t phys = block_tables[(int64_t)s * max_blocks_per_seq + pos / block_size];
    int64_t slot = phys * block_size + pos % block_size;
    if (phys < 0 || slot > INT32_MAX)
      return pa_fail(PA_ERR_INVALID, "pa_slot_mapping: block id out of range");
    slot_mapping[i] = (int32_t)slot;
  }
  return PA_OK;
}

}  // extern "C"
