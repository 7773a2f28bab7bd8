// Host-side block pool: FIFO free queue + per-block reference counts.
//
// Semantics follow "Paged KV cache" (ai-infra-handbooks), class BlockPool
// (free queue initialised 0..n-1, take from the head, return to the tail,
// allocation refused without side effects when short) and "4.6 PagedAttention
// & KV-Cache Memory Management" (llm-stack-book), BlockManager.fork and
// cow_append (copy-on-write decided per block from its reference count).
//
// The free queue is a fixed-capacity ring buffer: every block is either in
// the queue (ref count 0) or referenced (ref count >= 1), so the queue never
// holds more than num_blocks ids and no operation allocates after creation.
#include <cstdint>
#include <cstdlib>
#include <new>
#include <vector>

#include "pa.h"
#include "pa_host.h"

struct pa_pool {
  int32_t n = 0;
  std::vector<int32_t> ref;   // ref count per block
  std::vector<int32_t> ring;  // free queue storage, capacity n
  int32_t head = 0;           // index of the queue head in ring
  int32_t count = 0;          // number of free blocks

  void push_tail(int32_t b) {
    ring[(head + count) % n] = b;
    ++count;
  }
  int32_t pop_head() {
    int32_t b = ring[head];
    head = (head + 1) % n;
    --count;
    return b;
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
    p->ring.assign(num_blocks, 0);
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
  for (int32_t i = 0; i < pool->count && i < cap; ++i)
    out[i] = pool->ring[(pool->head + i) % pool->n];
  return pool->count;
}

pa_status pa_pool_alloc(pa_pool* pool, int32_t n, int32_t* out_blocks) {
  if (!pool || n < 0 || (n > 0 && !out_blocks))
    return pa_fail(PA_ERR_INVALID, "pa_pool_alloc: bad arguments");
  if (n > pool->count)
    return pa_fail(PA_ERR_OOM, "pa_pool_alloc: not enough free blocks");
  for (int32_t i = 0; i < n; ++i) {
    int32_t b = pool->pop_head();
    pool->ref[b] = 1;
    out_blocks[i] = b;
  }
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
  int32_t fresh = pool->pop_head();
  pool->ref[fresh] = 1;
  --pool->ref[block];
  *out_dst = fresh;
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
