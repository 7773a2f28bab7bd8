/*
 * pa.h -- C ABI of the GB300-native paged-KV decode library (libpa.so).
 *
 * The operations are those of vLLM-style PagedAttention as described on the
 * pages "4.6 PagedAttention & KV-Cache Memory Management" (llm-stack-book,
 * cited below as [LSB]), "Paged KV cache" (ai-infra-handbooks, [PKV]),
 * "Allocate the Cache: Blocks, Waste, and PagedAttention" (int8ai.com, [ATC])
 * and "PagedAttention - Explained" (mohdvasim.com, [PAE]).
 *
 * Conventions shared by every device entry point
 *  - Device pointers are raw CUDA device addresses; the caller owns every
 *    buffer (including the decode workspace) and keeps it alive until the
 *    work queued on `stream` has finished.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  The library allocates no device memory and
 *    performs no host<->device synchronisation or copy.
 *  - Host-visible arguments are validated before anything is launched; on a
 *    failed check nothing is launched and PA_ERR_INVALID or
 *    PA_ERR_UNSUPPORTED is returned.  A failed launch returns PA_ERR_CUDA.
 *    pa_last_error() gives a one-line description of the last failure on
 *    the calling thread.
 *  - Contents of device buffers (block ids, slots, context lengths) are not
 *    visible to the host and are not validated there.  Kernels skip any
 *    block id outside [0, num_blocks) or slot outside [0, num_blocks *
 *    block_size) instead of touching memory out of bounds; the affected
 *    outputs are then unspecified.
 *
 * Cache layout (per layer, one tensor for K and one for V):
 *    [num_blocks, block_size, num_kv_heads, head_dim], row-major, elements
 *    bf16 or fp8-e4m3.  [LSB] "Block Tables, the Allocator & Copy-on-Write"
 *    (BlockManager docstring); [PKV] "Implementation" (PagedKVCache).
 *    Token slot s = phys_block * block_size + offset addresses row
 *    s of the flat view [num_blocks * block_size, num_kv_heads, head_dim].
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID = 1,     /* a host-visible argument is malformed */
  PA_ERR_OOM = 2,         /* the block pool has too few free blocks */
  PA_ERR_CUDA = 3,        /* a CUDA launch or driver call failed */
  PA_ERR_UNSUPPORTED = 4  /* valid, but a shape this build has no kernel for */
} pa_status;

typedef enum { PA_KV_BF16 = 0, PA_KV_FP8_E4M3 = 1 } pa_kv_dtype;

/* Shape of one K (or V) cache tensor.  Supported: head_dim in {64, 128};
 * block_size >= 1; num_kv_heads >= 1; dtype a pa_kv_dtype. */
typedef struct {
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t dtype; /* pa_kv_dtype */
} pa_cache_desc;

/* cudaStream_t without the CUDA headers. */
typedef struct CUstream_st* pa_stream_t;

/* ------------------------------------------------------------------------
 * pa_reshape_and_cache -- slot-mapped cache write.
 * [PKV] "Implementation", PagedKVCache.write: token i's K/V go to slot
 * slot_mapping[i] of the flat pool; [LSB] "From Python bookkeeping to the
 * tensors the kernel actually takes" (one index copy over the flat pool).
 *
 *  key, value    device, [num_tokens, num_kv_heads, head_dim] bf16,
 *                contiguous, 16-byte aligned.
 *  k_cache, v_cache  device, layout above; written in place.
 *  slot_mapping  device, [num_tokens] int32.  A negative slot skips the
 *                token (padding).
 *  k_scale, v_scale  device float scalars for PA_KV_FP8_E4M3 (the cache
 *                holds e4m3(x / scale), x / scale in IEEE fp32, rounded to
 *                nearest-even and saturated to +-448); must be NULL for bf16.
 *  num_tokens == 0 is valid and launches nothing.
 * ---------------------------------------------------------------------- */
pa_status pa_reshape_and_cache(const void* key, const void* value,
                               void* k_cache, void* v_cache,
                               pa_cache_desc cache,
                               const int32_t* slot_mapping, int32_t num_tokens,
                               const float* k_scale, const float* v_scale,
                               pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_decode_workspace_size -- bytes of scratch pa_decode needs for a call
 * with these sizes (split-K partial results; 0 if none can be needed).
 * Any workspace at least this large is accepted.
 * ---------------------------------------------------------------------- */
size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_heads,
                                int32_t head_dim, int32_t max_blocks_per_seq,
                                int32_t block_size);

/* Workspace bytes for pa_decode_ex with an explicit split-K partition
 * length (a power of two in [64, 65536]); 0 means the automatic choice. */
size_t pa_decode_workspace_size_ex(int32_t num_seqs, int32_t num_heads,
                                   int32_t head_dim,
                                   int32_t max_blocks_per_seq,
                                   int32_t block_size,
                                   int32_t partition_tokens);

/* Tuning knobs of pa_decode_ex.  Zero means "choose automatically".
 *  kernel 1: SIMT kernel (CUDA cores, cp.async ring, fixed split-K
 *            partitions of partition_tokens, separate combine kernel); serves
 *            every supported shape.
 *  kernel 2: tensor-core kernel (tcgen05 MMA, TMA loads -- 16-byte cp.async
 *            gathers for block_size below 8 --, persistent CTAs that each
 *            stream an equal share of 128-token (bf16) or 256-token (e4m3)
 *            chunks, in-kernel merge of split units); needs head_dim 128 and
 *            at most 1024 sequences, else PA_ERR_UNSUPPORTED.  For an e4m3 cache the MMAs take the cache
 *            bytes as they are (kind::f8f6f4); q and the softmax weights are
 *            split into e4m3 parts (three for q, two for the weights) whose
 *            sum keeps them to about 2^-12 and 2^-8 relative.
 *            partition_tokens is ignored.  It sets workspace word 0 (int32)
 *            to a nonzero code if one of its bounded internal waits expired
 *            or a block id was out of range; the library never clears that
 *            word, so a caller that wants to check it zeroes it first.
 *  kernel 3: head-packed tensor-core kernel: one TMA copy moves a block's
 *            rows for 8 KV heads (16 when the GQA group is 1), the MMA
 *            columns are those heads' query heads, and each column keeps only
 *            its own KV head's rows.  Blocks smaller than 128 / heads per
 *            tile tokens are copied whole (every token's rows of those heads,
 *            1 to 4 KiB per token).  An e4m3 cache is read as it is, with q
 *            and the softmax weights split into e4m3 parts as in kernel 2.
 *            Needs head_dim 128, GQA group 1, 2 or 4, num_kv_heads a
 *            multiple of those heads per tile, at most 1024 sequences, one
 *            token per sequence, else PA_ERR_UNSUPPORTED.  Error word as
 *            kernel 2.
 *  kernel 0: kernel 3 where it applies and either the blocks hold fewer
 *            than 8 tokens or (bf16 cache) the batch has many units (per
 *            unit: a sequence and its 8 or 16 KV heads; at least twice the
 *            SM count, or half of it for GQA group 1); else kernel 2 where it
 *            applies (below 8 tokens per block only for several tokens per
 *            sequence: its gathered loads stream slower than the SIMT
 *            kernel); else kernel 1. */
typedef struct {
  int32_t partition_tokens; /* split-K partition length: power of two >= 64 */
  int32_t kernel;           /* 0 auto, 1 SIMT, 2 tensor-core, 3 head-packed tensor-core */
} pa_decode_opts;

/* ------------------------------------------------------------------------
 * pa_decode -- decode-time paged attention, one query token per sequence.
 * [LSB] "The PagedAttention Kernel" (online softmax over the sequence's
 * blocks, GQA head map h -> h / G; a CTA per (sequence, KV head));
 * [LSB] "Performance considerations" (split-K over the sequence, as in
 * PagedAttention v2); [PKV] "Paged attention" (block_tables, seq_lens).
 *
 *  out           device, [num_seqs, num_heads, head_dim] bf16 (written):
 *                out[i,h] = softmax(scale * q[i,h] . K_i[:, h/G]^T) V_i[:, h/G]
 *                over the first context_lens[i] tokens of sequence i, in
 *                fp32, rounded to nearest-even bf16.  context_lens[i] == 0
 *                gives a zero row.
 *  q             device, [num_seqs, num_heads, head_dim] bf16, contiguous.
 *  block_tables  device, [num_seqs, max_blocks_per_seq] int32; entry j of
 *                row i is the physical block of logical block j.  Entries
 *                at or past ceil(context_lens[i] / block_size) are not read.
 *  context_lens  device, [num_seqs] int32: valid tokens of each sequence
 *                after this step's write (so pa_reshape_and_cache must run
 *                first on the same stream); at most
 *                max_blocks_per_seq * block_size.
 *  num_heads     query heads; a multiple of cache.num_kv_heads, with
 *                G = num_heads / num_kv_heads in {1, 2, 4, 8}.
 *  scale         logit scale (typically 1/sqrt(head_dim)).
 *  k_scale, v_scale  device float scalars for fp8 caches, NULL for bf16.
 *  workspace     device scratch of at least pa_decode_workspace_size(...)
 *                bytes, 256-byte aligned; its contents need no
 *                initialisation and are clobbered.  One workspace may serve
 *                successive calls of different shapes on one stream; calls
 *                that share it must not overlap on the GPU.
 * ---------------------------------------------------------------------- */
pa_status pa_decode(void* out, const void* q, const void* k_cache,
                    const void* v_cache, pa_cache_desc cache,
                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* context_lens, int32_t num_seqs,
                    int32_t num_heads, float scale, const float* k_scale,
                    const float* v_scale, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream);

/* pa_decode with explicit tuning knobs (opts may be NULL). */
pa_status pa_decode_ex(void* out, const void* q, const void* k_cache,
                       const void* v_cache, pa_cache_desc cache,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* context_lens, int32_t num_seqs,
                       int32_t num_heads, float scale, const float* k_scale,
                       const float* v_scale, void* workspace,
                       size_t workspace_bytes, const pa_decode_opts* opts,
                       pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_write_and_decode -- one decode step: pa_reshape_and_cache of the new
 * tokens followed by pa_decode, in one call.  [LSB] "Putting It Together: A
 * Minimal Paged Serving Loop" (serve_step: write the token's K/V at its
 * slot, then attend over the sequence's blocks).
 *
 * Arguments are those of the two calls (num_tokens new tokens; decode with
 * the automatic kernel choice).  Because the library itself launches the
 * write just before the decode, the tensor-core decode kernel starts while
 * the write still runs and reads lengths, block tables and q at once; it
 * waits for the write only before its first cache read.  Results are those
 * of the two separate calls.
 * ---------------------------------------------------------------------- */
pa_status pa_write_and_decode(const void* key, const void* value,
                              const int32_t* slot_mapping, int32_t num_tokens,
                              void* out, const void* q, void* k_cache,
                              void* v_cache, pa_cache_desc cache,
                              const int32_t* block_tables,
                              int32_t max_blocks_per_seq,
                              const int32_t* context_lens, int32_t num_seqs,
                              int32_t num_heads, float scale,
                              const float* k_scale, const float* v_scale,
                              void* workspace, size_t workspace_bytes,
                              pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_decode_noalloc -- pa_decode for callers that cannot provide scratch.
 * The source pages have no counterpart to this entry point; it is a
 * library convenience.
 *
 * pa_decode needs a caller-owned workspace for its split-K partial results.
 * Some callers cannot hand out device memory at the call site: a plugin
 * whose host application owns every device allocation, or a
 * latency-critical serving loop that must not call cudaMalloc because
 * cudaMalloc can synchronise the device.  This variant takes the same
 * arguments minus the workspace and keeps the partials in a fixed array of
 * PA_DECODE_NOALLOC_SCRATCH_BYTES bytes compiled into the library (every GPU
 * that loads the library holds it until the process exits).  It allocates
 * nothing and calls no allocating routine.
 *
 *  - Output and numerics are those of pa_decode with the automatic kernel
 *    choice.  When that choice is the SIMT kernel (head_dim other than 128,
 *    or a head layout the tensor-core kernels do not take), its split-K
 *    partition length is the shortest
 *    power of two from 256 tokens whose partials fit; the tensor-core
 *    kernels ignore partition lengths and use their fixed per-CTA slots.
 *  - PA_ERR_UNSUPPORTED, with nothing launched, when the sizes need more
 *    scratch than the array holds even with 65536-token partitions; use
 *    pa_decode with a workspace then.
 *  - Device-side faults the tensor-core kernels detect (an expired bounded
 *    wait, an out-of-range block id, which they replace by block 0) set a
 *    status word kept in the array.  Decode calls never clear it; read and
 *    clear it with pa_decode_noalloc_error.  The SIMT kernel reports
 *    nothing there.
 *  - The first call on each device looks up the array's device address
 *    (with that device current) and caches it; make that first call before
 *    any stream capture begins.
 *  - All calls on a device share the one array, which keeps the last call's
 *    contents (nothing in it has to start at zero).  Calls whose GPU work
 *    overlaps -- e.g. issued on two streams without ordering -- race on the
 *    array and give wrong results: order them on one stream.
 * ---------------------------------------------------------------------- */
#define PA_DECODE_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
pa_status pa_decode_noalloc(void* out, const void* q, const void* k_cache,
                            const void* v_cache, pa_cache_desc cache,
                            const int32_t* block_tables,
                            int32_t max_blocks_per_seq,
                            const int32_t* context_lens, int32_t num_seqs,
                            int32_t num_heads, float scale,
                            const float* k_scale, const float* v_scale,
                            pa_stream_t stream);

/* pa_decode_noalloc_error -- enqueue on `stream` a copy of the current
 * device's pa_decode_noalloc status word into *code, then clear the word.
 * 0 means no pa_decode_noalloc call on this device reported a device-side
 * fault since the word was last read; a nonzero value is the code of such a
 * fault: 3 for a block id outside the pool, any other value for a bounded
 * wait that expired (the value names the wait).
 * `code` may be device memory or host memory (page-locked for the copy to
 * stay asynchronous); its value is valid once the stream has reached the
 * copy.  Like pa_decode_noalloc, it allocates nothing.  PA_ERR_INVALID for
 * a NULL code, PA_ERR_CUDA if the copy or the clear cannot be enqueued. */
pa_status pa_decode_noalloc_error(int32_t* code, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_copy_blocks -- device side of copy-on-write: for each (src, dst) pair,
 * k_cache[dst] = k_cache[src] and v_cache[dst] = v_cache[src], bit-exact.
 * [LSB] "Copy-on-write for shared prefixes" (cow_append returns (src, dst);
 * "kernel copies src->dst, then writes").
 *
 *  block_pairs   device, [num_pairs, 2] int32 (src, dst).  Pairs must not
 *                chain (no dst of one pair is the src of another) and no dst
 *                may repeat; the copies of one call run concurrently.
 *  num_pairs == 0 is valid and launches nothing.
 * ---------------------------------------------------------------------- */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, pa_cache_desc cache,
                         const int32_t* block_pairs, int32_t num_pairs,
                         pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_slot_mapping -- host-side slot computation for a step's new tokens.
 * slot = table[pos / block_size] * block_size + pos % block_size.
 * [LSB] BlockManager.slot_index; [PKV] slot_mapping_for; [ATC] "How the
 * Block Table Works"; [PAE] "The Custom CUDA Kernel Overview".
 *
 *  block_tables  host, [num_seqs, max_blocks_per_seq] int32.
 *  token_seq     host, [num_tokens] sequence index of each token, or NULL
 *                meaning token i belongs to sequence i (decode).
 *  token_pos     host, [num_tokens] logical position of each token.
 *  slot_mapping  host, [num_tokens] int32 (written).
 *  Returns PA_ERR_INVALID if a position or sequence index is out of range.
 * ---------------------------------------------------------------------- */
pa_status pa_slot_mapping(const int32_t* block_tables, int32_t num_seqs,
                          int32_t max_blocks_per_seq, int32_t block_size,
                          const int32_t* token_seq, const int32_t* token_pos,
                          int32_t num_tokens, int32_t* slot_mapping);

/* ------------------------------------------------------------------------
 * pa_varlen_attention -- paged attention for a step whose requests add any
 * number of new tokens (multi-token decode, chunked prefill, full prefill).
 * [PKV] "Paged attention" (paged_attention, query_start_loc): request i's
 * new tokens are q[qsl[i]:qsl[i+1]], the last num_new tokens of its context
 * of seq_lens[i] tokens; new token j sits at position seq_len - num_new + j
 * and attends causally to positions 0..seq_len - num_new + j, query head h
 * to KV head h / (num_heads / num_kv_heads).  Each new token is computed as
 * a decode over the first seq_len - num_new + j + 1 tokens of its request
 * (one virtual sequence per token, the decode kernels of pa_decode), so a
 * request's context is read once per new token: efficient for a few new
 * tokens per request, bandwidth-heavy for long prefill chunks.
 *
 *  out, q            device, [num_tokens, num_heads, head_dim] bf16.
 *  block_tables      device, [num_seqs, max_blocks_per_seq] int32.
 *  seq_lens          device, [num_seqs] int32: context length after this
 *                    step's write (the new tokens' K/V are already cached).
 *  query_start_loc   device, [num_seqs + 1] int32, non-decreasing, from 0 to
 *                    num_tokens (cu_seqlens_q).  A request whose num_new
 *                    exceeds its seq_len gets zero output rows.
 *  workspace         device, >= pa_varlen_workspace_size(...) bytes, 256-byte
 *                    aligned (expanded tables, lengths, decode scratch).
 *  Other arguments as pa_decode.  At most 65535 new tokens per call.
 * ---------------------------------------------------------------------- */
size_t pa_varlen_workspace_size(int32_t num_tokens, int32_t num_heads, int32_t head_dim,
                                int32_t max_blocks_per_seq, int32_t block_size);
pa_status pa_varlen_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                              pa_cache_desc cache, const int32_t* block_tables,
                              int32_t max_blocks_per_seq, const int32_t* seq_lens,
                              const int32_t* query_start_loc, int32_t num_seqs,
                              int32_t num_tokens, int32_t num_heads, float scale,
                              const float* k_scale, const float* v_scale, void* workspace,
                              size_t workspace_bytes, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_varlen_attention_ex -- pa_varlen_attention with the method chosen.
 *  method 1: one decode per new token, as described above (every shape
 *            pa_decode serves; reads a request's context once per token).
 *  method 2: tensor-core prefill tiles: a work item is a request's tile of
 *            128 / G new tokens for one KV head (G = the GQA group), its 128
 *            (token, query head) rows on the MMA's M side against 128-key
 *            chunks of the paged context, online softmax with one thread per
 *            row and O kept in tensor memory; the context is read once per
 *            tile.  For an e4m3 cache the MMAs take the cache bytes as they
 *            are (kind::f8f6f4): each q row is split into three e4m3 parts
 *            under its own power-of-two scale and the weights into two, and
 *            P V is computed as its transpose.  Needs head_dim 128, G in
 *            {1, 2, 4, 8}, block_size >= 8, at most 256 requests and
 *            scale > 0, else PA_ERR_UNSUPPORTED.  Sets workspace word 0 (int32) to a nonzero
 *            code if a bounded internal wait expired or a block id was out of
 *            range; the library never clears it.  Workspace word 1 is the
 *            tiles' work counter, zeroed on `stream` before each launch (an
 *            asynchronous memset, captured with the kernel in a graph).
 *  method 0: where method 2 applies: method 2 for every request when the
 *            step adds at least 16 new tokens per request on average;
 *            otherwise, when it adds 16 or more in all, method 2 for the
 *            requests adding 16 or more and method 1 for the others (two
 *            launches on `stream`; word 0 is then the tiles' error word,
 *            zeroed by the call before the tiles run); else method 1.
 *  Other arguments as pa_varlen_attention.
 * ---------------------------------------------------------------------- */
pa_status pa_varlen_attention_ex(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, pa_cache_desc cache,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* seq_lens, const int32_t* query_start_loc,
                                 int32_t num_seqs, int32_t num_tokens, int32_t num_heads,
                                 float scale, const float* k_scale, const float* v_scale,
                                 int32_t method, void* workspace, size_t workspace_bytes,
                                 pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_decode_multi -- pa_varlen_attention for the common case in which every
 * request adds the same number of tokens (multi-token / speculative decode):
 * q and out are [num_seqs * tokens_per_seq, num_heads, head_dim], request
 * i's tokens at rows i * tokens_per_seq + j, the last tokens_per_seq
 * positions of its context_lens[i]-token context, each causal as in
 * pa_varlen_attention ([PKV] "Paged attention").  When group x
 * tokens_per_seq fits the tensor-core kernel's columns (16 for bf16, 8 for
 * e4m3; powers of two) one pass reads each context once and computes all
 * its (token, head) columns together; otherwise each token runs as its own
 * decode, as in pa_varlen_attention.
 *  workspace  >= pa_decode_multi_workspace_size(...) bytes, 256-byte aligned.
 * ---------------------------------------------------------------------- */
size_t pa_decode_multi_workspace_size(int32_t num_seqs, int32_t tokens_per_seq,
                                      int32_t num_heads, int32_t head_dim,
                                      int32_t max_blocks_per_seq, int32_t block_size);
pa_status pa_decode_multi(void* out, const void* q, const void* k_cache, const void* v_cache,
                          pa_cache_desc cache, const int32_t* block_tables,
                          int32_t max_blocks_per_seq, const int32_t* context_lens,
                          int32_t num_seqs, int32_t tokens_per_seq, int32_t num_heads,
                          float scale, const float* k_scale, const float* v_scale,
                          void* workspace, size_t workspace_bytes, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_decode_shared_prefix -- pa_decode for a batch whose consecutive groups
 * of group_size sequences were forked from a common prefix (parallel
 * sampling, beam search, or requests sharing a system prompt through the
 * prefix cache): the shared blocks are read once per group instead of once
 * per member.  [LSB] "Copy-on-write for shared prefixes" (members' tables
 * point at the same physical blocks); [LSB] "How Paging Unlocks
 * High-Throughput Serving" (a prefix stored once and reused).  The pages
 * share the memory; reading it once is this library's addition, with the
 * same result as pa_decode.
 *
 * Sequence i belongs to group i / group_size.  A group's prefix is found on
 * the device: the longest run of leading block-table entries equal in all
 * its members' rows, capped at every member's whole blocks.  Pass 1 attends
 * each group's prefix once with all members' queries as the tensor-core
 * kernel's columns; pass 2 attends each sequence's remaining blocks; a
 * third kernel merges the two results by their log-sum-exp.  Needs the
 * tensor-core kernel for both passes (group x GQA group <= 16 for bf16, 8
 * for e4m3); otherwise, and for group_size 1, it runs pa_decode.
 *  workspace  >= pa_decode_shared_prefix_workspace_size(...), 256-byte aligned.
 *  Other arguments as pa_decode; num_seqs must be a multiple of group_size.
 * ---------------------------------------------------------------------- */
size_t pa_decode_shared_prefix_workspace_size(int32_t num_seqs, int32_t group_size,
                                              int32_t num_heads, int32_t head_dim,
                                              int32_t max_blocks_per_seq, int32_t block_size);
pa_status pa_decode_shared_prefix(void* out, const void* q, const void* k_cache,
                                  const void* v_cache, pa_cache_desc cache,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens, int32_t num_seqs,
                                  int32_t group_size, int32_t num_heads, float scale,
                                  const float* k_scale, const float* v_scale, void* workspace,
                                  size_t workspace_bytes, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_swap_blocks -- copy whole blocks between two caches of the same block
 * shape: dst[d] = src[s] for K and V, for every (s, d) pair.  An exhausted
 * pool must preempt a sequence ([LSB] BlockManager.allocate), and the
 * serving engine keeps a swap space of host RAM that preempted blocks move
 * into ([LSB] "The libraries that implement this", the swap-space knob);
 * they move back when the request resumes.  One cache is normally this GPU's pool and
 * the other a pinned host buffer of the same block layout (cudaHostAlloc /
 * torch pin_memory: with unified addressing the kernel reaches it through
 * its host pointer over the C2C link); both may also be device pools.
 * One kernel moves all pairs (16-byte vectors, one CTA per pair, K|V and
 * 32 KiB piece of the block): no per-block copy calls.
 *
 *  dst_k, dst_v      destination caches, [dst_num_blocks, B, H_kv, d].
 *  src_k, src_v      source caches, [src_num_blocks, B, H_kv, d].
 *  block_shape       B, H_kv, d and dtype (its num_blocks is ignored).
 *  block_pairs       device (or pinned host), [num_pairs, 2] int32 (src, dst);
 *                    pairs naming a block outside either cache are skipped.
 *                    Pairs must not write one destination block twice, and
 *                    source and destination blocks must not overlap.
 *  Returns PA_ERR_INVALID on bad sizes / NULL / misaligned pointers; runs
 *  asynchronously on `stream`; the caller keeps every buffer alive until
 *  the copy has run.
 * ---------------------------------------------------------------------- */
pa_status pa_swap_blocks(void* dst_k, void* dst_v, int32_t dst_num_blocks, const void* src_k,
                         const void* src_v, int32_t src_num_blocks, pa_cache_desc block_shape,
                         const int32_t* block_pairs, int32_t num_pairs, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_step_prepare -- a decode step's metadata, built on the device.
 * [LSB] "From Python bookkeeping to GPU tensors" rebuilds the slot mapping
 * and block tables on the host every step and copies them over, critical-
 * path work; here the tables and context lengths stay on the device and one
 * kernel updates them in place.  Per sequence i, in this order:
 *   1. every update (seq, idx, block) with seq == i sets
 *      block_tables[i][idx] = block (idx outside [0, max_blocks) is skipped);
 *   2. context_lens[i] += advance;
 *   3. slot_mapping[i] = table[i][(n-1)/B] * B + (n-1) % B for n =
 *      context_lens[i], the slot of the sequence's newest token ([LSB]
 *      BlockManager.slot_index), or -1 (pa_reshape_and_cache skips it) when
 *      n <= 0, (n-1)/B >= max_blocks, the entry is negative, or the slot
 *      does not fit in int32.
 *
 *  block_tables   device, [num_seqs, max_blocks_per_seq] int32, updated.
 *  context_lens   device, [num_seqs] int32, advanced in place.
 *  table_updates  device, [num_updates, 3] int32 (seq, logical block,
 *                 physical block) chosen by the host pool; may be NULL when
 *                 num_updates == 0.  Updates are not checked against a pool.
 *  advance        tokens added to every context length first (0 or more).
 *  slot_mapping   device, [num_seqs] int32, written.
 *  Returns PA_ERR_INVALID on bad sizes / NULL / misaligned pointers; runs
 *  asynchronously on `stream` and allocates nothing.
 * ---------------------------------------------------------------------- */
pa_status pa_step_prepare(int32_t* block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                          int32_t block_size, int32_t* context_lens,
                          const int32_t* table_updates, int32_t num_updates, int32_t advance,
                          int32_t* slot_mapping, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * Host-side block pool (off the hot path; not thread-safe: one owner).
 * Free queue is FIFO: allocation takes from the head, blocks whose ref count
 * drops to 0 join the tail.  [PKV] "Implementation" (BlockPool: deque free
 * queue, ref counts, allocate returns None when short); [LSB] BlockManager
 * (fork, cow_append, free_seq).  Allocation is all-or-nothing.
 * ---------------------------------------------------------------------- */
typedef struct pa_pool pa_pool;

/* Pool of num_blocks blocks, free queue 0..num_blocks-1.  NULL on bad size
 * or host OOM. */
pa_pool* pa_pool_create(int32_t num_blocks);
/* Pool whose initial free queue is `order` (a permutation of
 * 0..num_blocks-1, copied).  NULL if order is not a permutation. */
pa_pool* pa_pool_create_ordered(int32_t num_blocks, const int32_t* order);
void pa_pool_destroy(pa_pool* pool);
int32_t pa_pool_num_blocks(const pa_pool* pool);
int32_t pa_pool_num_free(const pa_pool* pool);
/* Ref count of a block, or -1 for an id outside the pool. */
int32_t pa_pool_refcount(const pa_pool* pool, int32_t block);
/* Copies the free queue, head first, into out[0..cap); returns its length. */
int32_t pa_pool_free_order(const pa_pool* pool, int32_t* out, int32_t cap);
/* Take n blocks from the head of the free queue (ref count 1 each) into
 * out_blocks[0..n).  PA_ERR_OOM (state unchanged) if fewer than n are free. */
pa_status pa_pool_alloc(pa_pool* pool, int32_t n, int32_t* out_blocks);
/* Fork: ref count += 1 for each listed block.  PA_ERR_INVALID (state
 * unchanged) if any block is outside the pool or free. */
pa_status pa_pool_incref(pa_pool* pool, const int32_t* blocks, int32_t n);
/* Release: ref count -= 1 for each listed block; blocks reaching 0 join the
 * tail of the free queue in list order.  PA_ERR_INVALID (state unchanged)
 * if the list would drive any ref count below 0. */
pa_status pa_pool_free(pa_pool* pool, const int32_t* blocks, int32_t n);
/* Copy-on-write decision before writing into `block`: ref count 1 gives
 * *out_dst = block (write in place); ref count > 1 takes a fresh block,
 * decrements the shared one and gives the fresh id (the caller copies
 * block -> *out_dst with pa_copy_blocks and remaps its table).  PA_ERR_OOM
 * (state unchanged) when no block is free; PA_ERR_INVALID for a free or
 * out-of-range block. */
pa_status pa_pool_cow(pa_pool* pool, int32_t block, int32_t* out_dst);

/* Prefix caching across requests, full blocks only.  The pages make the
 * full block the unit of sharing ([PKV] copy-on-write exercise: vLLM V1
 * shares only full blocks and each answer writes into its own block) and
 * point to cross-request reuse as the generalisation of shared prompt blocks
 * ([LSB] "Copy-on-write for shared prefixes"; "How Paging Unlocks
 * High-Throughput Serving": a system prompt stored once, reused by thousands
 * of requests).  The pages do not fix how a block is recognised; this pool
 * keys a full block by (parent block, the parent's generation, its B token
 * ids).  A block's generation advances each time it is handed out fresh,
 * which also drops its own entry, so a match always names the same content.
 * Freed cached blocks stay in the free queue (in freeing order, evicted
 * from the head like any free block) until a later prompt matches them.
 *
 * pa_pool_enable_prefix_cache: turn caching on for blocks of block_size
 * tokens (once; PA_ERR_INVALID if already on with another size). */
pa_status pa_pool_enable_prefix_cache(pa_pool* pool, int32_t block_size);
/* Blocks for a new sequence whose first num_tokens tokens are `tokens`:
 * out_blocks[0..ceil(num_tokens / B)) receives the leading full blocks found
 * in the cache (ref + 1; taken out of the free queue if they were free) and
 * then fresh blocks from the free-queue head.  Every fresh full block is
 * registered under its content at once, so the caller writes the K/V of
 * tokens [*num_cached_tokens, num_tokens) (its prefill) before the pool
 * serves another request.  *num_cached_tokens is a multiple of B: the
 * tokens whose K/V the shared blocks already hold.  All-or-nothing:
 * PA_ERR_OOM leaves the pool unchanged. */
pa_status pa_pool_alloc_prefix(pa_pool* pool, const int32_t* tokens, int32_t num_tokens,
                               int32_t* out_blocks, int32_t* num_cached_tokens);
/* Register a referenced block that has just become full (decode filled its
 * last slot) under (parent, its B tokens); parent is the sequence's previous
 * block or -1 for its first block.  A content already cached elsewhere is
 * not registered twice. */
pa_status pa_pool_register_block(pa_pool* pool, int32_t block, int32_t parent,
                                 const int32_t* tokens);
/* Blocks currently holding a registered entry (referenced or free). */
int32_t pa_pool_num_cached(const pa_pool* pool);

/* ------------------------------------------------------------------------
 * Diagnostics.
 * ---------------------------------------------------------------------- */
const char* pa_status_string(pa_status status);
/* Description of the last failure on the calling thread ("" if none). */
const char* pa_last_error(void);
/* Library version string, e.g. "0.1.0 sm_103a". */
const char* pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
