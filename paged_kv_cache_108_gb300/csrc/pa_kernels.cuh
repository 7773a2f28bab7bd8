// Internal declarations of the library's kernels and their launch helpers.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace pa {

constexpr int kSimtThreads = 128;  // threads per decode CTA (SIMT kernel)
constexpr int kChunkTokens = 64;   // tokens staged per pipeline stage
constexpr int kMinPartition = 64;  // split-K partitions are multiples of this

// Everything a decode kernel needs; device pointers except where noted.
struct DecodeParams {
  void* out;                   // [S, H, D] bf16
  const void* q;               // [S, H, D] bf16
  const void* k_cache;         // [NB, B, Hkv, D]
  const void* v_cache;
  const int32_t* block_tables;  // [S, max_blocks]
  const int32_t* context_lens;  // [S]
  float* ws_o;                 // [S, H, max_parts, D] unnormalised partials
  float2* ws_ml;               // [S, H, max_parts] (running max in log2 units, sum)
  const float* k_scale;        // fp8 only
  const float* v_scale;
  int32_t num_blocks;
  int32_t block_size;
  int32_t log2_block_size;
  int32_t num_kv_heads;
  int32_t num_heads;
  int32_t max_blocks;
  int32_t partition_tokens;  // multiple of kChunkTokens
  int32_t max_parts;         // partitions per sequence the grid covers
  float scale_log2;          // scale * log2(e)
};

// Launch the SIMT decode kernel for head_dim D in {64, 128}, group G in
// {1, 2, 4, 8}; grid (max_parts, num_kv_heads, num_seqs).
cudaError_t launch_decode_simt_bf16(const DecodeParams& p, int head_dim, int group,
                                    int num_seqs, cudaStream_t stream);
cudaError_t launch_decode_simt_fp8(const DecodeParams& p, int head_dim, int group,
                                   int num_seqs, cudaStream_t stream);
// Launch the split-K combine kernel.
cudaError_t launch_decode_reduce(const DecodeParams& p, int head_dim,
                                 int num_seqs, cudaStream_t stream);

// Tensor-core (tcgen05 + TMA) decode for a bf16 or fp8-e4m3 cache with head_dim 128.
struct TcLaunch {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  bool fp8;              // e4m3 cache with per-tensor k_scale / v_scale
  const float* k_scale;  // device scalars (fp8 only)
  const float* v_scale;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* workspace;  // >= tc_workspace_bytes(...)
  int num_seqs, num_heads, num_kv_heads, max_blocks, num_blocks, block_size;
  int num_ctas;     // persistent CTAs (one per SM)
  int tokens_per_seq;  // new tokens per sequence (1: decode); q/out hold S * this rows
  bool non_causal;     // all of a sequence's rows see all its keys (shared-prefix pass)
  float* lse;          // optional per-row log2-sum-exp output
  float scale;
  bool early_meta;  // the previous kernel only wrote the cache (see decode_tc.cu)
};
bool tc_supported(int head_dim, int group, bool fp8, int num_seqs, int block_size,
                  int tokens_per_seq = 1);
size_t tc_workspace_bytes(int64_t num_seqs, int64_t num_heads, int64_t max_ctx, int num_ctas,
                          int tokens_per_seq = 1);
cudaError_t launch_decode_tc(const TcLaunch& a, cudaStream_t stream);
// The head-packed tensor-core kernel (decode_hp.cu): a bf16 cache, one token
// per sequence, GQA group 1, 2 or 4, H_kv a multiple of its heads per tile
// (16 for group 1, else 8); any block size (head-major tiles for blocks of
// at least 128 / that many tokens, token-major below).
// Takes the same TcLaunch (fp8, tokens_per_seq and non_causal unused).
// Causal varlen attention for prefill chunks on the tensor cores
// (prefill_tc.cu): bf16 cache, head_dim 128, GQA group 1, 2, 4 or 8, at most
// 256 requests, blocks of at least 8 tokens.  workspace word 0 is the error
// word (an expired bounded wait or an out-of-range block id).
struct PrefillLaunch {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  void* workspace;
  int num_seqs, num_tokens, num_heads, num_kv_heads, max_blocks, num_blocks, block_size;
  int num_ctas;
  int min_tokens;  // requests with fewer new tokens get no tiles (0: every request)
  float scale;
  bool fp8;                // e4m3 cache: k_scale / v_scale are device scalars
  const float* k_scale;
  const float* v_scale;
};
bool prefill_supported(int head_dim, int group, bool fp8, int num_seqs, int block_size);
cudaError_t launch_prefill_tc(const PrefillLaunch& a, cudaStream_t stream);

bool hp_supported(int head_dim, int group, bool fp8, int num_seqs, int num_kv_heads,
                  int block_size, int tokens_per_seq);
size_t hp_workspace_bytes(int64_t num_seqs, int64_t num_heads, int num_ctas);
cudaError_t launch_decode_hp(const TcLaunch& a, cudaStream_t stream);

cudaError_t launch_reshape_and_cache(const void* key, const void* value,
                                     void* k_cache, void* v_cache,
                                     int64_t num_slots, int num_kv_heads,
                                     int head_dim, bool fp8,
                                     const int32_t* slot_mapping,
                                     int num_tokens, const float* k_scale,
                                     const float* v_scale,
                                     cudaStream_t stream);

cudaError_t launch_cascade_meta(const int32_t* block_tables, int max_blocks, int block_size,
                                const int32_t* context_lens, int num_seqs, int group,
                                int32_t* ptables, int32_t* plens, int32_t* stables,
                                int32_t* slens, cudaStream_t stream);
cudaError_t launch_lse_merge(const void* o1, const float* l1, const void* o2, const float* l2,
                             void* out, int64_t rows, int head_dim, cudaStream_t stream);

cudaError_t launch_varlen_meta(const int32_t* block_tables, int max_blocks, int block_size,
                               const int32_t* seq_lens, const int32_t* query_start_loc,
                               int uniform_tokens, int num_seqs, int num_tokens, int32_t* vtables,
                               int32_t* vlens, cudaStream_t stream, int tile_min = 0);

cudaError_t launch_step_prepare(int32_t* block_tables, int max_blocks, int block_size,
                                int32_t* context_lens, int num_seqs, const int32_t* updates,
                                int num_updates, int advance, int32_t* slot_mapping,
                                cudaStream_t stream);

cudaError_t launch_copy_blocks_between(void* dst_k, void* dst_v, int dst_blocks,
                                       const void* src_k, const void* src_v, int src_blocks,
                                       int64_t block_bytes, const int32_t* pairs, int num_pairs,
                                       cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache,
                               int64_t block_bytes, int num_blocks,
                               const int32_t* pairs, int num_pairs,
                               cudaStream_t stream);

}  // namespace pa
