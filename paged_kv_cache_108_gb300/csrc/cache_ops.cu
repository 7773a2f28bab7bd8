// Cache write (reshape_and_cache) and block copy (copy-on-write) kernels.
//
// reshape_and_cache: "Paged KV cache" (ai-infra-handbooks), PagedKVCache.write
// -- row i of key/value [N, H_kv, d] lands in row slot_mapping[i] of the pool
// viewed flat as [num_blocks*block_size, H_kv, d].  One thread moves one
// 16-byte piece of input (8 bf16 elements); consecutive threads cover
// consecutive pieces of a token's H_kv*d contiguous elements, so both the
// read and the scattered write are fully coalesced per token.  For an e4m3
// cache each element becomes e4m3_rne_satfinite(x / scale) with x / scale an
// IEEE fp32 division (fp8 KV cache: "4.6 PagedAttention & KV-Cache Memory
// Management", section "The libraries that implement this").
//
// copy_blocks: "4.6 PagedAttention & KV-Cache Memory Management", section
// "Copy-on-write for shared prefixes" -- the device copies block src -> dst
// before the diverging token is written.  Whole blocks are contiguous
// (block_size*H_kv*d*b bytes), so the copy is a plain 16-byte vector memcpy.
#include <cuda_bf16.h>

#include "pa_device.cuh"
#include "pa_kernels.cuh"

namespace pa {

namespace {

__device__ __forceinline__ uint16_t e4m3x2_rn_sat(float lo, float hi) {
  uint16_t r;
  // the first source lands in the upper byte, the second in the lower byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

template <bool FP8>
__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                             void* __restrict__ k_cache, void* __restrict__ v_cache,
                             int64_t num_slots, int pieces_per_token,
                             const int32_t* __restrict__ slot_mapping, int num_tokens,
                             const float* __restrict__ k_scale,
                             const float* __restrict__ v_scale) {
  // let a dependent decode kernel start its prologue while this one runs
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int64_t total = (int64_t)num_tokens * pieces_per_token;
  float ks = 1.f, vs = 1.f;
  if (FP8) {
    ks = *k_scale;
    vs = *v_scale;
  }
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tok = idx / pieces_per_token;
    const int64_t r = idx - tok * pieces_per_token;
    const int64_t slot = slot_mapping[tok];
    if (slot < 0 || slot >= num_slots) continue;  // padding token or bad slot
    const int64_t dst = slot * pieces_per_token + r;
    const uint4 kv = key[idx];
    const uint4 vv = value[idx];
    if (!FP8) {
      reinterpret_cast<uint4*>(k_cache)[dst] = kv;
      reinterpret_cast<uint4*>(v_cache)[dst] = vv;
    } else {
      float kf[8], vf[8];
      Unpack16<false>::run(kv, kf);
      Unpack16<false>::run(vv, vf);
      uint32_t kw[2], vw[2];
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const uint16_t k01 = e4m3x2_rn_sat(__fdiv_rn(kf[4 * w + 0], ks), __fdiv_rn(kf[4 * w + 1], ks));
        const uint16_t k23 = e4m3x2_rn_sat(__fdiv_rn(kf[4 * w + 2], ks), __fdiv_rn(kf[4 * w + 3], ks));
        const uint16_t v01 = e4m3x2_rn_sat(__fdiv_rn(vf[4 * w + 0], vs), __fdiv_rn(vf[4 * w + 1], vs));
        const uint16_t v23 = e4m3x2_rn_sat(__fdiv_rn(vf[4 * w + 2], vs), __fdiv_rn(vf[4 * w + 3], vs));
        kw[w] = (uint32_t)k01 | ((uint32_t)k23 << 16);
        vw[w] = (uint32_t)v01 | ((uint32_t)v23 << 16);
      }
      reinterpret_cast<uint2*>(k_cache)[dst] = make_uint2(kw[0], kw[1]);
      reinterpret_cast<uint2*>(v_cache)[dst] = make_uint2(vw[0], vw[1]);
    }
  }
}

constexpr int kCopyThreads = 256;
constexpr int64_t kCopyChunk = 32 * 1024;  // bytes per CTA

// Block copies between two caches of the same block shape (the same cache
// for copy-on-write; a device cache and a pinned host cache for a swap).
// Grid: (pair, K|V, 32 KiB piece of the block).  Pairs naming a block
// outside either cache are skipped.
__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(char* __restrict__ dst_k, char* __restrict__ dst_v, int dst_blocks,
                       const char* __restrict__ src_k, const char* __restrict__ src_v,
                       int src_blocks, int64_t block_bytes, const int32_t* __restrict__ pairs) {
  const int pi = blockIdx.x;
  const char* sbase = blockIdx.y ? src_v : src_k;
  char* dbase = blockIdx.y ? dst_v : dst_k;
  const int src = pairs[2 * pi];
  const int dst = pairs[2 * pi + 1];
  if ((unsigned)src >= (unsigned)src_blocks || (unsigned)dst >= (unsigned)dst_blocks) return;
  const int64_t off = (int64_t)blockIdx.z * kCopyChunk;
  if (off >= block_bytes) return;
  const int64_t len = min(kCopyChunk, block_bytes - off) / 16;
  const uint4* s = reinterpret_cast<const uint4*>(sbase + (int64_t)src * block_bytes + off);
  uint4* d = reinterpret_cast<uint4*>(dbase + (int64_t)dst * block_bytes + off);
  constexpr int U = 8;
  for (int64_t j0 = 0; j0 < len; j0 += (int64_t)U * kCopyThreads) {
    uint4 tmp[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t j = j0 + u * kCopyThreads + threadIdx.x;
      if (j < len) tmp[u] = s[j];
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t j = j0 + u * kCopyThreads + threadIdx.x;
      if (j < len) d[j] = tmp[u];
    }
  }
}

// Step metadata on the device ("4.6 PagedAttention & KV-Cache Memory
// Management", section "From Python bookkeeping to GPU tensors": the slot
// mapping and block tables are rebuilt every step; here they change in place
// on the device).  Thread i owns sequence i: it applies the block-table
// updates addressed to its sequence (the host pool chose the blocks), adds
// `advance` to its context length, and computes the slot of its newest token,
//   slot = table[i][(n - 1) / B] * B + (n - 1) % B,
// or -1 when n <= 0, the position lies past the table, or the entry is < 0.
__global__ void step_prepare_kernel(int32_t* __restrict__ block_tables, int max_blocks,
                                    int block_size, int32_t* __restrict__ context_lens,
                                    int num_seqs, const int32_t* __restrict__ updates,
                                    int num_updates, int advance,
                                    int32_t* __restrict__ slot_mapping) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= num_seqs) return;
  int32_t* row = block_tables + (int64_t)i * max_blocks;
  for (int u = 0; u < num_updates; ++u) {
    if (updates[3 * u] != i) continue;
    const int idx = updates[3 * u + 1];
    if ((unsigned)idx < (unsigned)max_blocks) row[idx] = updates[3 * u + 2];
  }
  int n = context_lens[i];
  if (advance) {
    n += advance;
    context_lens[i] = n;
  }
  int slot = -1;
  if (n > 0) {
    const int pos = n - 1;
    const int lb = pos / block_size;
    if (lb < max_blocks) {
      const int blk = row[lb];
      const int64_t sl = (int64_t)blk * block_size + pos % block_size;
      if (blk >= 0 && sl <= 0x7fffffff) slot = (int)sl;
    }
  }
  slot_mapping[i] = slot;
}

// Varlen (multi-token) attention as decode over one virtual sequence per
// new token ("Paged KV cache", section "Paged attention": request i's new
// token j sits at position seq_len - num_new + j and sees positions up to
// it).  CTA t handles token t: it finds its request i (qsl[i] <= t <
// qsl[i+1], binary search), writes the causal context length
// seq_len - num_new + j + 1 (0 when the request's numbers are inconsistent:
// num_new > seq_len), and copies the first ceil(ctx / B) entries of the
// request's block-table row into the token's row.
// qsl == nullptr: every request adds `uniform_tokens` tokens (token t
// belongs to request t / uniform_tokens).
__global__ void varlen_meta_kernel(const int32_t* __restrict__ block_tables, int max_blocks,
                                   int block_size, const int32_t* __restrict__ seq_lens,
                                   const int32_t* __restrict__ qsl, int uniform_tokens,
                                   int num_seqs, int tile_min, int32_t* __restrict__ vtables,
                                   int32_t* __restrict__ vlens) {
  const int t = blockIdx.x;
  __shared__ int s_req, s_ctx;
  if (threadIdx.x == 0) {
    int a, start, num_new;
    if (qsl) {
      a = 0;
      int b = num_seqs - 1;  // last request with qsl[i] <= t
      while (a < b) {
        const int m = (a + b + 1) >> 1;
        if (qsl[m] <= t) a = m; else b = m - 1;
      }
      start = qsl[a];
      num_new = qsl[a + 1] - qsl[a];
    } else {
      a = t / uniform_tokens;
      start = a * uniform_tokens;
      num_new = uniform_tokens;
    }
    const int n = seq_lens[a];
    int ctx = n - num_new + (t - start) + 1;
    if (num_new > n || t >= start + num_new || ctx < 1) ctx = 0;
    // tokens of requests the prefill tiles serve: an empty virtual sequence
    if (tile_min > 0 && num_new >= tile_min) ctx = 0;
    if ((int64_t)ctx > (int64_t)max_blocks * block_size) ctx = 0;
    s_req = a;
    s_ctx = ctx;
    vlens[t] = ctx;
  }
  __syncthreads();
  const int nb = (s_ctx + block_size - 1) / block_size;
  const int32_t* src = block_tables + (int64_t)s_req * max_blocks;
  int32_t* dst = vtables + (int64_t)t * max_blocks;
  for (int k = threadIdx.x; k < nb; k += blockDim.x) dst[k] = src[k];
}

// Shared-prefix (cascade) split of a batch whose consecutive groups of m
// sequences were forked from a common prefix.  CTA i handles sequence i of
// group v = i / m (leader L = v * m).  The group's shared prefix is the
// longest run of leading block-table entries equal in every member's row,
// capped at each member's whole blocks (a member never attends past its own
// context); the leader's CTA writes the prefix row (its first P blocks) and
// length, and every CTA writes its sequence's suffix row (the entries after
// the prefix) and length n_i - P * B.
__global__ void cascade_meta_kernel(const int32_t* __restrict__ block_tables, int max_blocks,
                                    int block_size, const int32_t* __restrict__ context_lens,
                                    int group, int32_t* __restrict__ ptables,
                                    int32_t* __restrict__ plens, int32_t* __restrict__ stables,
                                    int32_t* __restrict__ slens) {
  const int i = blockIdx.x;
  const int L = i - i % group;
  __shared__ int s_pb;
  if (threadIdx.x == 0) {
    int pb = max_blocks;
    for (int j = 0; j < group; ++j) {
      const int n = context_lens[L + j];
      pb = min(pb, n > 0 ? n / block_size : 0);
    }
    s_pb = pb;
  }
  __syncthreads();
  // first index where some member's row differs from the leader's
  const int32_t* lead = block_tables + (int64_t)L * max_blocks;
  for (int k = threadIdx.x; k < s_pb; k += blockDim.x) {
    bool same = true;
    for (int j = 1; j < group; ++j) same &= block_tables[(int64_t)(L + j) * max_blocks + k] == lead[k];
    if (!same) atomicMin(&s_pb, k);
  }
  __syncthreads();
  const int pb = s_pb;
  if (i == L) {
    for (int k = threadIdx.x; k < pb; k += blockDim.x) ptables[(int64_t)(L / group) * max_blocks + k] = lead[k];
    if (threadIdx.x == 0) plens[L / group] = pb * block_size;
  }
  const int n = max(context_lens[i], 0);
  const int nb = (n + block_size - 1) / block_size;
  const int32_t* row = block_tables + (int64_t)i * max_blocks;
  for (int k = threadIdx.x; k + pb < nb; k += blockDim.x)
    stables[(int64_t)i * max_blocks + k] = row[pb + k];
  if (threadIdx.x == 0) slens[i] = n - pb * block_size;
}

// out = the two partial results combined by their log2-sum-exp weights
// (rows with both weights zero, i.e. no key at all, get zeros).
__global__ void lse_merge_kernel(const __nv_bfloat16* __restrict__ o1,
                                 const float* __restrict__ l1,
                                 const __nv_bfloat16* __restrict__ o2,
                                 const float* __restrict__ l2, __nv_bfloat16* __restrict__ out,
                                 int64_t rows, int head_dim) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * head_dim) return;
  const int64_t r = idx / head_dim;
  const float a = l1[r], b = l2[r];
  const float m = fmaxf(a, b);
  float res = 0.f;
  if (m != -INFINITY) {
    const float wa = exp2f(a - m), wb = exp2f(b - m);
    res = (wa * __bfloat162float(o1[idx]) + wb * __bfloat162float(o2[idx])) / (wa + wb);
  }
  out[idx] = __float2bfloat16_rn(res);
}

}  // namespace

cudaError_t launch_cascade_meta(const int32_t* block_tables, int max_blocks, int block_size,
                                const int32_t* context_lens, int num_seqs, int group,
                                int32_t* ptables, int32_t* plens, int32_t* stables,
                                int32_t* slens, cudaStream_t stream) {
  cascade_meta_kernel<<<num_seqs, 128, 0, stream>>>(block_tables, max_blocks, block_size,
                                                    context_lens, group, ptables, plens, stables,
                                                    slens);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const void* o1, const float* l1, const void* o2, const float* l2,
                             void* out, int64_t rows, int head_dim, cudaStream_t stream) {
  const int64_t n = rows * head_dim;
  lse_merge_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o1), l1, static_cast<const __nv_bfloat16*>(o2), l2,
      static_cast<__nv_bfloat16*>(out), rows, head_dim);
  return cudaGetLastError();
}

cudaError_t launch_varlen_meta(const int32_t* block_tables, int max_blocks, int block_size,
                               const int32_t* seq_lens, const int32_t* query_start_loc,
                               int uniform_tokens, int num_seqs, int num_tokens, int32_t* vtables,
                               int32_t* vlens, cudaStream_t stream, int tile_min) {
  varlen_meta_kernel<<<num_tokens, 128, 0, stream>>>(block_tables, max_blocks, block_size,
                                                     seq_lens, query_start_loc, uniform_tokens,
                                                     num_seqs, tile_min, vtables, vlens);
  return cudaGetLastError();
}

cudaError_t launch_step_prepare(int32_t* block_tables, int max_blocks, int block_size,
                                int32_t* context_lens, int num_seqs, const int32_t* updates,
                                int num_updates, int advance, int32_t* slot_mapping,
                                cudaStream_t stream) {
  const int threads = 128;
  step_prepare_kernel<<<(num_seqs + threads - 1) / threads, threads, 0, stream>>>(
      block_tables, max_blocks, block_size, context_lens, num_seqs, updates, num_updates,
      advance, slot_mapping);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const void* key, const void* value,
                                     void* k_cache, void* v_cache,
                                     int64_t num_slots, int num_kv_heads,
                                     int head_dim, bool fp8,
                                     const int32_t* slot_mapping,
                                     int num_tokens, const float* k_scale,
                                     const float* v_scale,
                                     cudaStream_t stream) {
  const int ppt = num_kv_heads * head_dim / 8;  // 16-byte input pieces per token
  const int64_t total = (int64_t)num_tokens * ppt;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  const int grid = (int)(blocks < 65535 * 8 ? blocks : 65535 * 8);
  if (fp8)
    reshape_and_cache_kernel<true><<<grid, threads, 0, stream>>>(
        static_cast<const uint4*>(key), static_cast<const uint4*>(value), k_cache, v_cache,
        num_slots, ppt, slot_mapping, num_tokens, k_scale, v_scale);
  else
    reshape_and_cache_kernel<false><<<grid, threads, 0, stream>>>(
        static_cast<const uint4*>(key), static_cast<const uint4*>(value), k_cache, v_cache,
        num_slots, ppt, slot_mapping, num_tokens, k_scale, v_scale);
  return cudaGetLastError();
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, int64_t block_bytes,
                               int num_blocks, const int32_t* pairs, int num_pairs,
                               cudaStream_t stream) {
  return launch_copy_blocks_between(k_cache, v_cache, num_blocks, k_cache, v_cache, num_blocks,
                                    block_bytes, pairs, num_pairs, stream);
}

cudaError_t launch_copy_blocks_between(void* dst_k, void* dst_v, int dst_blocks,
                                       const void* src_k, const void* src_v, int src_blocks,
                                       int64_t block_bytes, const int32_t* pairs, int num_pairs,
                                       cudaStream_t stream) {
  const int64_t chunks = (block_bytes + kCopyChunk - 1) / kCopyChunk;
  dim3 grid(num_pairs, 2, (unsigned)chunks);
  copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>(
      static_cast<char*>(dst_k), static_cast<char*>(dst_v), dst_blocks,
      static_cast<const char*>(src_k), static_cast<const char*>(src_v), src_blocks, block_bytes,
      pairs);
  return cudaGetLastError();
}

}  // namespace pa
