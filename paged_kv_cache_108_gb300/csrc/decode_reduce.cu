// Split-K combine for paged decode ("4.6 PagedAttention & KV-Cache Memory
// Management", section "Performance considerations": PagedAttention v2
// splits a long sequence across CTAs and reduces over the sequence).
//
// Partition j of a (sequence, query head) left an unnormalised accumulator
// o_j = sum_t 2^(s_t - m_j) v_t, its running max m_j (log2 units) and its sum
// l_j = sum_t 2^(s_t - m_j).  With M = max_j m_j and w_j = 2^(m_j - M):
//   out = (sum_j w_j o_j) / (sum_j w_j l_j),
// the same online-softmax identity that merges chunks inside one CTA.
// Sequences that fit in one partition were finished by the decode kernel.
#include <cuda_bf16.h>

#include "pa_device.cuh"
#include "pa_kernels.cuh"

namespace pa {

namespace {

constexpr int kReduceThreads = 128;

__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, v, off);
    v = is_max ? fmaxf(v, o) : v + o;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();  // red may still be read by a previous reduction
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kReduceThreads / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
  return r;
}

__global__ void __launch_bounds__(kReduceThreads)
    decode_reduce_kernel(const DecodeParams p, int head_dim) {
  extern __shared__ float w_s[];  // [max_parts] partition weights
  __shared__ float red[kReduceThreads / 32];
  const int h = blockIdx.x;
  const int seq = blockIdx.y;
  const int n = min(p.context_lens[seq], p.max_blocks << p.log2_block_size);
  const int P = (n + p.partition_tokens - 1) / p.partition_tokens;
  if (P <= 1) return;
  const int64_t row = (int64_t)seq * p.num_heads + h;
  const float2* ml = p.ws_ml + row * p.max_parts;

  float m = -INFINITY;
  for (int j = threadIdx.x; j < P; j += kReduceThreads) m = fmaxf(m, ml[j].x);
  const float M = block_reduce(m, red, true);
  float lsum = 0.f;
  for (int j = threadIdx.x; j < P; j += kReduceThreads) {
    const float2 v = ml[j];
    const float w = fast_exp2(v.x - M);
    w_s[j] = w;
    lsum += w * v.y;
  }
  const float L = block_reduce(lsum, red, false);  // also publishes w_s
  const float inv = 1.f / L;
  const float* o = p.ws_o + row * p.max_parts * head_dim;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + row * head_dim;
  for (int e = threadIdx.x; e < head_dim; e += kReduceThreads) {
    float a0 = 0.f, a1 = 0.f;
    int j = 0;
    for (; j + 1 < P; j += 2) {
      a0 = fmaf(w_s[j], o[(int64_t)j * head_dim + e], a0);
      a1 = fmaf(w_s[j + 1], o[(int64_t)(j + 1) * head_dim + e], a1);
    }
    if (j < P) a0 = fmaf(w_s[j], o[(int64_t)j * head_dim + e], a0);
    out[e] = __float2bfloat16_rn((a0 + a1) * inv);
  }
}

}  // namespace

cudaError_t launch_decode_reduce(const DecodeParams& p, int head_dim, int num_seqs,
                                 cudaStream_t stream) {
  dim3 grid(p.num_heads, num_seqs);
  const size_t smem = sizeof(float) * (size_t)p.max_parts;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(decode_reduce_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  decode_reduce_kernel<<<grid, kReduceThreads, smem, stream>>>(p, head_dim);
  return cudaGetLastError();
}

}  // namespace pa
