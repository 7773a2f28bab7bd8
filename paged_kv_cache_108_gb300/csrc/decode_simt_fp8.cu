// Instantiations of the SIMT paged decode kernel for a fp8 KV cache.
#include <cuda_bf16.h>

#include <atomic>

#include "decode_simt.cuh"

namespace pa {

namespace {

template <int D, int G>
cudaError_t launch_one(const DecodeParams& p, int num_seqs, cudaStream_t stream) {
  using C = SimtCfg<D, G, true>;
  const int table_entries = (p.partition_tokens >> p.log2_block_size) > 1
                                ? (p.partition_tokens >> p.log2_block_size)
                                : 1;
  const size_t smem = (size_t)C::FIXED_B + 4 * (size_t)table_entries;
  static std::atomic<size_t> configured{0};
  if (configured.load(std::memory_order_relaxed) < smem) {
    cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel<D, G, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured.store(smem, std::memory_order_relaxed);
  }
  dim3 grid(p.max_parts, p.num_kv_heads, num_seqs);
  decode_simt_kernel<D, G, true><<<grid, C::NT, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t by_group(const DecodeParams& p, int group, int num_seqs, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_one<D, 1>(p, num_seqs, stream);
    case 2: return launch_one<D, 2>(p, num_seqs, stream);
    case 4: return launch_one<D, 4>(p, num_seqs, stream);
    case 8: return launch_one<D, 8>(p, num_seqs, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_simt_fp8(const DecodeParams& p, int head_dim, int group,
                                   int num_seqs, cudaStream_t stream) {
  switch (head_dim) {
    case 64: return by_group<64>(p, group, num_seqs, stream);
    case 128: return by_group<128>(p, group, num_seqs, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
