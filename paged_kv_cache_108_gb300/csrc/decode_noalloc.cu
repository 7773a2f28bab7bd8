// pa_decode_noalloc: paged decode whose split-K scratch lives in a fixed
// array inside this library instead of a buffer the caller provides.
//
// Why it exists: pa_decode asks its caller for a workspace, which most
// callers get from their allocator.  Some callers cannot hand out device
// memory at the point of the call -- for example a plugin whose host
// application owns every device allocation, or a latency-critical serving
// loop that must not call cudaMalloc because cudaMalloc can synchronise the
// device.  For them this entry point uses a file-scope __device__ array of
// PA_DECODE_NOALLOC_SCRATCH_BYTES bytes.  Every GPU that loads the library
// holds that array until the process exits.
//
// It reuses pa_decode_ex unchanged: it only picks a split-K partition length
// whose scratch fits in the array (the smallest power of two from 256 tokens
// up), then passes the array as the workspace.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <mutex>

#include "pa.h"
#include "pa_host.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
std::atomic<void*> g_scratch_ptr[kMaxDevices];  // device address per device, once looked up

// Device address of the scratch array on the current device; looked up once
// per device (with that device current) and cached.
pa_status scratch_for_current_device(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pa_fail(PA_ERR_CUDA, "pa_decode_noalloc: cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices)
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode_noalloc: device index beyond 63");
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p) {
        char buf[200];
        snprintf(buf, sizeof buf, "pa_decode_noalloc: cudaGetSymbolAddress failed: %s",
                 cudaGetErrorString(e));
        return pa_fail(PA_ERR_CUDA, buf);
      }
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *ptr = p;
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, pa_cache_desc cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, int32_t num_seqs,
                                       int32_t num_heads, float scale, const float* k_scale,
                                       const float* v_scale, pa_stream_t stream) {
  if (num_seqs <= 0 || num_heads <= 0 || max_blocks_per_seq <= 0 || cache.head_dim <= 0 ||
      cache.block_size <= 0) {
    // let pa_decode_ex report the precise problem (or do nothing for 0 sequences)
    return pa_decode_ex(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                        context_lens, num_seqs, num_heads, scale, k_scale, v_scale, nullptr, 0,
                        nullptr, stream);
  }
  // the smallest partition length (fewest idle SMs) whose partials fit
  int32_t partition = 0;
  for (int32_t ps = 256; ps <= 65536; ps *= 2) {
    const size_t need = pa_decode_workspace_size_ex(num_seqs, num_heads, cache.head_dim,
                                                    max_blocks_per_seq, cache.block_size, ps);
    if (need <= (size_t)PA_DECODE_NOALLOC_SCRATCH_BYTES) {
      partition = ps;
      break;
    }
  }
  if (partition == 0) {
    char buf[240];
    snprintf(buf, sizeof buf,
             "pa_decode_noalloc: %d sequences x %d heads x %d tokens need more than the %u-byte "
             "built-in scratch; use pa_decode with a caller workspace",
             num_seqs, num_heads, max_blocks_per_seq * cache.block_size,
             (unsigned)PA_DECODE_NOALLOC_SCRATCH_BYTES);
    return pa_fail(PA_ERR_UNSUPPORTED, buf);
  }
  void* scratch = nullptr;
  pa_status st = scratch_for_current_device(&scratch);
  if (st != PA_OK) return st;
  // no part of the scratch has to start at zero: every split-K partial is
  // written by the decode kernel before the combine kernel reads it
  pa_decode_opts opts{partition, 0};
  return pa_decode_ex(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                      context_lens, num_seqs, num_heads, scale, k_scale, v_scale, scratch,
                      (size_t)PA_DECODE_NOALLOC_SCRATCH_BYTES, &opts, stream);
}
