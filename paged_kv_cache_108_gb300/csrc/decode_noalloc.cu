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
//
// Status word.  The tensor-core kernels report an expired bounded wait or an
// out-of-range block id by writing a nonzero code into word 0 of their
// workspace; they never clear it.  Here word 0 of the array is that word for
// every call that runs a tensor-core kernel (the array's start is their
// workspace), and the SIMT kernel, which reports nothing, gets the array from
// byte 256 on so its partials never land on the word.  The word therefore
// keeps the first call's zero (a __device__ array starts zeroed) until a
// kernel reports a fault, and stays set until pa_decode_noalloc_error reads
// and clears it.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <mutex>

#include "pa.h"
#include "pa_host.h"

namespace {

// Bytes at the array's start kept clear of SIMT partials (word 0 = status).
constexpr size_t kStatusBytes = 256;

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
  // the tensor-core kernels take the whole array (word 0 is their error word);
  // the SIMT kernel takes it from kStatusBytes on
  const int kernel = pa_decode_auto_kernel(cache, num_heads, num_seqs, 1);
  const size_t offset = kernel == 1 ? kStatusBytes : 0;
  const size_t room = (size_t)PA_DECODE_NOALLOC_SCRATCH_BYTES - offset;
  // the smallest partition length (fewest idle SMs) whose partials fit
  int32_t partition = 0;
  for (int32_t ps = 256; ps <= 65536; ps *= 2) {
    const size_t need = pa_decode_workspace_size_ex(num_seqs, num_heads, cache.head_dim,
                                                    max_blocks_per_seq, cache.block_size, ps);
    if (need <= room) {
      partition = ps;
      break;
    }
  }
  if (partition == 0) {
    char buf[240];
    snprintf(buf, sizeof buf,
             "pa_decode_noalloc: %d sequences x %d heads x %lld tokens need more than the "
             "%u-byte built-in scratch; use pa_decode with a caller workspace",
             num_seqs, num_heads, (long long)max_blocks_per_seq * cache.block_size,
             (unsigned)PA_DECODE_NOALLOC_SCRATCH_BYTES);
    return pa_fail(PA_ERR_UNSUPPORTED, buf);
  }
  void* scratch = nullptr;
  pa_status st = scratch_for_current_device(&scratch);
  if (st != PA_OK) return st;
  // no part of the workspace has to start at zero: every split-K partial is
  // written before it is read, and the merge counters carry a per-call tag
  pa_decode_opts opts{partition, kernel};
  return pa_decode_ex(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                      context_lens, num_seqs, num_heads, scale, k_scale, v_scale,
                      static_cast<unsigned char*>(scratch) + offset, room, &opts, stream);
}

extern "C" pa_status pa_decode_noalloc_error(int32_t* code, pa_stream_t stream) {
  if (!code) return pa_fail(PA_ERR_INVALID, "pa_decode_noalloc_error: NULL code");
  void* scratch = nullptr;
  pa_status st = scratch_for_current_device(&scratch);
  if (st != PA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(code, scratch, sizeof(int32_t), cudaMemcpyDefault, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) {
    char buf[200];
    snprintf(buf, sizeof buf, "pa_decode_noalloc_error: %s", cudaGetErrorString(e));
    return pa_fail(PA_ERR_CUDA, buf);
  }
  return PA_OK;
}
