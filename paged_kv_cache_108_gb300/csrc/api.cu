// C entry points: argument validation, launch configuration, dispatch.
// The contract of every function is stated in include/pa.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>

#include "pa.h"
#include "pa_host.h"
#include "pa_kernels.cuh"

namespace {

thread_local std::string g_last_error;

constexpr int kAutoPartition = 512;     // default split-K partition (tokens)
constexpr int kAutoPartitionMin = 256;  // smallest automatic choice
constexpr int kMaxPartition = 65536;
// pa_varlen_attention method 0: requests adding this many new tokens or more
// take the tensor-core prefill tiles
constexpr int kTileMinTokens = 16;

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

int ilog2(int64_t x) {
  int r = 0;
  while ((int64_t(1) << r) < x) ++r;
  return r;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Workspace layout for a given partition length: partial accumulators
// [S, H, P, D] fp32 then (m, l) pairs [S, H, P] at a 256-byte boundary.
struct WorkspaceLayout {
  int64_t parts = 0;
  size_t o_bytes = 0;
  size_t ml_offset = 0;
  size_t total = 0;
};

WorkspaceLayout workspace_layout(int64_t num_seqs, int64_t num_heads, int64_t head_dim,
                                 int64_t max_ctx, int64_t partition) {
  WorkspaceLayout w;
  w.parts = ceil_div(max_ctx, partition);
  if (w.parts <= 1 || num_seqs <= 0 || num_heads <= 0) {
    w.parts = w.parts < 1 ? 1 : w.parts;
    return w;  // a single partition writes the output directly
  }
  w.o_bytes = (size_t)(num_seqs * num_heads * w.parts * head_dim) * sizeof(float);
  w.ml_offset = align_up(w.o_bytes, 256);
  w.total = w.ml_offset + (size_t)(num_seqs * num_heads * w.parts) * 2 * sizeof(float);
  return w;
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 152;
  return n;
}

int auto_partition(int64_t num_seqs, int64_t num_kv_heads, int64_t max_ctx) {
  // Split long contexts so that enough CTAs exist to fill the machine a few
  // times over (short sequences stay in one partition and skip the combine).
  int ps = kAutoPartition;
  const int64_t want = 4LL * num_sms();
  while (ps > kAutoPartitionMin && num_seqs * num_kv_heads * ceil_div(max_ctx, ps) < want)
    ps /= 2;
  return ps;
}

pa_status check_cache(const pa_cache_desc& c, const char* fn) {
  char buf[192];
  if (c.num_blocks <= 0 || c.block_size <= 0 || c.num_kv_heads <= 0 || c.head_dim <= 0) {
    snprintf(buf, sizeof buf, "%s: cache sizes must be positive", fn);
    return pa_fail(PA_ERR_INVALID, buf);
  }
  if (c.dtype != PA_KV_BF16 && c.dtype != PA_KV_FP8_E4M3) {
    snprintf(buf, sizeof buf, "%s: unknown cache dtype %d", fn, c.dtype);
    return pa_fail(PA_ERR_INVALID, buf);
  }
  if (c.head_dim != 64 && c.head_dim != 128) {
    snprintf(buf, sizeof buf, "%s: head_dim %d unsupported (64 or 128)", fn, c.head_dim);
    return pa_fail(PA_ERR_UNSUPPORTED, buf);
  }
  if (!is_pow2(c.block_size) || c.block_size > 1024) {
    snprintf(buf, sizeof buf, "%s: block_size %d unsupported (power of two <= 1024)", fn,
             c.block_size);
    return pa_fail(PA_ERR_UNSUPPORTED, buf);
  }
  if ((int64_t)c.num_blocks * c.block_size > INT32_MAX) {
    snprintf(buf, sizeof buf, "%s: num_blocks * block_size exceeds 2^31-1 slots", fn);
    return pa_fail(PA_ERR_UNSUPPORTED, buf);
  }
  return PA_OK;
}

pa_status check_scales(const pa_cache_desc& c, const float* ks, const float* vs, const char* fn) {
  char buf[160];
  if (c.dtype == PA_KV_FP8_E4M3 && (!ks || !vs)) {
    snprintf(buf, sizeof buf, "%s: fp8 cache needs k_scale and v_scale", fn);
    return pa_fail(PA_ERR_INVALID, buf);
  }
  if (c.dtype == PA_KV_BF16 && (ks || vs)) {
    snprintf(buf, sizeof buf, "%s: k_scale/v_scale must be NULL for a bf16 cache", fn);
    return pa_fail(PA_ERR_INVALID, buf);
  }
  return PA_OK;
}

pa_status cuda_status(cudaError_t e, const char* fn) {
  if (e == cudaSuccess) return PA_OK;
  char buf[256];
  snprintf(buf, sizeof buf, "%s: %s", fn, cudaGetErrorString(e));
  return pa_fail(PA_ERR_CUDA, buf);
}

}  // namespace

void pa_set_error(const char* msg) { g_last_error = msg ? msg : ""; }

pa_status pa_fail(pa_status st, const char* msg) {
  pa_set_error(msg);
  return st;
}

extern "C" {

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID: return "PA_ERR_INVALID";
    case PA_ERR_OOM: return "PA_ERR_OOM";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
  }
  return "PA_ERR_UNKNOWN";
}

const char* pa_last_error(void) { return g_last_error.c_str(); }

const char* pa_version(void) { return "0.1.0 sm_103a"; }

pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache,
                               void* v_cache, pa_cache_desc cache,
                               const int32_t* slot_mapping, int32_t num_tokens,
                               const float* k_scale, const float* v_scale,
                               pa_stream_t stream) {
  const char* fn = "pa_reshape_and_cache";
  pa_status st = check_cache(cache, fn);
  if (st != PA_OK) return st;
  if ((st = check_scales(cache, k_scale, v_scale, fn)) != PA_OK) return st;
  if (num_tokens < 0) return pa_fail(PA_ERR_INVALID, "pa_reshape_and_cache: num_tokens < 0");
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping)
    return pa_fail(PA_ERR_INVALID, "pa_reshape_and_cache: NULL pointer");
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 4))
    return pa_fail(PA_ERR_INVALID, "pa_reshape_and_cache: misaligned pointer");
  const int64_t num_slots = (int64_t)cache.num_blocks * cache.block_size;
  return cuda_status(pa::launch_reshape_and_cache(key, value, k_cache, v_cache, num_slots,
                                                  cache.num_kv_heads, cache.head_dim,
                                                  cache.dtype == PA_KV_FP8_E4M3, slot_mapping,
                                                  num_tokens, k_scale, v_scale,
                                                  reinterpret_cast<cudaStream_t>(stream)),
                     fn);
}

size_t pa_decode_workspace_size_ex(int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                                   int32_t max_blocks_per_seq, int32_t block_size,
                                   int32_t partition_tokens) {
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 ||
      block_size <= 0)
    return 0;
  int64_t ps = partition_tokens > 0 ? partition_tokens : kAutoPartitionMin;
  if (partition_tokens > 0 && (!is_pow2(ps) || ps < pa::kMinPartition || ps > kMaxPartition))
    return 0;
  const int64_t max_ctx = (int64_t)max_blocks_per_seq * block_size;
  size_t need = workspace_layout(num_seqs, num_heads, head_dim, max_ctx, ps).total;
  if (head_dim == 128) {  // the tensor-core kernels may serve this shape
    const size_t tc = pa::tc_workspace_bytes(num_seqs, num_heads, max_ctx, num_sms());
    if (tc > need) need = tc;
    const size_t hp = pa::hp_workspace_bytes(num_seqs, num_heads, num_sms());
    if (hp > need) need = hp;
  }
  return need;
}

size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                                int32_t max_blocks_per_seq, int32_t block_size) {
  return pa_decode_workspace_size_ex(num_seqs, num_heads, head_dim, max_blocks_per_seq,
                                     block_size, 0);
}

}  // extern "C"

// The automatic kernel choice (pa_decode_opts.kernel 0) for a call of this
// shape: 3 head-packed, 2 per-head tensor-core, 1 SIMT.  The head-packed
// kernel streams faster (bigger copies) but its units (sequence x 8 or 16 KV
// heads) are long, and a unit split over several CTAs ends in a merge at the
// CTA's tail.  Measured on GB300 (GQA 4): 64 units (batch 64, ~1900 tokens)
// 94.5 vs 86.8 us; 256 units about equal; 512 units 2.5 % faster; 1000 short
// units 24 % faster.  For MHA the per-head kernel computes 16 columns for one
// head, so the head-packed one wins earlier (128 units: 3 % faster).
int pa_decode_auto_kernel(const pa_cache_desc& cache, int32_t num_heads, int32_t num_seqs,
                          int32_t tokens_per_seq) {
  if (cache.num_kv_heads <= 0 || num_heads % cache.num_kv_heads != 0) return 1;
  const int group = num_heads / cache.num_kv_heads;
  const bool fp8 = cache.dtype == PA_KV_FP8_E4M3;
  if (pa::hp_supported(cache.head_dim, group, fp8, num_seqs, cache.num_kv_heads,
                       cache.block_size, tokens_per_seq)) {
    // Below 8 tokens per block a per-head tile would be gathered row by row
    // (256 bytes each); the head-packed kernel copies a block's rows of 8
    // or 16 heads (2 or 4 KiB per token) with one TMA box.
    if (cache.block_size < 8) return 3;
    const int64_t hp_units = (int64_t)num_seqs * (cache.num_kv_heads / (group >= 2 ? 8 : 16));
    if (!fp8 && (group == 1 ? 2 * hp_units >= num_sms() : hp_units >= 2 * num_sms())) return 3;
  }
  // Below 8 tokens per block the tensor-core kernel gathers rows with cp.async
  // and publishes a stage only once its own copies have landed; measured on
  // GB300 at block size 1 (batch-64 layer): 220.8 us (2.28 TB/s) against the
  // SIMT kernel's 136.4 us (3.7 TB/s), both reading the algorithmic bytes.  A
  // single token per sequence therefore takes the SIMT kernel there; several
  // tokens per sequence take the tensor-core kernel, which reads the context
  // once instead of once per token.
  if (pa::tc_supported(cache.head_dim, group, fp8, num_seqs, cache.block_size, tokens_per_seq) &&
      (cache.block_size >= 8 || tokens_per_seq > 1))
    return 2;
  return 1;
}

// pa_decode_ex's body.  prev_writes_cache_only: the kernel launched just
// before on `stream` is this library's cache write, so the tensor-core
// kernel may read its metadata (lengths, tables, q) while that write is still
// running and wait for it only before its first cache read.
static pa_status decode_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                             pa_cache_desc cache, const int32_t* block_tables,
                             int32_t max_blocks_per_seq, const int32_t* context_lens,
                             int32_t num_seqs, int32_t num_heads, float scale,
                             const float* k_scale, const float* v_scale, void* workspace,
                             size_t workspace_bytes, const pa_decode_opts* opts,
                             pa_stream_t stream, bool prev_writes_cache_only,
                             int32_t tokens_per_seq = 1, bool non_causal = false,
                             float* lse = nullptr) {
  const char* fn = "pa_decode";
  char buf[224];
  pa_status st = check_cache(cache, fn);
  if (st != PA_OK) return st;
  if ((st = check_scales(cache, k_scale, v_scale, fn)) != PA_OK) return st;
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_heads <= 0)
    return pa_fail(PA_ERR_INVALID, "pa_decode: bad num_seqs / max_blocks_per_seq / num_heads");
  if (num_seqs == 0) return PA_OK;
  if (num_seqs > 65535) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode: more than 65535 sequences");
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return pa_fail(PA_ERR_INVALID, "pa_decode: NULL pointer");
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return pa_fail(PA_ERR_INVALID, "pa_decode: misaligned pointer");
  if (num_heads % cache.num_kv_heads != 0)
    return pa_fail(PA_ERR_INVALID, "pa_decode: num_heads is not a multiple of num_kv_heads");
  const int group = num_heads / cache.num_kv_heads;
  if (group != 1 && group != 2 && group != 4 && group != 8) {
    snprintf(buf, sizeof buf, "pa_decode: GQA group %d unsupported (1, 2, 4 or 8)", group);
    return pa_fail(PA_ERR_UNSUPPORTED, buf);
  }
  if (!std::isfinite(scale)) return pa_fail(PA_ERR_INVALID, "pa_decode: scale is not finite");
  const int64_t max_ctx = (int64_t)max_blocks_per_seq * cache.block_size;
  if (max_ctx > INT32_MAX / 2)
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode: max_blocks_per_seq * block_size too large");
  const int kernel = opts ? opts->kernel : 0;
  if (kernel < 0 || kernel > 3) {
    snprintf(buf, sizeof buf, "pa_decode: kernel %d not available in this build", kernel);
    return pa_fail(PA_ERR_UNSUPPORTED, buf);
  }

  const bool fp8 = cache.dtype == PA_KV_FP8_E4M3;
  const int chosen =
      kernel != 0 ? kernel : pa_decode_auto_kernel(cache, num_heads, num_seqs, tokens_per_seq);
  const bool hp_ok = chosen == 3 &&
                     pa::hp_supported(cache.head_dim, group, fp8, num_seqs, cache.num_kv_heads,
                                      cache.block_size, tokens_per_seq);
  if (kernel == 3 && !hp_ok)
    return pa_fail(PA_ERR_UNSUPPORTED,
                   "pa_decode: head-packed kernel needs head_dim 128, GQA group 1, 2 or 4, "
                   "num_kv_heads a multiple of 16 (group 1) or 8, at most 1024 sequences and "
                   "one token per sequence");
  if (hp_ok) {
    const int nsm = num_sms();
    const size_t need = pa::hp_workspace_bytes(num_seqs, num_heads, nsm);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) {
      snprintf(buf, sizeof buf, "pa_decode: workspace of %zu bytes (256-byte aligned) needed",
               need);
      return pa_fail(PA_ERR_INVALID, buf);
    }
    pa::TcLaunch a{};
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.fp8 = fp8;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.workspace = workspace;
    a.num_seqs = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = cache.num_kv_heads;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = cache.num_blocks;
    a.block_size = cache.block_size;
    a.num_ctas = nsm;
    a.tokens_per_seq = 1;
    a.lse = lse;
    a.scale = scale;
    a.early_meta = prev_writes_cache_only;
    return cuda_status(pa::launch_decode_hp(a, reinterpret_cast<cudaStream_t>(stream)), fn);
  }
  const bool tc_ok = chosen == 2 && pa::tc_supported(cache.head_dim, group, fp8, num_seqs,
                                                      cache.block_size, tokens_per_seq);
  if (tokens_per_seq > 1 && !tc_ok)  // the SIMT kernel serves one token per sequence
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode: several tokens per sequence need the "
                                       "tensor-core kernel");
  if (chosen == 2) {
    if (!tc_ok)
      return pa_fail(PA_ERR_UNSUPPORTED,
                     "pa_decode: tensor-core kernel needs head_dim 128 "
                     "and at most 1024 sequences");
    const int nsm = num_sms();
    const size_t need = pa::tc_workspace_bytes(num_seqs, num_heads, max_ctx, nsm, tokens_per_seq);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) {
      snprintf(buf, sizeof buf, "pa_decode: workspace of %zu bytes (256-byte aligned) needed",
               need);
      return pa_fail(PA_ERR_INVALID, buf);
    }
    pa::TcLaunch a{};
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.fp8 = fp8;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.workspace = workspace;
    a.num_seqs = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = cache.num_kv_heads;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = cache.num_blocks;
    a.block_size = cache.block_size;
    a.num_ctas = nsm;
    a.tokens_per_seq = tokens_per_seq;
    a.non_causal = non_causal;
    a.lse = lse;
    a.scale = scale;
    a.early_meta = prev_writes_cache_only;
    return cuda_status(pa::launch_decode_tc(a, reinterpret_cast<cudaStream_t>(stream)), fn);
  }

  int ps = opts ? opts->partition_tokens : 0;
  if (ps != 0 && (!is_pow2(ps) || ps < pa::kMinPartition || ps > kMaxPartition)) {
    snprintf(buf, sizeof buf, "pa_decode: partition_tokens %d is not a power of two in [64, %d]",
             ps, kMaxPartition);
    return pa_fail(PA_ERR_INVALID, buf);
  }
  if (ps == 0) ps = auto_partition(num_seqs, cache.num_kv_heads, max_ctx);
  const WorkspaceLayout wl = workspace_layout(num_seqs, num_heads, cache.head_dim, max_ctx, ps);
  if (wl.total > 0) {
    if (!workspace || workspace_bytes < wl.total) {
      snprintf(buf, sizeof buf, "pa_decode: workspace of %zu bytes needed, %zu given", wl.total,
               workspace ? workspace_bytes : (size_t)0);
      return pa_fail(PA_ERR_INVALID, buf);
    }
    if (!aligned(workspace, 16)) return pa_fail(PA_ERR_INVALID, "pa_decode: misaligned workspace");
  }
  if (wl.parts > 65535)
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode: too many partitions for one grid");

  pa::DecodeParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.ws_o = wl.total ? static_cast<float*>(workspace) : nullptr;
  p.ws_ml = wl.total ? reinterpret_cast<float2*>(static_cast<char*>(workspace) + wl.ml_offset)
                     : nullptr;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.num_blocks = cache.num_blocks;
  p.block_size = cache.block_size;
  p.log2_block_size = ilog2(cache.block_size);
  p.num_kv_heads = cache.num_kv_heads;
  p.num_heads = num_heads;
  p.max_blocks = max_blocks_per_seq;
  p.partition_tokens = ps;
  p.max_parts = (int32_t)wl.parts;
  p.scale_log2 = scale * 1.4426950408889634f;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cache.dtype == PA_KV_FP8_E4M3
                      ? pa::launch_decode_simt_fp8(p, cache.head_dim, group, num_seqs, s)
                      : pa::launch_decode_simt_bf16(p, cache.head_dim, group, num_seqs, s);
  if (e != cudaSuccess) return cuda_status(e, fn);
  if (wl.parts > 1) {
    e = pa::launch_decode_reduce(p, cache.head_dim, num_seqs, s);
    if (e != cudaSuccess) return cuda_status(e, "pa_decode (combine)");
  }
  return PA_OK;
}

extern "C" {

pa_status pa_decode_ex(void* out, const void* q, const void* k_cache, const void* v_cache,
                       pa_cache_desc cache, const int32_t* block_tables,
                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                       int32_t num_seqs, int32_t num_heads, float scale, const float* k_scale,
                       const float* v_scale, void* workspace, size_t workspace_bytes,
                       const pa_decode_opts* opts, pa_stream_t stream) {
  return decode_impl(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_heads, scale, k_scale, v_scale, workspace,
                     workspace_bytes, opts, stream, false);
}

pa_status pa_write_and_decode(const void* key, const void* value, const int32_t* slot_mapping,
                              int32_t num_tokens, void* out, const void* q, void* k_cache,
                              void* v_cache, pa_cache_desc cache, const int32_t* block_tables,
                              int32_t max_blocks_per_seq, const int32_t* context_lens,
                              int32_t num_seqs, int32_t num_heads, float scale,
                              const float* k_scale, const float* v_scale, void* workspace,
                              size_t workspace_bytes, pa_stream_t stream) {
  pa_status st = pa_reshape_and_cache(key, value, k_cache, v_cache, cache, slot_mapping,
                                      num_tokens, k_scale, v_scale, stream);
  if (st != PA_OK) return st;
  return decode_impl(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_heads, scale, k_scale, v_scale, workspace,
                     workspace_bytes, nullptr, stream, num_tokens > 0);
}

pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    pa_cache_desc cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* context_lens, int32_t num_seqs, int32_t num_heads, float scale,
                    const float* k_scale, const float* v_scale, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream) {
  return pa_decode_ex(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                      context_lens, num_seqs, num_heads, scale, k_scale, v_scale, workspace,
                      workspace_bytes, nullptr, stream);
}

pa_status pa_copy_blocks(void* k_cache, void* v_cache, pa_cache_desc cache,
                         const int32_t* block_pairs, int32_t num_pairs, pa_stream_t stream) {
  const char* fn = "pa_copy_blocks";
  pa_status st = check_cache(cache, fn);
  if (st != PA_OK) return st;
  if (num_pairs < 0) return pa_fail(PA_ERR_INVALID, "pa_copy_blocks: num_pairs < 0");
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !block_pairs)
    return pa_fail(PA_ERR_INVALID, "pa_copy_blocks: NULL pointer");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_pairs, 4))
    return pa_fail(PA_ERR_INVALID, "pa_copy_blocks: misaligned pointer");
  const int64_t elem = cache.dtype == PA_KV_FP8_E4M3 ? 1 : 2;
  const int64_t block_bytes =
      (int64_t)cache.block_size * cache.num_kv_heads * cache.head_dim * elem;
  return cuda_status(pa::launch_copy_blocks(k_cache, v_cache, block_bytes, cache.num_blocks,
                                            block_pairs, num_pairs,
                                            reinterpret_cast<cudaStream_t>(stream)),
                     fn);
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

size_t pa_varlen_workspace_size(int32_t num_tokens, int32_t num_heads, int32_t head_dim,
                                int32_t max_blocks_per_seq, int32_t block_size) {
  if (num_tokens <= 0 || num_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 ||
      block_size <= 0)
    return 0;
  const size_t meta = align256((size_t)num_tokens * max_blocks_per_seq * 4) +
                      align256((size_t)num_tokens * 4);
  // the decode part may legitimately need no scratch (no split partitions)
  return meta + pa_decode_workspace_size(num_tokens, num_heads, head_dim, max_blocks_per_seq,
                                         block_size);
}

}  // extern "C"

// Method 1 of pa_varlen_attention: one virtual decode sequence per new token
// (its request's table, its causal length).  Tokens of requests with
// tile_min or more new tokens (tile_min > 0) get empty virtual sequences.
static pa_status varlen_per_token(void* out, const void* q, const void* k_cache,
                                  const void* v_cache, pa_cache_desc cache,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* seq_lens, const int32_t* query_start_loc,
                                  int32_t num_seqs, int32_t num_tokens, int32_t num_heads,
                                  float scale, const float* k_scale, const float* v_scale,
                                  void* workspace, size_t workspace_bytes, pa_stream_t stream,
                                  int tile_min) {
  char* ws = static_cast<char*>(workspace);
  int32_t* vtables = reinterpret_cast<int32_t*>(ws);
  const size_t tb = align256((size_t)num_tokens * max_blocks_per_seq * 4);
  int32_t* vlens = reinterpret_cast<int32_t*>(ws + tb);
  const size_t meta = tb + align256((size_t)num_tokens * 4);
  cudaError_t e = pa::launch_varlen_meta(block_tables, max_blocks_per_seq, cache.block_size,
                                         seq_lens, query_start_loc, 0, num_seqs, num_tokens,
                                         vtables, vlens, reinterpret_cast<cudaStream_t>(stream),
                                         tile_min);
  if (e != cudaSuccess) return cuda_status(e, "pa_varlen_attention");
  return decode_impl(out, q, k_cache, v_cache, cache, vtables, max_blocks_per_seq, vlens,
                     num_tokens, num_heads, scale, k_scale, v_scale, ws + meta,
                     workspace_bytes - meta, nullptr, stream, false);
}

extern "C" {

pa_status pa_varlen_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                              pa_cache_desc cache, const int32_t* block_tables,
                              int32_t max_blocks_per_seq, const int32_t* seq_lens,
                              const int32_t* query_start_loc, int32_t num_seqs,
                              int32_t num_tokens, int32_t num_heads, float scale,
                              const float* k_scale, const float* v_scale, void* workspace,
                              size_t workspace_bytes, pa_stream_t stream) {
  return pa_varlen_attention_ex(out, q, k_cache, v_cache, cache, block_tables,
                                max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                                num_tokens, num_heads, scale, k_scale, v_scale, 0, workspace,
                                workspace_bytes, stream);
}

pa_status pa_varlen_attention_ex(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, pa_cache_desc cache,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* seq_lens, const int32_t* query_start_loc,
                                 int32_t num_seqs, int32_t num_tokens, int32_t num_heads,
                                 float scale, const float* k_scale, const float* v_scale,
                                 int32_t method, void* workspace, size_t workspace_bytes,
                                 pa_stream_t stream) {
  const char* fn = "pa_varlen_attention";
  if (method < 0 || method > 2)
    return pa_fail(PA_ERR_INVALID, "pa_varlen_attention: method must be 0, 1 or 2");
  char buf[192];
  if (num_seqs < 0 || num_tokens < 0 || max_blocks_per_seq <= 0)
    return pa_fail(PA_ERR_INVALID, "pa_varlen_attention: bad sizes");
  if (num_tokens == 0) return PA_OK;
  if (num_seqs == 0) return pa_fail(PA_ERR_INVALID, "pa_varlen_attention: tokens without requests");
  if (num_tokens > 65535)
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_varlen_attention: more than 65535 new tokens");
  if (!block_tables || !seq_lens || !query_start_loc || !workspace)
    return pa_fail(PA_ERR_INVALID, "pa_varlen_attention: NULL pointer");
  if (!aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(query_start_loc, 4) ||
      !aligned(workspace, 256))
    return pa_fail(PA_ERR_INVALID, "pa_varlen_attention: misaligned pointer");
  pa_status st = check_cache(cache, fn);
  if (st != PA_OK) return st;
  if ((st = check_scales(cache, k_scale, v_scale, fn)) != PA_OK) return st;
  const size_t need = pa_varlen_workspace_size(num_tokens, num_heads, cache.head_dim,
                                               max_blocks_per_seq, cache.block_size);
  if (need == 0 || workspace_bytes < need) {
    snprintf(buf, sizeof buf, "pa_varlen_attention: workspace of %zu bytes needed", need);
    return pa_fail(PA_ERR_INVALID, buf);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool fp8 = cache.dtype == PA_KV_FP8_E4M3;
  const int group = num_heads % cache.num_kv_heads == 0 ? num_heads / cache.num_kv_heads : 0;
  const bool tiles_fit = group > 0 && scale > 0.f &&
                         pa::prefill_supported(cache.head_dim, group, fp8, num_seqs,
                                               cache.block_size);
  if (method == 2 && !tiles_fit)
    return pa_fail(PA_ERR_UNSUPPORTED,
                   "pa_varlen_attention: prefill tiles need head_dim 128, GQA "
                   "group 1, 2, 4 or 8, block_size >= 8, at most 256 requests and scale > 0");
  // Method 0 with tiles available: when the step adds 16 or more tokens per
  // request on average, the tiles serve every request; otherwise requests
  // adding 16 or more tokens go to the tiles and the others to one decode per
  // new token (the long requests' tokens are empty virtual sequences there,
  // zero rows the tiles then overwrite), so one long prefill among many
  // single-token decodes no longer runs token by token.
  const bool tiles_all = method == 2 || (method == 0 && tiles_fit && num_tokens >= 16 * num_seqs);
  const bool tiles_mixed = !tiles_all && method == 0 && tiles_fit && num_tokens >= kTileMinTokens;
  if (tiles_all || tiles_mixed) {
    if (!out || !q || !k_cache || !v_cache)
      return pa_fail(PA_ERR_INVALID, "pa_varlen_attention: NULL pointer");
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
      return pa_fail(PA_ERR_INVALID, "pa_varlen_attention: misaligned pointer");
    if (!std::isfinite(scale)) return pa_fail(PA_ERR_INVALID, "pa_varlen_attention: scale is not finite");
    pa::PrefillLaunch a{};
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.query_start_loc = query_start_loc;
    a.workspace = workspace;
    a.num_seqs = num_seqs;
    a.num_tokens = num_tokens;
    a.num_heads = num_heads;
    a.num_kv_heads = cache.num_kv_heads;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = cache.num_blocks;
    a.block_size = cache.block_size;
    a.num_ctas = num_sms();
    a.scale = scale;
    a.min_tokens = tiles_all ? 0 : kTileMinTokens;
    a.fp8 = fp8;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    if (tiles_all) return cuda_status(pa::launch_prefill_tc(a, s), fn);
    // the short requests first (below), then the tiles on the same stream;
    // word 0 is the tiles' error word once the decode has used the metadata
    st = varlen_per_token(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                          seq_lens, query_start_loc, num_seqs, num_tokens, num_heads, scale,
                          k_scale, v_scale, workspace, workspace_bytes, stream, kTileMinTokens);
    if (st != PA_OK) return st;
    cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return cuda_status(e, fn);
    return cuda_status(pa::launch_prefill_tc(a, s), fn);
  }
  return varlen_per_token(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                          seq_lens, query_start_loc, num_seqs, num_tokens, num_heads, scale,
                          k_scale, v_scale, workspace, workspace_bytes, stream, 0);
}

size_t pa_decode_multi_workspace_size(int32_t num_seqs, int32_t tokens_per_seq,
                                      int32_t num_heads, int32_t head_dim,
                                      int32_t max_blocks_per_seq, int32_t block_size) {
  if (num_seqs <= 0 || tokens_per_seq <= 0 || num_heads <= 0 || head_dim <= 0 ||
      max_blocks_per_seq <= 0 || block_size <= 0)
    return 0;
  const int64_t max_ctx = (int64_t)max_blocks_per_seq * block_size;
  // either path: one pass over (token, head) columns, or one decode per token
  const size_t tc = pa::tc_workspace_bytes(num_seqs, num_heads, max_ctx, num_sms(),
                                           tokens_per_seq);
  const size_t per_token = pa_varlen_workspace_size(num_seqs * tokens_per_seq, num_heads,
                                                    head_dim, max_blocks_per_seq, block_size);
  return tc > per_token ? tc : per_token;
}

pa_status pa_decode_multi(void* out, const void* q, const void* k_cache, const void* v_cache,
                          pa_cache_desc cache, const int32_t* block_tables,
                          int32_t max_blocks_per_seq, const int32_t* context_lens,
                          int32_t num_seqs, int32_t tokens_per_seq, int32_t num_heads,
                          float scale, const float* k_scale, const float* v_scale,
                          void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  const char* fn = "pa_decode_multi";
  if (tokens_per_seq <= 0) return pa_fail(PA_ERR_INVALID, "pa_decode_multi: tokens_per_seq <= 0");
  if (tokens_per_seq == 1)
    return decode_impl(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, num_heads, scale, k_scale, v_scale, workspace,
                       workspace_bytes, nullptr, stream, false);
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_heads <= 0)
    return pa_fail(PA_ERR_INVALID, "pa_decode_multi: bad sizes");
  if (num_seqs == 0) return PA_OK;
  pa_status st = check_cache(cache, fn);
  if (st != PA_OK) return st;
  if (num_heads % cache.num_kv_heads != 0)
    return pa_fail(PA_ERR_INVALID, "pa_decode_multi: num_heads is not a multiple of num_kv_heads");
  if ((int64_t)num_seqs * tokens_per_seq > 65535)
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode_multi: more than 65535 new tokens");
  const int group = num_heads / cache.num_kv_heads;
  if (pa::tc_supported(cache.head_dim, group, cache.dtype == PA_KV_FP8_E4M3, num_seqs,
                       cache.block_size, tokens_per_seq))
    return decode_impl(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, num_heads, scale, k_scale, v_scale, workspace,
                       workspace_bytes, nullptr, stream, false, tokens_per_seq);
  // otherwise one virtual decode sequence per new token
  const int32_t n = num_seqs * tokens_per_seq;
  if (!block_tables || !context_lens || !workspace)
    return pa_fail(PA_ERR_INVALID, "pa_decode_multi: NULL pointer");
  if (!aligned(workspace, 256)) return pa_fail(PA_ERR_INVALID, "pa_decode_multi: misaligned workspace");
  const size_t need = pa_varlen_workspace_size(n, num_heads, cache.head_dim, max_blocks_per_seq,
                                               cache.block_size);
  if (workspace_bytes < need) {
    char buf[160];
    snprintf(buf, sizeof buf, "pa_decode_multi: workspace of %zu bytes needed", need);
    return pa_fail(PA_ERR_INVALID, buf);
  }
  char* ws = static_cast<char*>(workspace);
  int32_t* vtables = reinterpret_cast<int32_t*>(ws);
  const size_t tb = align256((size_t)n * max_blocks_per_seq * 4);
  int32_t* vlens = reinterpret_cast<int32_t*>(ws + tb);
  const size_t meta = tb + align256((size_t)n * 4);
  cudaError_t e = pa::launch_varlen_meta(block_tables, max_blocks_per_seq, cache.block_size,
                                         context_lens, nullptr, tokens_per_seq, num_seqs, n,
                                         vtables, vlens, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e, fn);
  return decode_impl(out, q, k_cache, v_cache, cache, vtables, max_blocks_per_seq, vlens, n,
                     num_heads, scale, k_scale, v_scale, ws + meta, workspace_bytes - meta,
                     nullptr, stream, false);
}

size_t pa_decode_shared_prefix_workspace_size(int32_t num_seqs, int32_t group_size,
                                              int32_t num_heads, int32_t head_dim,
                                              int32_t max_blocks_per_seq, int32_t block_size) {
  if (num_seqs <= 0 || group_size <= 0 || num_seqs % group_size || num_heads <= 0 ||
      head_dim <= 0 || max_blocks_per_seq <= 0 || block_size <= 0)
    return 0;
  const int64_t S = num_seqs, V = num_seqs / group_size, rows = S * num_heads;
  const int64_t max_ctx = (int64_t)max_blocks_per_seq * block_size;
  size_t off = align256((size_t)V * max_blocks_per_seq * 4) + align256((size_t)V * 4) +
               align256((size_t)S * max_blocks_per_seq * 4) + align256((size_t)S * 4);
  off += 2 * (align256((size_t)rows * head_dim * 2) + align256((size_t)rows * 4));
  const size_t pre = pa::tc_workspace_bytes(V, num_heads, max_ctx, num_sms(), group_size);
  const size_t suf = pa_decode_workspace_size(num_seqs, num_heads, head_dim, max_blocks_per_seq,
                                              block_size);
  return off + (pre > suf ? pre : suf);
}

pa_status pa_decode_shared_prefix(void* out, const void* q, const void* k_cache,
                                  const void* v_cache, pa_cache_desc cache,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens, int32_t num_seqs,
                                  int32_t group_size, int32_t num_heads, float scale,
                                  const float* k_scale, const float* v_scale, void* workspace,
                                  size_t workspace_bytes, pa_stream_t stream) {
  const char* fn = "pa_decode_shared_prefix";
  if (num_seqs < 0 || group_size <= 0 || max_blocks_per_seq <= 0 || num_heads <= 0)
    return pa_fail(PA_ERR_INVALID, "pa_decode_shared_prefix: bad sizes");
  if (num_seqs == 0) return PA_OK;
  if (num_seqs % group_size)
    return pa_fail(PA_ERR_INVALID, "pa_decode_shared_prefix: num_seqs is not a multiple of group_size");
  pa_status st = check_cache(cache, fn);
  if (st != PA_OK) return st;
  if (num_heads % cache.num_kv_heads != 0)
    return pa_fail(PA_ERR_INVALID, "pa_decode_shared_prefix: num_heads is not a multiple of num_kv_heads");
  const int gq = num_heads / cache.num_kv_heads;
  const bool fp8 = cache.dtype == PA_KV_FP8_E4M3;
  const int V = num_seqs / group_size;
  const bool tc = pa::tc_supported(cache.head_dim, gq, fp8, V, cache.block_size, group_size) &&
                  pa::tc_supported(cache.head_dim, gq, fp8, num_seqs, cache.block_size, 1);
  if (group_size == 1 || !tc)  // nothing to share, or the passes need the tensor cores
    return decode_impl(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, num_heads, scale, k_scale, v_scale, workspace,
                       workspace_bytes, nullptr, stream, false);
  if (!out || !q || !block_tables || !context_lens || !workspace)
    return pa_fail(PA_ERR_INVALID, "pa_decode_shared_prefix: NULL pointer");
  if (!aligned(workspace, 256) || !aligned(out, 16))
    return pa_fail(PA_ERR_INVALID, "pa_decode_shared_prefix: misaligned pointer");
  const size_t need = pa_decode_shared_prefix_workspace_size(
      num_seqs, group_size, num_heads, cache.head_dim, max_blocks_per_seq, cache.block_size);
  if (workspace_bytes < need) {
    char buf[160];
    snprintf(buf, sizeof buf, "pa_decode_shared_prefix: workspace of %zu bytes needed", need);
    return pa_fail(PA_ERR_INVALID, buf);
  }
  const int64_t rows = (int64_t)num_seqs * num_heads;
  char* ws = static_cast<char*>(workspace);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = ws + off;
    off += align256(bytes);
    return p;
  };
  int32_t* ptables = reinterpret_cast<int32_t*>(take((size_t)V * max_blocks_per_seq * 4));
  int32_t* plens = reinterpret_cast<int32_t*>(take((size_t)V * 4));
  int32_t* stables = reinterpret_cast<int32_t*>(take((size_t)num_seqs * max_blocks_per_seq * 4));
  int32_t* slens = reinterpret_cast<int32_t*>(take((size_t)num_seqs * 4));
  void* o_pre = take((size_t)rows * cache.head_dim * 2);
  float* l_pre = reinterpret_cast<float*>(take((size_t)rows * 4));
  void* o_suf = take((size_t)rows * cache.head_dim * 2);
  float* l_suf = reinterpret_cast<float*>(take((size_t)rows * 4));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = pa::launch_cascade_meta(block_tables, max_blocks_per_seq, cache.block_size,
                                          context_lens, num_seqs, group_size, ptables, plens,
                                          stables, slens, s);
  if (e != cudaSuccess) return cuda_status(e, fn);
  // pass 1: each group's shared prefix, read once, its members' queries as columns
  st = decode_impl(o_pre, q, k_cache, v_cache, cache, ptables, max_blocks_per_seq, plens, V,
                   num_heads, scale, k_scale, v_scale, ws + off, workspace_bytes - off, nullptr,
                   stream, false, group_size, true, l_pre);
  if (st != PA_OK) return st;
  // pass 2: every sequence's own blocks after the prefix
  st = decode_impl(o_suf, q, k_cache, v_cache, cache, stables, max_blocks_per_seq, slens,
                   num_seqs, num_heads, scale, k_scale, v_scale, ws + off, workspace_bytes - off,
                   nullptr, stream, false, 1, false, l_suf);
  if (st != PA_OK) return st;
  return cuda_status(pa::launch_lse_merge(o_pre, l_pre, o_suf, l_suf, out, rows, cache.head_dim, s),
                     fn);
}

pa_status pa_swap_blocks(void* dst_k, void* dst_v, int32_t dst_num_blocks, const void* src_k,
                         const void* src_v, int32_t src_num_blocks, pa_cache_desc block_shape,
                         const int32_t* block_pairs, int32_t num_pairs, pa_stream_t stream) {
  const char* fn = "pa_swap_blocks";
  pa_cache_desc c = block_shape;
  c.num_blocks = dst_num_blocks;
  pa_status st = check_cache(c, fn);
  if (st != PA_OK) return st;
  c.num_blocks = src_num_blocks;
  if ((st = check_cache(c, fn)) != PA_OK) return st;
  if (num_pairs < 0) return pa_fail(PA_ERR_INVALID, "pa_swap_blocks: num_pairs < 0");
  if (num_pairs == 0) return PA_OK;
  if (!dst_k || !dst_v || !src_k || !src_v || !block_pairs)
    return pa_fail(PA_ERR_INVALID, "pa_swap_blocks: NULL pointer");
  if (!aligned(dst_k, 16) || !aligned(dst_v, 16) || !aligned(src_k, 16) || !aligned(src_v, 16) ||
      !aligned(block_pairs, 4))
    return pa_fail(PA_ERR_INVALID, "pa_swap_blocks: misaligned pointer");
  const int64_t elem = block_shape.dtype == PA_KV_FP8_E4M3 ? 1 : 2;
  const int64_t block_bytes =
      (int64_t)block_shape.block_size * block_shape.num_kv_heads * block_shape.head_dim * elem;
  return cuda_status(pa::launch_copy_blocks_between(dst_k, dst_v, dst_num_blocks, src_k, src_v,
                                                    src_num_blocks, block_bytes, block_pairs,
                                                    num_pairs,
                                                    reinterpret_cast<cudaStream_t>(stream)),
                     fn);
}

pa_status pa_step_prepare(int32_t* block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                          int32_t block_size, int32_t* context_lens,
                          const int32_t* table_updates, int32_t num_updates, int32_t advance,
                          int32_t* slot_mapping, pa_stream_t stream) {
  const char* fn = "pa_step_prepare";
  if (num_seqs < 0 || num_updates < 0 || max_blocks_per_seq <= 0 || block_size <= 0)
    return pa_fail(PA_ERR_INVALID, "pa_step_prepare: bad sizes");
  if (advance < 0) return pa_fail(PA_ERR_INVALID, "pa_step_prepare: advance < 0");
  if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX)
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_step_prepare: max_blocks_per_seq * block_size too large");
  if (num_seqs == 0) return PA_OK;
  if (!block_tables || !context_lens || !slot_mapping || (num_updates > 0 && !table_updates))
    return pa_fail(PA_ERR_INVALID, "pa_step_prepare: NULL pointer");
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(slot_mapping, 4) ||
      (table_updates && !aligned(table_updates, 4)))
    return pa_fail(PA_ERR_INVALID, "pa_step_prepare: misaligned pointer");
  return cuda_status(pa::launch_step_prepare(block_tables, max_blocks_per_seq, block_size,
                                             context_lens, num_seqs, table_updates, num_updates,
                                             advance, slot_mapping,
                                             reinterpret_cast<cudaStream_t>(stream)),
                     fn);
}

}  // extern "C"
