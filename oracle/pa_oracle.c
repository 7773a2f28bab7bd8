/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for the paged-KV decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file.  Only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header, table or helper with
 * the CUDA path.
 *
 * What it computes, and where each step is defined:
 *
 *  - Cache write ("reshape_and_cache"): the new token i is stored at flat
 *    slot slot_mapping[i] of the pool viewed as [num_blocks*block_size,
 *    H_kv, d].  "Paged KV cache" (ai-infra-handbooks), PagedKVCache.write;
 *    "4.6 PagedAttention & KV-Cache Memory Management" (llm-stack-book),
 *    section "From Python bookkeeping to the tensors the kernel actually
 *    takes" (a single index copy over the flattened pool).  A negative slot
 *    means "padding token, write nothing" (a reading: the pages are silent).
 *  - fp8 KV ("--kv-cache-dtype fp8" halves b, llm-stack-book §4.6, section
 *    "The libraries that implement this"): e4m3 with one fp32 scale per
 *    tensor.  enc(x) = e4m3_rne_satfinite((float)x / scale), dec(c) = c*scale.
 *    The e4m3 format (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
 *    no infinities, NaN = S.1111.111, largest finite 448, subnormals down to
 *    2^-9) is the OCP 8-bit floating point specification's E4M3.
 *  - Block copy for copy-on-write: dst block := src block, K and V.
 *    llm-stack-book §4.6, section "Copy-on-write for shared prefixes"
 *    (cow_append: "kernel copies block contents src->dst").
 *  - Decode attention: for sequence i with context length n (valid tokens
 *    after this step's write), gather its K and V through the block table
 *    into contiguous fp64 arrays, then for each query head h with KV head
 *    g = h / G compute softmax(scale * q_h . K_g^T) V_g the textbook way
 *    (max, exp, sum, divide).  "Paged KV cache", PagedKVCache.gather and
 *    paged_attention (gather, repeat_interleave for GQA, einsum, softmax);
 *    llm-stack-book §4.6, section "The PagedAttention Kernel" (the math is
 *    unchanged; the block table is only an indirection).  n == 0 gives a
 *    zero output row (a reading: the pages are silent).
 *  - Varlen causal attention (several new tokens per request: multi-token
 *    decode, chunked and full prefill).  "Paged KV cache", section "Paged
 *    attention": request r's new tokens are queries qsl[r]..qsl[r+1]-1 and
 *    are the last num_new of its seq_len context tokens, so new token j sits
 *    at position seq_len - num_new + j and attends to positions 0 through
 *    that one.  Per (request, KV head): gather the request's rows through its
 *    block table, then for each new token and each query head of the group
 *    a textbook softmax over the visible positions.  A request whose
 *    num_new exceeds seq_len has no valid position for its first tokens; its
 *    rows are defined as zero (a reading: the pages are silent).
 *
 * No online softmax, no partitions, no blocking: each result is the plain
 * definition, written so it can be read against the pages.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_KV_BF16 0
#define ORC_KV_FP8_E4M3 1

/* ---- element formats ---------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double orc_bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP E4M3 decode: exponent field E (bias 7), mantissa field M (3 bits).
 * E == 0 is subnormal: M/8 * 2^-6.  E == 15, M == 7 is NaN (no infinities). */
double orc_e4m3_to_double(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m, -9); /* (m/8) * 2^-6 */
  else
    mag = ldexp(8.0 + (double)m, e - 7 - 3); /* (1 + m/8) * 2^(e-7) */
  return sign ? -mag : mag;
}

/* OCP E4M3 encode of a binary32 value: round to nearest, ties to even,
 * saturating to the largest finite magnitude (448) instead of overflowing.
 * NaN maps to the canonical NaN code 0x7F. */
uint8_t orc_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a > 448.0) return sign | 0x7E; /* saturate (also covers +-inf) */
  if (a < 0.015625) {                /* below the smallest normal 2^-6 */
    double q = a * 512.0;            /* units of the subnormal step 2^-9, exact */
    double r = rint(q);              /* default rounding mode: ties to even */
    /* r == 8 lands exactly on the smallest normal, whose code is 0x08 */
    return sign | (uint8_t)r;
  }
  int k;
  frexp(a, &k); /* a = f * 2^k, f in [0.5, 1) */
  int e = k - 1; /* a in [2^e, 2^(e+1)), e in [-6, 8] */
  double q = ldexp(a, 3 - e); /* in [8, 16): 1.mmm scaled by 8, exact */
  double r = rint(q);
  if (r == 16.0) { /* rounded up into the next binade */
    e += 1;
    r = 8.0;
  }
  if (e > 8) return sign | 0x7E; /* cannot happen for a <= 448 */
  return sign | (uint8_t)(((e + 7) << 3) | ((int)r - 8));
}

void orc_e4m3_encode_array(const float* x, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(x[i]);
}

void orc_e4m3_decode_array(const uint8_t* c, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_to_double(c[i]);
}

/* ---- cache write -------------------------------------------------------- */

/* key, value: [num_tokens, H_kv, d] bf16 bit patterns.
 * k_cache, v_cache: [num_blocks, block_size, H_kv, d] of bf16 (uint16) or
 * e4m3 (uint8).  Returns 0, or -1 if a slot is outside the pool. */
int orc_reshape_and_cache(const uint16_t* key, const uint16_t* value,
                          int32_t num_tokens, int32_t num_kv_heads,
                          int32_t head_dim, void* k_cache, void* v_cache,
                          int32_t num_blocks, int32_t block_size,
                          int32_t kv_dtype, const int32_t* slot_mapping,
                          float k_scale, float v_scale) {
  int64_t row = (int64_t)num_kv_heads * head_dim; /* elements per slot */
  int64_t num_slots = (int64_t)num_blocks * block_size;
  for (int32_t i = 0; i < num_tokens; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot < 0) continue; /* padding token: nothing is written */
    if (slot >= num_slots) return -1;
    /* the flat view [num_blocks*block_size, H_kv, d]: blk = slot / B and
     * off = slot % B address the same element as slot * row */
    int64_t dst = slot * row;
    int64_t src = (int64_t)i * row;
    if (kv_dtype == ORC_KV_BF16) {
      memcpy((uint16_t*)k_cache + dst, key + src, (size_t)row * 2);
      memcpy((uint16_t*)v_cache + dst, value + src, (size_t)row * 2);
    } else {
      for (int64_t e = 0; e < row; ++e) {
        float kf = (float)orc_bf16_to_double(key[src + e]);
        float vf = (float)orc_bf16_to_double(value[src + e]);
        /* IEEE binary32 division, correctly rounded, then E4M3 rounding */
        ((uint8_t*)k_cache)[dst + e] = orc_e4m3_encode(kf / k_scale);
        ((uint8_t*)v_cache)[dst + e] = orc_e4m3_encode(vf / v_scale);
      }
    }
  }
  return 0;
}

/* ---- block copy (copy-on-write) ----------------------------------------- */

/* pairs: [num_pairs, 2] (src, dst) physical block ids. */
int orc_copy_blocks(void* k_cache, void* v_cache, int32_t num_blocks,
                    int64_t block_bytes, const int32_t* pairs,
                    int32_t num_pairs) {
  for (int32_t p = 0; p < num_pairs; ++p) {
    int32_t src = pairs[2 * p], dst = pairs[2 * p + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks)
      return -1;
    memmove((char*)k_cache + (int64_t)dst * block_bytes,
            (char*)k_cache + (int64_t)src * block_bytes, (size_t)block_bytes);
    memmove((char*)v_cache + (int64_t)dst * block_bytes,
            (char*)v_cache + (int64_t)src * block_bytes, (size_t)block_bytes);
  }
  return 0;
}

/* ---- decode attention --------------------------------------------------- */

typedef struct {
  double* out;                 /* [num_seqs, H_q, d] fp64 */
  const uint16_t* q;           /* [num_seqs, H_q, d] bf16 */
  const void* k_cache;         /* [num_blocks, B, H_kv, d] */
  const void* v_cache;
  int32_t num_blocks, block_size, num_kv_heads, head_dim, kv_dtype;
  const int32_t* block_tables; /* [num_seqs, max_blocks] */
  int32_t max_blocks;
  const int32_t* context_lens; /* [num_seqs] */
  int32_t num_seqs, num_heads;
  double scale, k_scale, v_scale;
} orc_decode_args;

static double cache_elem(const orc_decode_args* a, const void* cache,
                         int64_t idx, double kv_scale) {
  if (a->kv_dtype == ORC_KV_BF16)
    return orc_bf16_to_double(((const uint16_t*)cache)[idx]);
  return orc_e4m3_to_double(((const uint8_t*)cache)[idx]) * kv_scale;
}

/* One (sequence, KV head) unit: all G query heads of the group.
 * Returns 0, or -1 on an out-of-range block id / context length. */
static int decode_unit(const orc_decode_args* a, int32_t seq, int32_t g) {
  const int32_t H = a->num_heads, Hkv = a->num_kv_heads, d = a->head_dim;
  const int32_t B = a->block_size, G = H / Hkv;
  const int32_t n = a->context_lens[seq];
  double* out0 = a->out + ((int64_t)seq * H + (int64_t)g * G) * d;
  if (n <= 0) { /* empty context: defined as a zero row */
    memset(out0, 0, sizeof(double) * (size_t)G * d);
    return n == 0 ? 0 : -1;
  }
  if ((int64_t)n > (int64_t)a->max_blocks * B) return -1;

  /* 1. gather: K[t], V[t] for t < n, through the block table */
  double* K = (double*)malloc(sizeof(double) * (size_t)n * d);
  double* V = (double*)malloc(sizeof(double) * (size_t)n * d);
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  if (!K || !V || !s) {
    free(K); free(V); free(s);
    return -2;
  }
  const int32_t* table = a->block_tables + (int64_t)seq * a->max_blocks;
  for (int32_t t = 0; t < n; ++t) {
    int32_t phys = table[t / B];
    if (phys < 0 || phys >= a->num_blocks) {
      free(K); free(V); free(s);
      return -1;
    }
    int64_t base = (((int64_t)phys * B + (t % B)) * Hkv + g) * d;
    for (int32_t e = 0; e < d; ++e) {
      K[(int64_t)t * d + e] = cache_elem(a, a->k_cache, base + e, a->k_scale);
      V[(int64_t)t * d + e] = cache_elem(a, a->v_cache, base + e, a->v_scale);
    }
  }

  /* 2. per query head of the group: textbook softmax(scale q K^T) V */
  for (int32_t j = 0; j < G; ++j) {
    const int32_t h = g * G + j; /* kv head of h is h / G == g */
    const uint16_t* qh = a->q + ((int64_t)seq * H + h) * d;
    double m = -INFINITY;
    for (int32_t t = 0; t < n; ++t) {
      double dot = 0.0;
      for (int32_t e = 0; e < d; ++e)
        dot += orc_bf16_to_double(qh[e]) * K[(int64_t)t * d + e];
      s[t] = a->scale * dot;
      if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int32_t t = 0; t < n; ++t) {
      s[t] = exp(s[t] - m);
      l += s[t];
    }
    double* o = out0 + (int64_t)j * d;
    for (int32_t e = 0; e < d; ++e) {
      double acc = 0.0;
      for (int32_t t = 0; t < n; ++t) acc += s[t] * V[(int64_t)t * d + e];
      o[e] = acc / l;
    }
  }
  free(K); free(V); free(s);
  return 0;
}

typedef struct {
  const orc_decode_args* a;
  const int32_t* units; /* [n_units, 2] (seq, kv head) */
  int32_t n_units;
  int32_t stride, first;
  int status;
} orc_worker;

static void* worker_main(void* p) {
  orc_worker* w = (orc_worker*)p;
  for (int32_t u = w->first; u < w->n_units; u += w->stride) {
    int st = decode_unit(w->a, w->units[2 * u], w->units[2 * u + 1]);
    if (st != 0) w->status = st;
  }
  return NULL;
}

/* Decode the listed (seq, kv head) units; units == NULL means all of them.
 * nthreads > 1 spreads the same per-unit function over POSIX threads (used
 * only to time a CPU baseline); nthreads <= 1 is a plain loop.
 * Returns 0 on success, -1 on a bad id or length, -2 on host OOM. */
int orc_decode(double* out, const uint16_t* q, const void* k_cache,
               const void* v_cache, int32_t num_blocks, int32_t block_size,
               int32_t num_kv_heads, int32_t head_dim, int32_t kv_dtype,
               const int32_t* block_tables, int32_t max_blocks,
               const int32_t* context_lens, int32_t num_seqs,
               int32_t num_heads, double scale, double k_scale,
               double v_scale, const int32_t* units, int32_t n_units,
               int32_t nthreads) {
  if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return -1;
  orc_decode_args a = {out, q, k_cache, v_cache, num_blocks, block_size,
                       num_kv_heads, head_dim, kv_dtype, block_tables,
                       max_blocks, context_lens, num_seqs, num_heads,
                       scale, k_scale, v_scale};
  int32_t* all = NULL;
  if (units == NULL) {
    n_units = num_seqs * num_kv_heads;
    all = (int32_t*)malloc(sizeof(int32_t) * 2 * (size_t)(n_units > 0 ? n_units : 1));
    if (!all) return -2;
    for (int32_t i = 0; i < num_seqs; ++i)
      for (int32_t g = 0; g < num_kv_heads; ++g) {
        all[2 * (i * num_kv_heads + g)] = i;
        all[2 * (i * num_kv_heads + g) + 1] = g;
      }
    units = all;
  }
  int status = 0;
  if (nthreads <= 1) {
    for (int32_t u = 0; u < n_units; ++u) {
      int st = decode_unit(&a, units[2 * u], units[2 * u + 1]);
      if (st != 0) status = st;
    }
  } else {
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    orc_worker* ws = (orc_worker*)malloc(sizeof(orc_worker) * (size_t)nthreads);
    if (!th || !ws) {
      free(th); free(ws); free(all);
      return -2;
    }
    for (int32_t t = 0; t < nthreads; ++t) {
      ws[t].a = &a; ws[t].units = units; ws[t].n_units = n_units;
      ws[t].stride = nthreads; ws[t].first = t; ws[t].status = 0;
      pthread_create(&th[t], NULL, worker_main, &ws[t]);
    }
    for (int32_t t = 0; t < nthreads; ++t) {
      pthread_join(th[t], NULL);
      if (ws[t].status != 0) status = ws[t].status;
    }
    free(th); free(ws);
  }
  free(all);
  return status;
}

/* ---- varlen causal attention --------------------------------------------- */

typedef struct {
  double* out;                 /* [N, H_q, d] fp64, N = qsl[num_reqs] */
  const uint16_t* q;           /* [N, H_q, d] bf16 */
  const void* k_cache;         /* [num_blocks, B, H_kv, d] */
  const void* v_cache;
  int32_t num_blocks, block_size, num_kv_heads, head_dim, kv_dtype;
  const int32_t* block_tables; /* [num_reqs, max_blocks] */
  int32_t max_blocks;
  const int32_t* seq_lens;     /* [num_reqs] context tokens after the step */
  const int32_t* qsl;          /* [num_reqs + 1] query start locations */
  int32_t num_reqs, num_heads;
  double scale, k_scale, v_scale;
} orc_varlen_args;

static double varlen_elem(const orc_varlen_args* a, const void* cache,
                          int64_t idx, double kv_scale) {
  if (a->kv_dtype == ORC_KV_BF16)
    return orc_bf16_to_double(((const uint16_t*)cache)[idx]);
  return orc_e4m3_to_double(((const uint8_t*)cache)[idx]) * kv_scale;
}

/* One (request, KV head g) unit.  Returns 0, -1 on a bad id / length, -2 on
 * host OOM. */
static int varlen_unit(const orc_varlen_args* a, int32_t r, int32_t g) {
  const int32_t H = a->num_heads, Hkv = a->num_kv_heads, d = a->head_dim;
  const int32_t B = a->block_size, G = H / Hkv;
  const int32_t first = a->qsl[r], num_new = a->qsl[r + 1] - a->qsl[r];
  const int32_t seq_len = a->seq_lens[r];
  if (num_new < 0 || seq_len < 0) return -1;
  if (num_new == 0) return 0;
  if (num_new > seq_len) { /* no valid position for the first tokens */
    for (int32_t j = 0; j < num_new; ++j)
      for (int32_t i = 0; i < G; ++i)
        memset(a->out + (((int64_t)first + j) * H + (int64_t)g * G + i) * d, 0,
               sizeof(double) * (size_t)d);
    return 0;
  }
  if ((int64_t)seq_len > (int64_t)a->max_blocks * B) return -1;

  /* gather the context rows of KV head g, widening only what is read */
  double* K = (double*)malloc(sizeof(double) * (size_t)seq_len * d);
  double* V = (double*)malloc(sizeof(double) * (size_t)seq_len * d);
  double* w = (double*)malloc(sizeof(double) * (size_t)seq_len);
  if (!K || !V || !w) {
    free(K); free(V); free(w);
    return -2;
  }
  const int32_t* table = a->block_tables + (int64_t)r * a->max_blocks;
  for (int32_t t = 0; t < seq_len; ++t) {
    int32_t phys = table[t / B];
    if (phys < 0 || phys >= a->num_blocks) {
      free(K); free(V); free(w);
      return -1;
    }
    int64_t base = (((int64_t)phys * B + (t % B)) * Hkv + g) * d;
    for (int32_t e = 0; e < d; ++e) {
      K[(int64_t)t * d + e] = varlen_elem(a, a->k_cache, base + e, a->k_scale);
      V[(int64_t)t * d + e] = varlen_elem(a, a->v_cache, base + e, a->v_scale);
    }
  }

  for (int32_t j = 0; j < num_new; ++j) {
    const int32_t last = seq_len - num_new + j; /* its own position */
    for (int32_t i = 0; i < G; ++i) {
      const int32_t h = g * G + i;
      const uint16_t* qh = a->q + (((int64_t)first + j) * H + h) * d;
      double top = -INFINITY;
      for (int32_t t = 0; t <= last; ++t) {
        double dot = 0.0;
        for (int32_t e = 0; e < d; ++e)
          dot += orc_bf16_to_double(qh[e]) * K[(int64_t)t * d + e];
        w[t] = a->scale * dot;
        if (w[t] > top) top = w[t];
      }
      double sum = 0.0;
      for (int32_t t = 0; t <= last; ++t) {
        w[t] = exp(w[t] - top);
        sum += w[t];
      }
      double* o = a->out + (((int64_t)first + j) * H + h) * d;
      for (int32_t e = 0; e < d; ++e) {
        double acc = 0.0;
        for (int32_t t = 0; t <= last; ++t) acc += w[t] * V[(int64_t)t * d + e];
        o[e] = acc / sum;
      }
    }
  }
  free(K); free(V); free(w);
  return 0;
}

typedef struct {
  const orc_varlen_args* a;
  int32_t n_units, stride, first;
  int status;
} orc_varlen_worker;

static void* varlen_worker_main(void* p) {
  orc_varlen_worker* w = (orc_varlen_worker*)p;
  const int32_t Hkv = w->a->num_kv_heads;
  for (int32_t u = w->first; u < w->n_units; u += w->stride) {
    int st = varlen_unit(w->a, u / Hkv, u % Hkv);
    if (st != 0) w->status = st;
  }
  return NULL;
}

/* Every (request, KV head) unit; nthreads > 1 spreads the same per-unit
 * function over POSIX threads (results do not depend on it).  Returns 0, -1
 * on a bad id, length or head count, -2 on host OOM. */
int orc_varlen(double* out, const uint16_t* q, const void* k_cache,
               const void* v_cache, int32_t num_blocks, int32_t block_size,
               int32_t num_kv_heads, int32_t head_dim, int32_t kv_dtype,
               const int32_t* block_tables, int32_t max_blocks,
               const int32_t* seq_lens, const int32_t* qsl, int32_t num_reqs,
               int32_t num_heads, double scale, double k_scale,
               double v_scale, int32_t nthreads) {
  if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || num_reqs < 0)
    return -1;
  orc_varlen_args a = {out, q, k_cache, v_cache, num_blocks, block_size,
                       num_kv_heads, head_dim, kv_dtype, block_tables,
                       max_blocks, seq_lens, qsl, num_reqs, num_heads,
                       scale, k_scale, v_scale};
  const int32_t n_units = num_reqs * num_kv_heads;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > n_units) nthreads = n_units > 0 ? n_units : 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  orc_varlen_worker* ws =
      (orc_varlen_worker*)malloc(sizeof(orc_varlen_worker) * (size_t)nthreads);
  if (!th || !ws) {
    free(th); free(ws);
    return -2;
  }
  int status = 0;
  for (int32_t t = 0; t < nthreads; ++t) {
    ws[t].a = &a; ws[t].n_units = n_units; ws[t].stride = nthreads;
    ws[t].first = t; ws[t].status = 0;
  }
  if (nthreads == 1) {
    varlen_worker_main(&ws[0]);
  } else {
    for (int32_t t = 0; t < nthreads; ++t)
      pthread_create(&th[t], NULL, varlen_worker_main, &ws[t]);
    for (int32_t t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  }
  for (int32_t t = 0; t < nthreads; ++t)
    if (ws[t].status != 0) status = ws[t].status;
  free(th); free(ws);
  return status;
}
