// Paged decode attention on the CUDA cores (SIMT), split-K capable.
//
// One CTA handles one work item (sequence i, KV head g, partition p): the
// tokens [p*PS, min((p+1)*PS, n_i)) of sequence i for all G query heads that
// share KV head g, so every K/V byte of the partition is read from HBM once
// ("4.6 PagedAttention & KV-Cache Memory Management", section "The
// PagedAttention Kernel": a CTA per (sequence, KV head), block-table gather,
// online softmax; section "Performance considerations": split-K over the
// sequence as in PagedAttention v2).
//
// Pipeline: the partition's block-table slice is staged in shared memory,
// then 64-token chunks of K and V rows are copied global->shared with 16-byte
// cp.async into a 3-stage ring.  Each row (one token of one KV head, d
// elements, d*b contiguous bytes) is stored with its 16-byte pieces XOR-
// swizzled by the row index so that both access patterns below are free of
// bank conflicts.  Per chunk:
//   QK   thread = (token, half of the heads) or (token, half of d) for G == 1;
//        q sits pre-scaled by scale*log2(e) in shared memory (broadcast reads).
//   max  per-head maximum over the chunk (warp shuffles + one smem exchange),
//        running max update, alpha = 2^(m_old - m_new), p = 2^(s - m_new).
//   PV   thread = (token group, 8 consecutive d elements) with G x 8 fp32
//        accumulators, rescaled by alpha once per chunk.
// Tokens past the end of the context are zero-filled in shared memory and
// get p = 0, so stale or non-finite bytes in a partially filled block never
// reach the output.
//
// Result: with one partition the normalised bf16 output row is written
// directly; otherwise the unnormalised fp32 accumulator and (m, l) go to the
// workspace for the combine kernel.
#pragma once

#include "pa_device.cuh"
#include "pa_kernels.cuh"

namespace pa {

template <int D, int G, bool FP8>
struct SimtCfg {
  static constexpr int NT = kSimtThreads;
  static constexpr int CH = kChunkTokens;
  static constexpr int NST = 3;
  static constexpr int EB = FP8 ? 1 : 2;
  static constexpr int ROWB = D * EB;     // bytes of one cache row
  static constexpr int CPR = ROWB / 16;   // 16-byte pieces per row
  static constexpr int EPP = 16 / EB;     // elements per piece
  static constexpr int STAGE_B = 2 * CH * ROWB;
  static constexpr int TOK_PER_THR = CH * CPR / NT;  // rows each thread copies (K and V)
  // QK split of the 128 threads over 64 tokens
  static constexpr int HSPLIT = G >= 2 ? 2 : 1;
  static constexpr int DSPLIT = 2 / HSPLIT;
  static constexpr int HPT = G / HSPLIT;
  static constexpr int QK_PIECES = CPR / DSPLIT;
  // PV: 8 elements per thread
  static constexpr int PV_TPR = D / 8;
  static constexpr int NG = NT / PV_TPR;
  static constexpr int TPG = CH / NG;
  // shared memory carve-up (bytes)
  static constexpr int RED_B = NG * G * D * 4;
  static constexpr int RING_B = (NST * STAGE_B > RED_B) ? NST * STAGE_B : RED_B;
  static constexpr int Q_OFF = RING_B;
  static constexpr int S_OFF = Q_OFF + G * D * 4;       // logits [CH][G] (+ [2][CH] partials)
  static constexpr int P_OFF = S_OFF + 2 * CH * (G > 1 ? G : 2) * 4;
  static constexpr int W_OFF = P_OFF + CH * G * 4;      // per-warp partials [4][G]
  static constexpr int A_OFF = W_OFF + (NT / 32) * G * 4;  // alpha [G]
  static constexpr int T_OFF = A_OFF + 8 * 4;           // block-table slice
  static constexpr int FIXED_B = T_OFF;
  static_assert(CPR * 16 == ROWB, "row must be a whole number of 16-byte pieces");
  static_assert(NT % CPR == 0 && (CH * CPR) % NT == 0, "copy mapping");
  static_assert(NT % PV_TPR == 0 && CH % NG == 0, "PV mapping");
};

template <int D, int G, bool FP8>
__global__ void __launch_bounds__(kSimtThreads, 2)
    decode_simt_kernel(const DecodeParams p) {
  using C = SimtCfg<D, G, FP8>;
  constexpr int NT = C::NT, CH = C::CH, NST = C::NST, CPR = C::CPR, ROWB = C::ROWB;
  extern __shared__ __align__(128) unsigned char smem[];
  float* q_s = reinterpret_cast<float*>(smem + C::Q_OFF);
  float* s_s = reinterpret_cast<float*>(smem + C::S_OFF);
  float* p_s = reinterpret_cast<float*>(smem + C::P_OFF);
  float* w_s = reinterpret_cast<float*>(smem + C::W_OFF);
  float* a_s = reinterpret_cast<float*>(smem + C::A_OFF);
  int32_t* t_s = reinterpret_cast<int32_t*>(smem + C::T_OFF);

  const int tid = threadIdx.x;
  const int part = blockIdx.x;
  const int g = blockIdx.y;
  const int seq = blockIdx.z;
  const int H = p.num_heads;
  // a length beyond the table's capacity is clamped so no read leaves the row
  const int n = min(p.context_lens[seq], p.max_blocks << p.log2_block_size);
  const int PS = p.partition_tokens;
  const int start = part * PS;
  const int num_parts = (n + PS - 1) / PS;

  if (n <= 0) {  // empty context: partition 0 writes zero rows
    if (part == 0) {
      __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) +
                         ((int64_t)seq * H + (int64_t)g * G) * D;
      for (int e = tid; e < G * D; e += NT) o[e] = __float2bfloat16_rn(0.f);
    }
    return;
  }
  if (start >= n) return;
  const int end = min(start + PS, n);
  const int lb_first = start >> p.log2_block_size;
  const int lb_cnt = ((end - 1) >> p.log2_block_size) - lb_first + 1;

  // ---- stage the block-table slice and the pre-scaled query ----
  const int32_t* table = p.block_tables + (int64_t)seq * p.max_blocks + lb_first;
  for (int j = tid; j < lb_cnt; j += NT) t_s[j] = table[j];
  {
    float qscale = p.scale_log2;
    if (FP8) qscale *= *p.k_scale;
    const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(p.q) +
                              ((int64_t)seq * H + (int64_t)g * G) * D;
    for (int e = tid; e < G * D; e += NT) q_s[e] = __bfloat162float(qg[e]) * qscale;
  }
  __syncthreads();

  // ---- per-thread copy assignment: TOK_PER_THR rows, one piece column ----
  const int cp_cc = tid % CPR;
  const int cp_tt0 = tid / CPR;  // rows cp_tt0 + (NT / CPR) * k
  const char* kbase = static_cast<const char*>(p.k_cache) + (int64_t)g * ROWB + cp_cc * 16;
  const char* vbase = static_cast<const char*>(p.v_cache) + (int64_t)g * ROWB + cp_cc * 16;
  const int64_t row_stride = (int64_t)p.num_kv_heads * ROWB;  // bytes between slots
  const uint32_t ring = smem_u32(smem);
  const int bmask = p.block_size - 1;
  const int nchunks = (end - start + CH - 1) / CH;

  auto issue_chunk = [&](int c) {
    if (c < nchunks) {
      const int cs = start + c * CH;
      const uint32_t st = ring + (c % NST) * C::STAGE_B;
#pragma unroll
      for (int k = 0; k < C::TOK_PER_THR; ++k) {
        const int tt = cp_tt0 + (NT / CPR) * k;
        const int t = cs + tt;
        const uint32_t dst = st + tt * ROWB + ((cp_cc ^ (tt % CPR)) * 16);
        const char* ks = kbase;
        const char* vs = vbase;
        uint32_t bytes = 0;
        if (t < end) {
          const int phys = t_s[(t >> p.log2_block_size) - lb_first];
          if ((unsigned)phys < (unsigned)p.num_blocks) {
            const int64_t off = ((int64_t)phys * p.block_size + (t & bmask)) * row_stride;
            ks += off;
            vs += off;
            bytes = 16;
          }
        }
        cp_async_16(dst, ks, bytes);
        cp_async_16(dst + CH * ROWB, vs, bytes);
      }
    }
    cp_async_commit();
  };

#pragma unroll
  for (int c = 0; c < NST - 1; ++c) issue_chunk(c);

  // softmax state: thread owns head hs = tid % G for the running max / sum
  const int hs = tid % G;
  float m_run = -INFINITY;
  float l_part = 0.f;
  float acc[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;

  // QK assignment
  const int qk_tt = tid % CH;
  const int qk_sel = tid / CH;
  // PV assignment
  const int pv_cc = tid % C::PV_TPR;
  const int pv_tg = tid / C::PV_TPR;

  for (int c = 0; c < nchunks; ++c) {
    cp_async_wait<NST - 2>();
    __syncthreads();  // chunk c visible; stage (c-1)%NST free
    issue_chunk(c + NST - 1);

    const int cs = start + c * CH;
    const unsigned char* sK = smem + (c % NST) * C::STAGE_B;
    const unsigned char* sV = sK + CH * ROWB;

    // ---- QK ----
    {
      float dot[C::HPT][2];  // even / odd elements: two independent FMA chains
#pragma unroll
      for (int j = 0; j < C::HPT; ++j) dot[j][0] = dot[j][1] = 0.f;
      const int piece0 = (C::DSPLIT == 2) ? qk_sel * C::QK_PIECES : 0;
#pragma unroll
      for (int pc = 0; pc < C::QK_PIECES; ++pc) {
        const int piece = piece0 + pc;
        const uint4 raw = *reinterpret_cast<const uint4*>(
            sK + qk_tt * ROWB + ((piece ^ (qk_tt % CPR)) * 16));
        float kf[C::EPP];
        Unpack16<FP8>::run(raw, kf);
#pragma unroll
        for (int j = 0; j < C::HPT; ++j) {
          const int h = (C::HSPLIT == 2) ? qk_sel + 2 * j : 0;
          const float4* qv = reinterpret_cast<const float4*>(q_s + h * D + piece * C::EPP);
#pragma unroll
          for (int v4 = 0; v4 < C::EPP / 4; ++v4) {
            const float4 qq = qv[v4];
            dot[j][0] = fmaf(qq.x, kf[4 * v4 + 0], dot[j][0]);
            dot[j][1] = fmaf(qq.y, kf[4 * v4 + 1], dot[j][1]);
            dot[j][0] = fmaf(qq.z, kf[4 * v4 + 2], dot[j][0]);
            dot[j][1] = fmaf(qq.w, kf[4 * v4 + 3], dot[j][1]);
          }
        }
      }
      if (C::HSPLIT == 2) {
#pragma unroll
        for (int j = 0; j < C::HPT; ++j) s_s[qk_tt * G + qk_sel + 2 * j] = dot[j][0] + dot[j][1];
      } else {
        s_s[qk_sel * CH + qk_tt] = dot[0][0] + dot[0][1];  // two d-halves, summed below
      }
    }
    __syncthreads();

    // ---- chunk max per head ----
    const int valid = end - cs;  // tokens of this chunk inside the context (>= 1)
    float sv[(CH * G + NT - 1) / NT];
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < (CH * G + NT - 1) / NT; ++k) {
      const int tt = tid / G + (NT / G) * k;
      float s = -INFINITY;
      if (tt < CH && tt < valid)
        s = (G > 1) ? s_s[tt * G + hs] : (s_s[tt] + s_s[CH + tt]);
      sv[k] = s;
      mx = fmaxf(mx, s);
    }
#pragma unroll
    for (int off = G; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((tid & 31) < G) w_s[(tid >> 5) * G + (tid & 31)] = mx;
    __syncthreads();
    float m_chunk = w_s[hs];
#pragma unroll
    for (int w = 1; w < NT / 32; ++w) m_chunk = fmaxf(m_chunk, w_s[w * G + hs]);
    const float m_new = fmaxf(m_run, m_chunk);
    const float alpha = fast_exp2(m_run - m_new);  // 0 on the first chunk
    m_run = m_new;
    float lsum = 0.f;
#pragma unroll
    for (int k = 0; k < (CH * G + NT - 1) / NT; ++k) {
      const int tt = tid / G + (NT / G) * k;
      if (tt < CH) {
        const float pv = (tt < valid) ? fast_exp2(sv[k] - m_new) : 0.f;
        p_s[tt * G + hs] = pv;
        lsum += pv;
      }
    }
    l_part = l_part * alpha + lsum;
    if (tid < G) a_s[tid] = alpha;
    __syncthreads();

    // ---- PV ----
    {
      float al[G];
#pragma unroll
      for (int h = 0; h < G; ++h) al[h] = a_s[h];
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] *= al[h];
#pragma unroll
      for (int k = 0; k < C::TPG; ++k) {
        const int tt = pv_tg + C::NG * k;
        float vf[8];
        if (!FP8) {
          const uint4 raw = *reinterpret_cast<const uint4*>(
              sV + tt * ROWB + ((pv_cc ^ (tt % CPR)) * 16));
          Unpack16<false>::run(raw, vf);
        } else {
          const uint2 raw = *reinterpret_cast<const uint2*>(
              sV + tt * ROWB + (((pv_cc >> 1) ^ (tt % CPR)) * 16) + (pv_cc & 1) * 8);
          float2 a = e4m3x2_to_float2(static_cast<uint16_t>(raw.x & 0xffffu));
          float2 b = e4m3x2_to_float2(static_cast<uint16_t>(raw.x >> 16));
          float2 cc2 = e4m3x2_to_float2(static_cast<uint16_t>(raw.y & 0xffffu));
          float2 d = e4m3x2_to_float2(static_cast<uint16_t>(raw.y >> 16));
          vf[0] = a.x; vf[1] = a.y; vf[2] = b.x; vf[3] = b.y;
          vf[4] = cc2.x; vf[5] = cc2.y; vf[6] = d.x; vf[7] = d.y;
        }
        float pr[G];
        if (G % 4 == 0) {
#pragma unroll
          for (int h4 = 0; h4 < G / 4; ++h4) {
            const float4 t4 = reinterpret_cast<const float4*>(p_s + tt * G)[h4];
            pr[4 * h4 + 0] = t4.x; pr[4 * h4 + 1] = t4.y;
            pr[4 * h4 + 2] = t4.z; pr[4 * h4 + 3] = t4.w;
          }
        } else {
#pragma unroll
          for (int h = 0; h < G; ++h) pr[h] = p_s[tt * G + h];
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(pr[h], vf[e], acc[h][e]);
      }
    }
  }

  // ---- finalize: reduce l over threads, acc over token groups ----
  cp_async_wait<0>();
  __syncthreads();  // all chunks consumed; the ring may be reused
#pragma unroll
  for (int off = G; off < 32; off <<= 1) l_part += __shfl_xor_sync(0xffffffffu, l_part, off);
  if ((tid & 31) < G) w_s[(tid >> 5) * G + (tid & 31)] = l_part;
  float* red = reinterpret_cast<float*>(smem);  // [NG][G][D]
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e4 = 0; e4 < 2; ++e4)
      *reinterpret_cast<float4*>(red + (pv_tg * G + h) * D + pv_cc * 8 + 4 * e4) =
          make_float4(acc[h][4 * e4], acc[h][4 * e4 + 1], acc[h][4 * e4 + 2], acc[h][4 * e4 + 3]);
  __syncthreads();

  float vscale = 1.f;
  if (FP8) vscale = *p.v_scale;
  const bool single = (num_parts == 1);
  for (int o2 = tid; o2 < G * D / 2; o2 += NT) {
    const int h = (2 * o2) / D;
    const int e = (2 * o2) % D;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int gi = 0; gi < C::NG; ++gi) {
      const float2 v = *reinterpret_cast<const float2*>(red + (gi * G + h) * D + e);
      s0 += v.x;
      s1 += v.y;
    }
    float l_tot = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) l_tot += w_s[w * G + h];
    const int64_t row = (int64_t)seq * H + (int64_t)g * G + h;
    if (single) {
      const float inv = vscale / l_tot;
      reinterpret_cast<uint32_t*>(p.out)[(row * D + e) / 2] = pack_bf16x2_rn(s0 * inv, s1 * inv);
    } else {
      float2* wo = reinterpret_cast<float2*>(p.ws_o + (row * p.max_parts + part) * D + e);
      *wo = make_float2(s0 * vscale, s1 * vscale);
    }
  }
  if (!single && tid < G) {
    float l_tot = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) l_tot += w_s[w * G + tid];
    const int64_t row = (int64_t)seq * H + (int64_t)g * G + tid;
    p.ws_ml[row * p.max_parts + part] = make_float2(m_run, l_tot);
  }
}

}  // namespace pa
