// Causal paged attention for prefill chunks on the 5th-generation tensor
// cores, for a bf16 or e4m3 cache with head_dim 128: the tensor-core path
// of pa_varlen_attention.
//
// What it computes is the varlen paged attention of "Paged attention"
// (query_start_loc, seq_lens, causal limit): request r's new tokens are
// q[qsl[r] .. qsl[r+1]), the last T_r positions of its seq_lens[r]-token
// context (their K/V already written to the cache), and new token j attends
// to keys 0 .. seq_len - T_r + j; query head h reads KV head h / G.
//
// Where the decode kernels put a few query heads on the MMA's N side and
// stream the context once per step, a prefill tile has many queries: a work
// item is (request, tile of 128 / G new tokens, KV head), whose 128 query
// rows -- token-major, row = token * G + head-in-group -- sit on the MMA's M
// side and share every K/V chunk:
//   S = Q K^T   tcgen05.mma M=128 rows, N=128 keys, K=128 (d); A = the q tile
//               (one 3-D TMA box {64 of d, G heads, 128 / G tokens} per
//               64-column half, rows past the batch zero-filled), B = the K
//               chunk (the decode kernels' 4-D block boxes);
//   softmax     two threads per row, 64 logits each from TMEM lane row; the
//               pair exchanges its half-row max through shared memory;
//   O += P V    M=128 rows, N=128 (d), K=128 keys; A = P (bf16, smem), B = the
//               V chunk read MN-major straight from the TMA layout; O lives in
//               TMEM across the item's chunks.
// O is rescaled only when a row's running max grows by more than 2^8 (p
// stays below 256, well inside bf16's range); otherwise later chunks keep
// the old reference max, which the final division by the sum of the same p
// cancels.  The sum adds each p before its bf16 rounding (the MMA's P is
// rounded): a relative difference below bf16's rounding error.  The scale
// must be positive (the max is taken over the raw logits and the scale
// folded into one FMA per logit).  Keys past a row's causal limit get p = 0 (a select,
// so stale cache bytes never reach the result); V rows past the item's last
// key are zeroed in smem.
//
// e4m3 caches (PCfg<true>).  The MMAs take the cache bytes as they are
// (kind::f8f6f4; K and V chunks of 128 keys x 128-byte rows).  At an item's
// start the softmax threads split the staged bf16 q rows, each scaled by
// the power of two that puts its max |q| in [128, 256), into three e4m3
// parts (three operand tiles; the logits are the sum of three MMAs).  P
// holds 2^(8 - R) p as two e4m3 parts, with the rescale threshold R = 3 so
// that it stays inside e4m3's range; the factor and the rounding cancel in
// O / l.  P V is computed as its transpose, O^T = V^T P^T (V the MN-major A
// operand, P's rows the K-major B operand), so a row of O is a column of
// the tensor-memory tile: a row's rescale is collective (each row publishes
// its factor and one reduction barrier tells every thread whether any row
// rescales), and the epilogue writes each thread's element d of 64 rows.
//
// Warp roles (352 threads): warps 0-7 softmax and epilogue, two threads per
// row (64 keys and 64 output columns each); warp 8 producer of the q tiles
// and the K chunks (3-stage ring, a stage freed when its logits MMA
// completes); warp 9 TMEM allocation and the MMA-issuing thread; warp 10
// producer of the V chunks (2-stage ring, freed after the PV MMA).  The K
// producer takes work items from a counter in the workspace (word 1, zeroed
// by the host before the launch) and publishes them through a 4-slot ring
// to the other roles, so a CTA that drew short items takes more of them.
// Every mbarrier wait is bounded (error word in the workspace, CTA
// aborted), as in the decode kernels.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_device.cuh"
#include "pa_kernels.cuh"
#include "tc_ptx.cuh"
#include "tc_sched.cuh"

namespace pa {
namespace pf {

using tc::Smem;
using tc::drain_bar;
using tc::kWaitClocks;
using tc::wait_bar;

constexpr int D = 128;
constexpr int CHK = 128;                  // keys per chunk

// Paired fp32 arithmetic (one instruction for two lanes of work): the
// softmax of a prefill tile is bound by instruction issue.
__device__ __forceinline__ float2 fma_x2(float2 a, float2 b, float2 c) {
  unsigned long long ra, rb, rc, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}
__device__ __forceinline__ float2 add_x2(float2 a, float2 b) {
  unsigned long long ra, rb, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}
// K and V rings: a K chunk is free once its logits MMA completes, a V chunk
// only after its PV MMA, so K runs one stage further ahead
constexpr int NSTK = 3, NSTV = 2;
constexpr int kMaxReqs = 256;
constexpr int HALF_B = 128 * 128;         // one 128-byte-wide column block of 128 rows
constexpr int QTILE_B = 128 * D * 2;      // the bf16 q tile: 128 rows
constexpr int NRING = 4;  // work items published ahead by the K producer
constexpr int NSOFT = 256;  // softmax threads: two per q tile row
constexpr int NTHREADS = NSOFT + 96;
constexpr int PROD_WARP = NSOFT / 32, MMA_WARP = PROD_WARP + 1, VPROD_WARP = MMA_WARP + 1;
constexpr int TMEM_COLS = 512;  // S[2] at 0 and 128, O at 256
constexpr int S_COL = 0, O_COL = 256;
constexpr int B_FULL_K = 0, B_FULL_V = B_FULL_K + NSTK, B_EMPTY_K = B_FULL_V + NSTV,
              B_EMPTY_V = B_EMPTY_K + NSTK, B_Q_FULL = B_EMPTY_V + NSTV,
              B_Q_EMPTY = B_Q_FULL + 1, B_S_FULL = B_Q_EMPTY + 1, B_S_EMPTY = B_S_FULL + 2,
              B_P_FULL = B_S_EMPTY + 2, B_P_EMPTY = B_P_FULL + 1, B_O_FULL = B_P_EMPTY + 1,
              B_O_EMPTY = B_O_FULL + 2, B_ITEM_FULL = B_O_EMPTY + 1,
              B_ITEM_EMPTY = B_ITEM_FULL + 4, B_QP_FULL = B_ITEM_EMPTY + 4,
              B_QP_EMPTY = B_QP_FULL + 1, NBARS = B_QP_EMPTY + 1;

// Shared-memory layout for a bf16 or an e4m3 cache.  e4m3: K and V chunks are
// 128 bytes a row; the bf16 q tile is staged, then split by the softmax
// threads into three e4m3 parts (rows scaled by a power of two each); P is
// two e4m3 parts.
template <bool FP8>
struct PCfg {
  static constexpr int ELT = FP8 ? 1 : 2;
  static constexpr int TILE_B = CHK * D * ELT;   // one K or V chunk
  static constexpr int NQPART = FP8 ? 3 : 0;
  static constexpr int QPART_B = 128 * D;        // one e4m3 part of the q tile
  static constexpr int NPPART = FP8 ? 2 : 1;
  static constexpr int PPART_B = 128 * CHK * ELT;  // P (bf16) or one e4m3 part of it
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NSTK * TILE_B;
  static constexpr int OFF_Q = OFF_V + NSTV * TILE_B;
  static constexpr int OFF_QP = OFF_Q + QTILE_B;
  static constexpr int OFF_P = OFF_QP + NQPART * QPART_B;
  static constexpr int OFF_BAR = OFF_P + NPPART * PPART_B;  // one P buffer
  static constexpr int OFF_TMEM = OFF_BAR + NBARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEM + 4;
  static constexpr int OFF_RING = OFF_ABORT + 4;  // [NRING] item indices
  // tile prefix per request, [R+1]; 16 bits suffice: at most 65535 new tokens
  static constexpr int OFF_TP = OFF_RING + NRING * 4;
  static constexpr int OFF_XCH = (OFF_TP + (kMaxReqs + 1) * 2 + 15) / 16 * 16;  // [256] floats
  // e4m3: per-row rescale factors [2][128] (by chunk parity) and final sums [128]
  static constexpr int OFF_ALPHA = OFF_XCH + 256 * 4;
  static constexpr int OFF_LSUM = OFF_ALPHA + (FP8 ? 2 * 128 * 4 : 0);
  static constexpr int SMEM_BYTES = OFF_LSUM + (FP8 ? 128 * 4 : 0) + 1024;  // + alignment slack
  // O is rescaled when a row's max grows by more than 2^R: p <= 2^R.  e4m3
  // P holds p * 2^(8 - R) <= 256 (inside e4m3's 448), so a smaller R keeps
  // small weights above e4m3's 2^-9 floor
  static constexpr float kRescaleLog2 = FP8 ? 3.f : 8.f;
  static constexpr float kPScale = FP8 ? 32.f : 1.f;  // 2^(8 - R)
  static constexpr float kPScaleLog2 = FP8 ? 5.f : 0.f;  // 8 - R
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(OFF_BAR % 1024 == 0, "tiles stay 1024-byte aligned");
};

struct Params {
  void* out;                    // [num_tokens, H, D] bf16
  const int32_t* block_tables;  // [R, max_blocks]
  const int32_t* seq_lens;      // [R]
  const int32_t* qsl;           // [R + 1]
  int* err;                     // workspace word 0
  unsigned* next_item;          // workspace word 1: items handed out (zeroed before launch)
  int num_seqs, num_tokens, num_heads, num_kv_heads, max_blocks, num_blocks, block_size, log2_bs;
  int box_tok, log2_box;
  int min_tokens;  // requests with fewer new tokens get no tiles
  float scale_log2;
  const float* k_scale;  // e4m3: per-tensor dequantisation scales (device scalars)
  const float* v_scale;
};

// One work item: request r, query tile qt (tokens qt*MQ ..), KV head g.
struct Item {
  int r, qt, g;
  int q0;      // first q row of the request
  int T;       // its new tokens
  int ctx;     // keys before its first new token (seq_len - T)
  int ntok;    // new tokens in this tile
  int kv_end;  // keys the tile's last token sees
  int nch;     // K/V chunks (0: the request's rows are zero, T > seq_len)
};

template <int G>
__device__ __forceinline__ Item item_of(long long i, const uint16_t* tp, int R,
                                        const Params& p) {
  constexpr int MQ = 128 / G;
  Item it;
  const long long tile = i / p.num_kv_heads;
  it.g = (int)(i - tile * p.num_kv_heads);
  int lo = 0, hi = R;  // the request holding this tile: tp[r] <= tile < tp[r+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tp[mid] <= tile) lo = mid;
    else hi = mid;
  }
  it.r = lo;
  it.qt = (int)(tile - tp[lo]);
  it.q0 = __ldg(&p.qsl[lo]);
  it.T = __ldg(&p.qsl[lo + 1]) - it.q0;
  const int sl = __ldg(&p.seq_lens[lo]);
  it.ctx = sl - it.T;
  it.ntok = min(MQ, it.T - it.qt * MQ);
  it.kv_end = it.ctx + it.qt * MQ + it.ntok;
  const int cap = p.max_blocks << p.log2_bs;
  it.nch = (it.ctx < 0 || it.kv_end > cap) ? 0 : (it.kv_end + CHK - 1) / CHK;
  return it;
}

template <int G, bool FP8>
__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_q, const Params p) {
  using C = PCfg<FP8>;
  constexpr int TILE_B = C::TILE_B, QPART_B = C::QPART_B, PPART_B = C::PPART_B;
  constexpr int OFF_K = C::OFF_K, OFF_V = C::OFF_V, OFF_Q = C::OFF_Q, OFF_QP = C::OFF_QP,
                OFF_P = C::OFF_P, OFF_BAR = C::OFF_BAR, OFF_TMEM = C::OFF_TMEM,
                OFF_ABORT = C::OFF_ABORT, OFF_RING = C::OFF_RING, OFF_TP = C::OFF_TP,
                OFF_XCH = C::OFF_XCH;
  constexpr float kRescaleLog2 = C::kRescaleLog2;
  constexpr int MQ = 128 / G;  // new tokens per tile
  extern __shared__ unsigned char smem_raw[];
  Smem sm;
  {
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t aligned = (raw + 1023u) & ~1023u;
    sm.base = smem_raw + (aligned - raw);
    sm.base_u32 = aligned;
    sm.off_bar = OFF_BAR;
    sm.off_abort = OFF_ABORT;
  }
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int R = p.num_seqs;
  uint16_t* tp = reinterpret_cast<uint16_t*>(sm.base + OFF_TP);

  // ---------------- prologue ----------------
  ptx::grid_dependency_wait();
  if (warp == MMA_WARP) {
    ptx::tmem_alloc(sm.base_u32 + OFF_TMEM, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < NBARS; ++i) {
      uint32_t cnt = 1;
      if ((i >= B_S_EMPTY && i < B_S_EMPTY + 2) || i == B_P_FULL || i == B_O_EMPTY ||
          i == B_QP_FULL)
        cnt = NSOFT;
      // e4m3: the softmax threads read the staged q tile (and free it)
      if (FP8 && i == B_Q_EMPTY) cnt = NSOFT;
      // an item slot is read by the V producer, the MMA thread and the 8
      // softmax warps (one arrival each)
      if (i >= B_ITEM_EMPTY && i < B_ITEM_EMPTY + NRING) cnt = 2 + NSOFT / 32;
      ptx::mbar_init(sm.bar(i), cnt);
    }
    *sm.abort_flag() = 0;
    ptx::fence_mbar_init();
  }
  if (warp == PROD_WARP && lane == 0) {
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    ptx::prefetch_tmap(&tm_q);
  }
  // tiles per request, then an exclusive prefix (warp 0)
  for (int r = tid; r < R; r += NTHREADS) {
    const int T = __ldg(&p.qsl[r + 1]) - __ldg(&p.qsl[r]);
    tp[r] = (uint16_t)(T > 0 && T >= p.min_tokens ? (T + MQ - 1) / MQ : 0);
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < R; base += 32) {
      const int i = base + lane;
      const int v = i < R ? tp[i] : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (i < R) tp[i] = (uint16_t)(carry + incl - v);
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tp[R] = (uint16_t)carry;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm.base + OFF_TMEM);
  const long long total = (long long)tp[R] * p.num_kv_heads;  // work items
  // Items are handed out dynamically (a counter in the workspace): the K
  // producer takes the next index and publishes it in a ring slot; the
  // other roles read the slots in order.  An index >= total ends the CTA.
  volatile int* ring_s = reinterpret_cast<volatile int*>(sm.base + OFF_RING);
  auto read_item = [&](int k, bool arrive_lane0) -> long long {
    const int slot = k & (NRING - 1);
    if (!wait_bar(sm, sm.bar(B_ITEM_FULL + slot), (uint32_t)(k / NRING) & 1, p.err, 30))
      return total;
    const long long i = ring_s[slot];
    __syncwarp();
    if (arrive_lane0) ptx::mbar_arrive(sm.bar(B_ITEM_EMPTY + slot));
    return i;
  };

  if (warp == PROD_WARP || warp == VPROD_WARP) {
    // ================= producers (K and the q tiles: warp 8; V: warp 10) ====
    const bool isk = warp == PROD_WARP;
    const int nst = isk ? NSTK : NSTV;
    const uint32_t ring = sm.base_u32 + (isk ? OFF_K : OFF_V);
    const void* tm = isk ? (const void*)&tm_k : (const void*)&tm_v;
    const int b_full = isk ? B_FULL_K : B_FULL_V, b_empty = isk ? B_EMPTY_K : B_EMPTY_V;
    int qk = 0;        // items with chunks so far (q tile loads)
    long long ck = 0;  // chunks so far
    for (int k = 0;; ++k) {
      long long i;
      if (isk) {
        // publish the next item (after every reader has taken the slot's last one)
        const int slot = k & (NRING - 1);
        if (!wait_bar(sm, sm.bar(B_ITEM_EMPTY + slot), ((uint32_t)(k / NRING) & 1) ^ 1, p.err,
                      29))
          break;
        long long got = 0;
        if (lane == 0) {
          got = atomicAdd(p.next_item, 1u);
          ring_s[slot] = (int)(got < total ? got : total);
          ptx::mbar_arrive(sm.bar(B_ITEM_FULL + slot));
        }
        i = __shfl_sync(0xffffffffu, got, 0);
      } else {
        i = read_item(k, lane == 0);
      }
      if (i >= total) break;
      const Item it = item_of<G>(i, tp, R, p);
      if (it.nch == 0) continue;
      if (isk) {
        if (qk > 0 && !wait_bar(sm, sm.bar(B_Q_EMPTY), (qk - 1) & 1, p.err, 21)) break;
        if (lane == 0) {
          // rows token * G + i: box {64 of d, G heads, MQ tokens} per half
          const uint32_t dst = sm.base_u32 + OFF_Q;
          const int row = it.q0 + it.qt * MQ;
          ptx::mbar_arrive_expect_tx(sm.bar(B_Q_FULL), (uint32_t)QTILE_B);
          ptx::tma_load_3d(dst, &tm_q, sm.bar(B_Q_FULL), 0, it.g * G, row);
          ptx::tma_load_3d(dst + HALF_B, &tm_q, sm.bar(B_Q_FULL), 64, it.g * G, row);
        }
      }
      ++qk;
      bool ok = true;
      for (int j = 0; j < it.nch; ++j, ++ck) {
        const int s = (int)(ck % nst);
        const uint32_t ph = (uint32_t)(ck / nst) & 1;
        const int keys = min(CHK, it.kv_end - j * CHK);
        const int nbox = (keys + p.box_tok - 1) >> p.log2_box;
        // the chunk's block ids, read while the stage drains
        int phys = 0;
        if (lane < nbox)
          phys = __ldg(&p.block_tables[(int64_t)it.r * p.max_blocks +
                                       ((j * CHK + lane * p.box_tok) >> p.log2_bs)]);
        if (!wait_bar(sm, sm.bar(b_empty + s), ph ^ 1, p.err, 22)) {
          ok = false;
          break;
        }
        if (lane < nbox && (unsigned)phys >= (unsigned)p.num_blocks) {
          atomicExch(p.err, 3);  // bad block id: load block 0 instead of faulting
          phys = 0;
        }
        if (lane == 0)
          ptx::mbar_arrive_expect_tx(sm.bar(b_full + s),
                                     (uint32_t)nbox * p.box_tok * (uint32_t)(D * C::ELT));
        __syncwarp();
        if (lane < nbox) {
          // a row is one 128-byte box column (e4m3: all of d; bf16: two
          // 64-column halves HALF_B apart)
          const uint32_t dst = ring + s * TILE_B + (uint32_t)(lane * p.box_tok) * 128u;
          const int off = (j * CHK + lane * p.box_tok) & (p.block_size - 1);
          ptx::tma_load_4d(dst, tm, sm.bar(b_full + s), 0, it.g, off, phys);
          if (!FP8) ptx::tma_load_4d(dst + HALF_B, tm, sm.bar(b_full + s), 64, it.g, off, phys);
        }
      }
      if (!ok) break;
    }
    // drain: the last loads issued must land before the CTA can exit
    __syncwarp();
    if (lane == 0) {
      for (long long l = ck > nst ? ck - nst : 0; l < ck; ++l)
        drain_bar(sm.bar(b_full + (int)(l % nst)), (uint32_t)(l / nst) & 1);
      if (isk && qk > 0) drain_bar(sm.bar(B_Q_FULL), (qk - 1) & 1);
    }
  } else if (warp == MMA_WARP) {
    // ================= MMA issuer =================
    // Two cursors over the same chunk sequence: the logits MMA of chunk nq
    // (needs its K chunk, a free S buffer and, at an item's first chunk, the
    // q tile) and the PV MMA of chunk npv < nq (needs P, the V chunk and, at
    // an item's first chunk, O read out by the previous item's epilogue).
    if (lane == 0) {
      // e4m3 uses the operand forms of the e4m3 decode kernel: both K-major
      // for the logits; for P V the transposed product O^T = V^T P^T, V the
      // MN-major A operand and P's rows the K-major B operand
      constexpr uint32_t IDESC_QK = FP8 ? ptx::idesc_e4m3_f32(128, CHK, false)
                                        : ptx::idesc_bf16_f32_ab(128, CHK, false, false);
      constexpr uint32_t IDESC_PV = FP8 ? ptx::idesc_e4m3_f32(D, 128, true)
                                        : ptx::idesc_bf16_f32_ab(128, D, false, true);
      // the MMA's q operand: the bf16 tile, or (e4m3) its three parts
      const uint32_t qbase = sm.base_u32 + (FP8 ? OFF_QP : OFF_Q);
      const int b_qfull = FP8 ? B_QP_FULL : B_Q_FULL, b_qempty = FP8 ? B_QP_EMPTY : B_Q_EMPTY;
      // QK cursor: pulls items from the ring; the PV cursor follows through a
      // short local queue (it lags by at most the chunks in flight)
      constexpr int NQUEUE = 8;
      Item queue[NQUEUE];
      int kr = 0;          // ring slots read
      bool ring_done = false, have_q = false;
      Item qit{};
      int qj = 0, qk = 0;  // chunk in item, items with chunks so far
      bool q_ready = false;
      Item pit{};
      int pj = 0, pk = 0;
      long long nq = 0, npv = 0;
      long long t_idle = clock64();
      while (true) {
        bool progress = false;
        if (!have_q && !ring_done) {
          const int slot = kr & (NRING - 1);
          if (ptx::mbar_test_wait(sm.bar(B_ITEM_FULL + slot), (uint32_t)(kr / NRING) & 1)) {
            const long long i = ring_s[slot];
            ptx::mbar_arrive(sm.bar(B_ITEM_EMPTY + slot));
            ++kr;
            if (i >= total) {
              ring_done = true;
            } else {
              const Item it = item_of<G>(i, tp, R, p);
              if (it.nch > 0) {
                qit = it;
                queue[qk % NQUEUE] = it;
                have_q = true;
                qj = 0;
                q_ready = false;
              }
            }
            progress = true;
          }
        }
        if (have_q) {
          if (qj == 0 && !q_ready && ptx::mbar_test_wait(sm.bar(b_qfull), qk & 1)) {
            q_ready = true;
            progress = true;
          }
          const int s = (int)(nq % NSTK);
          const int b = (int)(nq & 1);
          if (q_ready && ptx::mbar_test_wait(sm.bar(B_FULL_K + s), (uint32_t)(nq / NSTK) & 1) &&
              ptx::mbar_test_wait(sm.bar(B_S_EMPTY + b), ((uint32_t)(nq >> 1) & 1) ^ 1)) {
            ptx::tc_fence_after();
            const uint32_t kbase = sm.base_u32 + OFF_K + s * TILE_B;
            if constexpr (FP8) {
              // S = sum over the three q parts of part K^T: rows and keys are
              // 128-byte rows (all of d), 32 bytes of d per MMA
#pragma unroll
              for (int part = 0; part < 3; ++part)
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk) {
                  const uint64_t da =
                      ptx::smem_desc_sw128(qbase + part * QPART_B + kk * 32, 16, 1024);
                  const uint64_t db = ptx::smem_desc_sw128(kbase + kk * 32, 16, 1024);
                  ptx::tc_mma_f8(tmem + S_COL + CHK * b, da, db, IDESC_QK, part > 0 || kk > 0);
                }
            } else {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t da =
                    ptx::smem_desc_sw128(qbase + (kk >> 2) * HALF_B + (kk & 3) * 32, 16, 1024);
                const uint64_t db =
                    ptx::smem_desc_sw128(kbase + (kk >> 2) * HALF_B + (kk & 3) * 32, 16, 1024);
                ptx::tc_mma_f16(tmem + S_COL + CHK * b, da, db, IDESC_QK, kk > 0);
              }
            }
            ptx::tc_commit(sm.bar(B_S_FULL + b));
            ptx::tc_commit(sm.bar(B_EMPTY_K + s));  // the K chunk may be reloaded
            ++nq;
            if (++qj == qit.nch) {
              ptx::tc_commit(sm.bar(b_qempty));  // the q tile (parts) may be rewritten
              qj = 0;
              ++qk;
              q_ready = false;
              have_q = false;
            }
            progress = true;
          }
        }
        if (npv < nq) {
          pit = queue[pk % NQUEUE];
          const int s = (int)(npv % NSTV);
          const int b = (int)(npv & 1);
          const uint32_t bph = (uint32_t)(npv >> 1) & 1;
          const bool o_free = pj > 0 || pk == 0 || ptx::mbar_test_wait(sm.bar(B_O_EMPTY), (pk - 1) & 1);
          if (o_free && ptx::mbar_test_wait(sm.bar(B_P_FULL), (uint32_t)(npv & 1)) &&
              ptx::mbar_test_wait(sm.bar(B_FULL_V + s), (uint32_t)(npv / NSTV) & 1)) {
            ptx::tc_fence_after();
            const uint32_t vbase = sm.base_u32 + OFF_V + s * TILE_B;
            const uint32_t pbase = sm.base_u32 + OFF_P;
            if constexpr (FP8) {
              // O^T (tensor-memory lane = d, column = q row) += V^T P^T: A = the
              // V chunk read MN-major (a 128-byte row is all of d; 32 keys per
              // MMA), B = the two e4m3 parts of P, K-major (a q row's 128 keys
              // in one 128-byte row)
#pragma unroll
              for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int kk = 0; kk < CHK / 32; ++kk) {
                  const uint64_t da = ptx::smem_desc_sw128(vbase + kk * 4096, TILE_B, 1024);
                  const uint64_t db =
                      ptx::smem_desc_sw128(pbase + part * PPART_B + kk * 32, 16, 1024);
                  ptx::tc_mma_f8(tmem + O_COL, da, db, IDESC_PV, pj > 0 || part > 0 || kk > 0);
                }
            } else {
              // A = P, K-major (64 keys per 128-byte swizzled half); B = V read
              // MN-major (16 keys per MMA, d halves HALF_B apart)
#pragma unroll
              for (int kk = 0; kk < CHK / 16; ++kk) {
                const uint64_t da =
                    ptx::smem_desc_sw128(pbase + (kk >> 2) * HALF_B + (kk & 3) * 32, 16, 1024);
                const uint64_t db = ptx::smem_desc_sw128(vbase + kk * 2048, HALF_B, 1024);
                ptx::tc_mma_f16(tmem + O_COL, da, db, IDESC_PV, pj > 0 || kk > 0);
              }
            }
            ptx::tc_commit(sm.bar(B_O_FULL + b));
            ptx::tc_commit(sm.bar(B_P_EMPTY));
            ptx::tc_commit(sm.bar(B_EMPTY_V + s));
            ++npv;
            if (++pj == pit.nch) {
              pj = 0;
              ++pk;
            }
            progress = true;
          }
        } else if (ring_done && !have_q) {
          break;
        }
        if (progress) {
          t_idle = clock64();
        } else {
          if (*sm.abort_flag()) break;
          if (clock64() - t_idle > kWaitClocks) {
            *sm.abort_flag() = 1;
            atomicExch(p.err, 28);
            break;
          }
        }
      }
      // drain: every commit this thread issued must land before exit
      if (nq > 0) {
        drain_bar(sm.bar(B_S_FULL + (int)((nq - 1) & 1)), (uint32_t)((nq - 1) >> 1) & 1);
        drain_bar(sm.bar(B_EMPTY_K + (int)((nq - 1) % NSTK)), (uint32_t)((nq - 1) / NSTK) & 1);
      }
      if (qk > 0) drain_bar(sm.bar(b_qempty), (qk - 1) & 1);
      if (npv > 0) {
        const long long L = npv - 1;
        drain_bar(sm.bar(B_EMPTY_V + (int)(L % NSTV)), (uint32_t)(L / NSTV) & 1);
        drain_bar(sm.bar(B_P_EMPTY), (uint32_t)(L & 1));
        drain_bar(sm.bar(B_O_FULL + (int)(L & 1)), (uint32_t)(L >> 1) & 1);
      }
    }
  } else {
    // ================= softmax + epilogue (warps 0-7) =================
    // Two threads per q tile row: thread t takes keys (and O columns)
    // half * 64 .. half * 64 + 63 of row t & 127; warps w and w + 4 read the
    // same TMEM lanes.  The pair exchanges its half-row max (and, at the end,
    // its half-row sum) through shared memory.
    const int row = tid & 127;
    const int half = tid >> 7;
    const int tok = row / G;   // the row's token within the tile
    const int hd = row % G;    // its query head within the KV head's group
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    float* xch = reinterpret_cast<float*>(sm.base + OFF_XCH);
    // warps w and w + 4 only: the first barrier keeps a slot from being
    // rewritten before the partner has read the previous value
    auto partner = [&](float v) -> float {
      ptx::bar_sync_named(1 + (warp & 3), 64);
      xch[tid] = v;
      ptx::bar_sync_named(5 + (warp & 3), 64);
      return xch[tid ^ 128];
    };
    long long ck = 0;
    int qk_s = 0;  // items with chunks so far (e4m3: q tiles converted)
    const float ksc = FP8 ? __ldg(p.k_scale) : 1.f;
    const float vsc = FP8 ? __ldg(p.v_scale) : 1.f;
    for (int k = 0;; ++k) {
      const long long i = read_item(k, lane == 0);
      if (i >= total) break;
      const Item it = item_of<G>(i, tp, R, p);
      const int rt = it.qt * MQ + tok;  // the row's token within the request
      const bool row_ok = tok < it.ntok;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) +
                            ((int64_t)(it.q0 + rt) * p.num_heads + it.g * G + hd) * D + half * 64;
      if (it.nch == 0) {
        if (row_ok) {
#pragma unroll
          for (int c = 0; c < 8; ++c) reinterpret_cast<uint4*>(orow)[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int lim = row_ok ? it.ctx + rt + 1 : 0;  // keys < lim are visible to the row
      float m_ref = -INFINITY, l = 0.f;
      bool good = true;
      float rs = p.scale_log2;  // logit scale of this row, log2 units
      if constexpr (FP8) {
        // ---- the q tile's three e4m3 parts (the MMA's A operand) ----
        // Row r of the staged bf16 tile, scaled by the power of two 2^e that
        // puts its max |q| in [128, 256), is hi + mid + lo, each part the
        // e4m3 rounding of what the previous ones leave (exact residuals):
        // about 2^-12 relative.  2^-e and k_scale fold into the row's scale.
        good = wait_bar(sm, sm.bar(B_Q_FULL), qk_s & 1, p.err, 31);
        const unsigned char* qrow = sm.base + OFF_Q + half * HALF_B + row * 128;
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(qrow + ((c ^ (row & 7)) << 4));
          w[4 * c] = v.x;
          w[4 * c + 1] = v.y;
          w[4 * c + 2] = v.z;
          w[4 * c + 3] = v.w;
        }
        ptx::mbar_arrive(sm.bar(B_Q_EMPTY));  // the staged tile may be reloaded
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c)
          amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[c])), fabsf(bf16_hi(w[c]))));
        amax = fmaxf(amax, partner(amax));
        const int eb = (int)(__float_as_uint(amax) >> 23);  // 0 for zero / subnormal
        const int e = max(-126, min(126, eb == 0 ? 0 : 134 - eb));
        const float mul = __int_as_float((127 + e) << 23);
        rs = p.scale_log2 * ksc * __int_as_float((127 - e) << 23);
        if (qk_s > 0) good = wait_bar(sm, sm.bar(B_QP_EMPTY), (qk_s - 1) & 1, p.err, 32) && good;
        unsigned char* qp = sm.base + OFF_QP + row * 128;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {  // 16 values of d: one 16-byte piece per part
          uint32_t pw[3][4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const uint32_t w0 = w[c4 * 8 + 2 * q4], w1 = w[c4 * 8 + 2 * q4 + 1];
            float a0 = bf16_lo(w0) * mul, a1 = bf16_hi(w0) * mul;
            float a2 = bf16_lo(w1) * mul, a3 = bf16_hi(w1) * mul;
#pragma unroll
            for (int part = 0; part < 3; ++part) {
              const uint16_t c01 = pack_e4m3x2_rn(a0, a1), c23 = pack_e4m3x2_rn(a2, a3);
              const float2 f01 = e4m3x2_to_float2(c01), f23 = e4m3x2_to_float2(c23);
              a0 -= f01.x;
              a1 -= f01.y;
              a2 -= f23.x;
              a3 -= f23.y;
              pw[part][q4] = (uint32_t)c01 | ((uint32_t)c23 << 16);
            }
          }
          const int o = (((half * 4 + c4) ^ (row & 7)) << 4);
#pragma unroll
          for (int part = 0; part < 3; ++part)
            *reinterpret_cast<uint4*>(qp + part * QPART_B + o) =
                make_uint4(pw[part][0], pw[part][1], pw[part][2], pw[part][3]);
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(sm.bar(B_QP_FULL));
        ++qk_s;
      }
      for (int j = 0; j < it.nch; ++j, ++ck) {
        const int b = (int)(ck & 1);
        const uint32_t bph = (uint32_t)(ck >> 1) & 1;
        const int s = (int)(ck % NSTV);  // the V stage of this chunk
        const uint32_t ph = (uint32_t)(ck / NSTV) & 1;
        // ---- this thread's 64 logits of the row ----
        float sv[2][32];
        good = wait_bar(sm, sm.bar(B_S_FULL + b), bph, p.err, 23) && good;
        ptx::tc_fence_after();
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2)
          ptx::tmem_ld_x32(tmem + lane_base + S_COL + CHK * b + half * 64 + 32 * q2, sv[q2]);
        ptx::tmem_ld_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(sm.bar(B_S_EMPTY + b));
        // every row of a full tile sees every key of a chunk that ends before
        // the tile's first token: no mask (the common case on long contexts)
        const bool whole = it.ntok == MQ && (j + 1) * CHK <= it.ctx + it.qt * MQ + 1;
        const int kl = lim - j * CHK - half * 64;  // visible keys among this thread's 64
        // max of the raw logits (scale > 0), four independent chains
        float hm4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (whole) {
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2)
#pragma unroll
            for (int e = 0; e < 32; ++e) hm4[e & 3] = fmaxf(hm4[e & 3], sv[q2][e]);
        } else {
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2)
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float x = (good && q2 * 32 + e < kl) ? sv[q2][e] : -INFINITY;
              sv[q2][e] = x;
              hm4[e & 3] = fmaxf(hm4[e & 3], x);
            }
        }
        const float hm = fmaxf(fmaxf(hm4[0], hm4[1]), fmaxf(hm4[2], hm4[3]));
        // the row's chunk max in log2 units, the same in both threads
        const float cm = fmaxf(hm, partner(hm)) * rs;
        if constexpr (FP8) {
          // O^T: row r of O is column r of the tensor-memory tile, spread over
          // all 128 lanes (d).  Each row publishes its factor (1 when it keeps
          // its reference max); if any row rescales, every thread rescales its
          // 64 columns once the previous chunk's PV has landed.  The factors
          // alternate between two buffers by chunk, and the reduction barrier
          // below is passed by every thread once per chunk, so a buffer is
          // rewritten only after every thread has used it.
          float alpha = 1.f;
          if (cm > m_ref + kRescaleLog2) {
            if (m_ref != -INFINITY) alpha = fast_exp2(m_ref - cm);
            m_ref = cm;
          }
          float* al = reinterpret_cast<float*>(sm.base + C::OFF_ALPHA) + (int)(ck & 1) * 128;
          if (half == 0) al[row] = alpha;
          if (ptx::bar_red_or(9, NSOFT, alpha != 1.f)) {
            const long long L = ck - 1;
            wait_bar(sm, sm.bar(B_O_FULL + (int)(L & 1)), (uint32_t)(L >> 1) & 1, p.err, 24);
            ptx::tc_fence_after();
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
              float o[32];
              const uint32_t ta = tmem + lane_base + O_COL + half * 64 + 32 * q2;
              ptx::tmem_ld_x32(ta, o);
              ptx::tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] *= al[half * 64 + 32 * q2 + e];
              ptx::tmem_st_x32(ta, o);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
          }
          l *= alpha;
        } else if (cm > m_ref + kRescaleLog2) {
          if (m_ref != -INFINITY) {
            // rescale this half of the row of O (earlier chunks): after their PV
            const float alpha = fast_exp2(m_ref - cm);
            const long long L = ck - 1;
            wait_bar(sm, sm.bar(B_O_FULL + (int)(L & 1)), (uint32_t)(L >> 1) & 1, p.err, 24);
            ptx::tc_fence_after();
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
              float o[32];
              const uint32_t ta = tmem + lane_base + O_COL + half * 64 + 32 * q2;
              ptx::tmem_ld_x32(ta, o);
              ptx::tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] *= alpha;
              ptx::tmem_st_x32(ta, o);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            l *= alpha;
          }
          m_ref = cm;
        }
        const float msafe = m_ref == -INFINITY ? 0.f : m_ref;
        // ---- P (and the V rows past the item's last key) ----
        wait_bar(sm, sm.bar(B_P_EMPTY), (uint32_t)(ck & 1) ^ 1, p.err, 25);
        if (j == it.nch - 1) {
          const int kc = it.kv_end - j * CHK;
          if (kc < CHK) {
            wait_bar(sm, sm.bar(B_FULL_V + s), ph, p.err, 26);
            if (row >= kc) {
              // this thread's 64 columns of V row `row` (e4m3: bytes half * 64
              // .. of the 128-byte row; bf16: the row's 64-column half)
              if constexpr (FP8) {
                unsigned char* vrow = sm.base + OFF_V + s * TILE_B + row * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  *reinterpret_cast<uint4*>(vrow + (((half * 4 + c) ^ (row & 7)) << 4)) =
                      make_uint4(0, 0, 0, 0);
              } else {
                unsigned char* vrow = sm.base + OFF_V + s * TILE_B + half * HALF_B + row * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                  const int cc = (c + row) & 7;
                  *reinterpret_cast<uint4*>(vrow + cc * 16) = make_uint4(0, 0, 0, 0);
                }
              }
            }
          }
        }
        float l4[4] = {0.f, 0.f, 0.f, 0.f};  // this chunk's sum, four chains
        if constexpr (FP8) {
          // 2^(8 - R) p (at most 256) as hi + lo e4m3 parts: bytes half * 64 ..
          // of the row's 128-byte row in each part; the sum adds the parts, so
          // the factor and the rounding cancel in O / l
          unsigned char* prow = sm.base + OFF_P + row * 128;
          // 2^(8 - R) p = 2^(s * scale - m + 8 - R): the factor folds into the
          // FMA's bias; logits and sums go two to an instruction
          const float2 rs2 = make_float2(rs, rs);
          const float bias = C::kPScaleLog2 - msafe;
          const float2 nb2 = make_float2(bias, bias);
          float2 l2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int e = c4 * 16 + q4 * 4;  // key among this thread's 64
              const float2 a01 = fma_x2(make_float2(sv[e >> 5][e & 31], sv[(e + 1) >> 5][(e + 1) & 31]),
                                        rs2, nb2);
              const float2 a23 = fma_x2(make_float2(sv[(e + 2) >> 5][(e + 2) & 31],
                                                    sv[(e + 3) >> 5][(e + 3) & 31]), rs2, nb2);
              const float x[4] = {fast_exp2(a01.x), fast_exp2(a01.y), fast_exp2(a23.x),
                                  fast_exp2(a23.y)};
              const uint16_t h01 = pack_e4m3x2_rn(x[0], x[1]), h23 = pack_e4m3x2_rn(x[2], x[3]);
              const float2 f01 = e4m3x2_to_float2(h01), f23 = e4m3x2_to_float2(h23);
              const uint16_t g01 = pack_e4m3x2_rn(x[0] - f01.x, x[1] - f01.y);
              const uint16_t g23 = pack_e4m3x2_rn(x[2] - f23.x, x[3] - f23.y);
              const float2 r01 = e4m3x2_to_float2(g01), r23 = e4m3x2_to_float2(g23);
              l2[q4] = add_x2(add_x2(l2[q4], add_x2(f01, r01)), add_x2(f23, r23));
              hw[q4] = (uint32_t)h01 | ((uint32_t)h23 << 16);
              lw[q4] = (uint32_t)g01 | ((uint32_t)g23 << 16);
            }
            const int o = (((half * 4 + c4) ^ (row & 7)) << 4);
            *reinterpret_cast<uint4*>(prow + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(prow + PPART_B + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) l4[q4] = l2[q4].x + l2[q4].y;
        } else {
          // keys half * 64 ..: the row's 128-byte half `half` of the P tile
          unsigned char* prow = sm.base + OFF_P + half * HALF_B + row * 128;
          float2 l2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
          const float2 rs2 = make_float2(rs, rs), nm2 = make_float2(-msafe, -msafe);
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            uint32_t w[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const int e = (c8 & 3) * 8 + 2 * e2;
              // p = 2^(s * scale - m): one paired FMA per two logits (masked
              // logits are -inf)
              const float2 x2 =
                  fma_x2(make_float2(sv[c8 >> 2][e], sv[c8 >> 2][e + 1]), rs2, nm2);
              const float2 p2 = make_float2(fast_exp2(x2.x), fast_exp2(x2.y));
              l2[e2] = add_x2(l2[e2], p2);  // before the bf16 rounding the MMA sees
              const __nv_bfloat162 pb = __floats2bfloat162_rn(p2.x, p2.y);
              w[e2] = *reinterpret_cast<const uint32_t*>(&pb);
            }
            *reinterpret_cast<uint4*>(prow + ((c8 ^ (row & 7)) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) l4[e2] = l2[e2].x + l2[e2].y;
        }
        l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(sm.bar(B_P_FULL));
      }
      // ---- epilogue: this half of the row of O after the item's last PV ----
      if constexpr (FP8) {
        // O^T: this thread holds element d = its lane of the 64 q rows of its
        // half (columns).  Every row's sum is published first (0 for rows past
        // the tile's tokens, which are not stored).
        const long long L = ck - 1;
        wait_bar(sm, sm.bar(B_O_FULL + (int)(L & 1)), (uint32_t)(L >> 1) & 1, p.err, 27);
        ptx::tc_fence_after();
        const float lsum = l + partner(l);
        float* ls = reinterpret_cast<float*>(sm.base + C::OFF_LSUM);
        if (half == 0) ls[row] = row_ok ? lsum : 0.f;
        ptx::bar_sync_named(10, NSOFT);
        __nv_bfloat16* ocol = reinterpret_cast<__nv_bfloat16*>(p.out) +
                              ((int64_t)(it.q0 + it.qt * MQ) * p.num_heads + it.g * G) * D + row;
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          float o[32];
          ptx::tmem_ld_x32(tmem + lane_base + O_COL + half * 64 + 32 * q2, o);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int r = half * 64 + 32 * q2 + e;  // q row of the tile: token r / G, head r % G
            const float lr = ls[r];
            if (lr > 0.f)
              ocol[((int64_t)(r / G) * p.num_heads + (r % G)) * D] =
                  __float2bfloat16_rn((o[e] * vsc) / lr);
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(sm.bar(B_O_EMPTY));
      } else {
        const long long L = ck - 1;
        wait_bar(sm, sm.bar(B_O_FULL + (int)(L & 1)), (uint32_t)(L >> 1) & 1, p.err, 27);
        ptx::tc_fence_after();
        const float lsum = l + partner(l);
        const bool store = row_ok && lsum > 0.f;
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          float o[32];
          ptx::tmem_ld_x32(tmem + lane_base + O_COL + half * 64 + 32 * q2, o);
          ptx::tmem_ld_wait();
          if (store) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t w[4];
#pragma unroll
              for (int e2 = 0; e2 < 4; ++e2) {
                const int e = c * 8 + 2 * e2;
                const __nv_bfloat162 ob = __floats2bfloat162_rn(o[e] / lsum, o[e + 1] / lsum);
                w[e2] = *reinterpret_cast<const uint32_t*>(&ob);
              }
              reinterpret_cast<uint4*>(orow)[q2 * 4 + c] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(sm.bar(B_O_EMPTY));
      }
    }
  }

  // ---------------- teardown ----------------
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------- host side ----------------

template <int G, bool FP8>
cudaError_t launch_g(const Params& prm, const CUtensorMap& mk, const CUtensorMap& mv,
                     const CUtensorMap& mq, int num_ctas, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<G, FP8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PCfg<FP8>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_ctas);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = PCfg<FP8>::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_tc_kernel<G, FP8>, mk, mv, mq, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pf

bool prefill_supported(int head_dim, int group, bool fp8, int num_seqs, int block_size) {
  // block_size >= 8 keeps every K/V box 1024-byte aligned in smem (whole
  // 128-byte-swizzle atoms), as in the decode kernels
  return head_dim == pf::D && (group == 1 || group == 2 || group == 4 || group == 8) &&
         num_seqs <= pf::kMaxReqs && block_size >= 8 && tc::encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const PrefillLaunch& a, cudaStream_t stream) {
  using namespace pf;
  tc::EncodeTiledFn enc = tc::encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int group = a.num_heads / a.num_kv_heads;
  const int box_tok = a.block_size < 128 ? a.block_size : 128;
  CUtensorMap mk, mv, mq;
  {
    // [blocks, block_size, H_kv, d] as in the decode kernels: a box is one
    // 128-byte column block (64 bf16 or all 128 e4m3 of d) of box_tok tokens
    // of one KV head
    const cuuint64_t elt = a.fp8 ? 1 : 2;
    const CUtensorMapDataType dt =
        a.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // L2 fills of a row's own size (a 256-byte fill of a 128-byte e4m3 row
    // would also pull the next KV head's row)
    const CUtensorMapL2promotion promo =
        a.fp8 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)a.num_kv_heads, (cuuint64_t)a.block_size,
                          (cuuint64_t)a.num_blocks};
    cuuint64_t strides[3] = {(cuuint64_t)D * elt, (cuuint64_t)a.num_kv_heads * D * elt,
                             (cuuint64_t)a.block_size * a.num_kv_heads * D * elt};
    cuuint32_t box[4] = {(cuuint32_t)(128 / elt), 1, (cuuint32_t)box_tok, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&mk, dt, 4, const_cast<void*>(a.k_cache), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (enc(&mv, dt, 4, const_cast<void*>(a.v_cache), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // q as [num_tokens, H, d]; a tile's box is {64 of d, G heads, 128 / G
    // tokens}: rows token * G + head, tokens past the batch read as zeros
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.num_heads, (cuuint64_t)a.num_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.num_heads * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)(128 / group)};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  Params prm{};
  prm.out = a.out;
  prm.block_tables = a.block_tables;
  prm.seq_lens = a.seq_lens;
  prm.qsl = a.query_start_loc;
  prm.err = static_cast<int*>(a.workspace);
  prm.next_item = reinterpret_cast<unsigned*>(static_cast<char*>(a.workspace) + 4);
  // the item counter starts at zero for every launch (a memset node when captured)
  cudaError_t ez = cudaMemsetAsync(prm.next_item, 0, sizeof(unsigned), stream);
  if (ez != cudaSuccess) return ez;
  prm.min_tokens = a.min_tokens;
  prm.num_seqs = a.num_seqs;
  prm.num_tokens = a.num_tokens;
  prm.num_heads = a.num_heads;
  prm.num_kv_heads = a.num_kv_heads;
  prm.max_blocks = a.max_blocks;
  prm.num_blocks = a.num_blocks;
  prm.block_size = a.block_size;
  int lb = 0;
  while ((1 << lb) < a.block_size) ++lb;
  prm.log2_bs = lb;
  prm.box_tok = box_tok;
  int lx = 0;
  while ((1 << lx) < box_tok) ++lx;
  prm.log2_box = lx;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  prm.k_scale = a.k_scale;
  prm.v_scale = a.v_scale;
  if (a.fp8) {
    switch (group) {
      case 1: return launch_g<1, true>(prm, mk, mv, mq, a.num_ctas, stream);
      case 2: return launch_g<2, true>(prm, mk, mv, mq, a.num_ctas, stream);
      case 4: return launch_g<4, true>(prm, mk, mv, mq, a.num_ctas, stream);
      case 8: return launch_g<8, true>(prm, mk, mv, mq, a.num_ctas, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (group) {
    case 1: return launch_g<1, false>(prm, mk, mv, mq, a.num_ctas, stream);
    case 2: return launch_g<2, false>(prm, mk, mv, mq, a.num_ctas, stream);
    case 4: return launch_g<4, false>(prm, mk, mv, mq, a.num_ctas, stream);
    case 8: return launch_g<8, false>(prm, mk, mv, mq, a.num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
