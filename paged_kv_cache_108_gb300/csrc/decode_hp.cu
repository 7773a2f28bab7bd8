// Paged decode attention on the tensor cores with the KV heads of a cache
// block packed into one tile ("head-packed"), for a bf16 cache with
// head_dim 128.
//
// Same mathematics as the other decode kernels ("4.6 PagedAttention &
// KV-Cache Memory Management", section "The PagedAttention Kernel":
// block-table gather, GQA head map h -> h / G, online softmax; section
// "Performance considerations": split long work across CTAs and merge).
//
// Why packed heads.  In the cache layout [blocks, block_size, H_kv, d] the
// rows of HB consecutive KV heads for TT consecutive tokens of one block form
// one 3-D box, so a single TMA copy {64 of d, TT tokens, HB heads} moves
// 16 KiB where a per-head tile needs eight 2 KiB copies.  Measured on GB300
// with a streaming probe (one CTA per SM, no compute): 16 KiB boxes stream at
// 7.6 TB/s marginal, as fast as plain 32 KiB bulk copies, against 7.0 TB/s
// for 2 KiB boxes.
//
// Tile.  The 128 rows of a K or V tile are (head, token) pairs, head-major:
// row r = hh * TT + tt (the tensor map lists tokens before heads, so the TMA
// writes this order).  The MMA columns are the N = HB x G query heads that
// read those KV heads, column c = hh * G + i.  S = K q^T is computed for all
// rows and columns; column c keeps only the rows of its own KV head (the
// other products are discarded, the tensor pipe being nearly idle in
// decode), and P is block-diagonal, so O = V^T P^T adds only matching rows.
// A head's TT rows lie in one warp: its max and sum reduce with shuffles.
//
// Work split.  A unit is (sequence, group of HB KV heads); its KV is cut into
// chunks of TT tokens, all chunks are numbered (group, sequence, chunk), and
// each persistent CTA (one per SM) takes an equal contiguous range (the walk
// of tc_sched.cuh).  A unit whose chunks fall in one CTA is finished there.
// A piece of a split unit leaves an unnormalised partial (m, l, o) in a slot
// of the CTA that computed it -- slot 0 for the unit its range ends in, slot
// 1 for the unit it starts in -- and the last piece to arrive merges.  The
// merge warp merges pieces finished while the CTA still has work; a CTA's
// final piece is merged by its softmax warps, without counting when every
// other piece has already arrived (the usual case: neighbours take their
// shared units first).  Both read all pieces from the slots in CTA order
// with the same roundings, so the output does not depend on who merges.
//
// Token-major tiles (blocks of fewer than TT tokens).  A chunk is TT
// tokens of whole blocks; its rows are (token, head), r = tt * HB + hh, so
// one copy per block brings that block's rows of all HB heads (the cache
// rows of one token's heads are contiguous).  A column's rows then span the
// four softmax warps: the chunk maximum takes one shared-memory exchange,
// and each thread picks its own head's G columns of the logits.
//
// e4m3 caches.  The MMAs take the cache bytes as they are (kind::f8f6f4):
// the q warp writes each unit's bf16 q, scaled by a power of two, as three
// e4m3 parts (operand rows part * N + c) whose logits add up to q . k; the
// softmax writes 256 p as two e4m3 parts (P rows c and N + c).  The factor
// 256 cancels in o / l, k_scale and the power of two fold into the logit
// scale, v_scale multiplies the output.  Token-major e4m3 tiles of 8 heads
// are loaded by row gathers (four tokens' 1 KiB rows per copy) that land
// unswizzled; the q parts and the outputs are permuted to match (see G4 in
// Cfg).
//
// Warp roles (256 threads):
//   warps 0-3  softmax + epilogue: thread t owns TMEM lane t (row t of the
//              logits tile; element d = t of the output tile);
//   warp 4     producer: per chunk the block ids (a cp.async ring a few
//              chunks ahead) and the chunk's TMA copies (head-major: K and V
//              boxes; token-major: one box per block, or row gathers) into a
//              3-stage (bf16) or 5-stage (e4m3) ring;
//   warp 5     TMEM allocation; one thread issues the MMAs and, for bf16,
//              the q tile's loads (one buffer, reloaded when a unit starts);
//   warp 6     merge warp;
//   warp 7     e4m3: the q warp (q parts, two buffers); bf16: no role after
//              the prologue.
//
// Every mbarrier wait gives up after ~2^31 clocks: the thread records an
// error code in the workspace's first word and marks the CTA aborted, so the
// kernel always terminates; copies in flight are drained (again with a
// bound) before TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_device.cuh"
#include "pa_kernels.cuh"
#include "tc_ptx.cuh"
#include "tc_sched.cuh"

namespace pa {
namespace hp {

using tc::ChunkWalk;
using tc::Smem;
using tc::arrive;
using tc::arrive_expect_last;
using tc::cta_of;
using tc::drain_bar;
using tc::kWaitClocks;
using tc::piece_slot;
using tc::range_lo;
using tc::wait_bar;

constexpr int D = 128;
constexpr int kMaxSeqs = 1024;
constexpr int TAB_SLOTS = 4, TAB_AHEAD = 3;  // block-id ring: one id per chunk
constexpr int kMaxPieces = 160;  // pieces of one split unit: at most the persistent CTAs

// G query heads per KV head (1, 2 or 4).  TM: token-major tiles, for blocks
// of fewer than TT tokens.  FP8: an e4m3 cache.  (Both are described at the
// top of this file.)
template <int G, bool TM, bool FP8>
struct Cfg {
  static constexpr int HB = G >= 2 ? 8 : 16;  // KV heads per tile
  static constexpr int TT = 128 / HB;         // tokens per chunk
  static constexpr int N = HB * G;            // the tile's query heads
  static constexpr int NW = N / 4;            // columns of one softmax warp's heads
  static constexpr int ELT = FP8 ? 1 : 2;     // bytes per K/V element
  // K/V ring stages: 3 x 64 KiB (bf16) or 5 x 32 KiB (e4m3)
  static constexpr int NST = FP8 ? 5 : 3;
  static constexpr int TILE_B = 128 * D * ELT;  // one K or V tile: 128 rows of d
  static constexpr int HALF_B = 128 * 128;      // bf16: one 64-column half of a tile
  // bf16: where the 64-column half h of the 8-row group a of a tile starts:
  // head-major a * 1024 + h * HALF_B; token-major a * 2048 + h * 1024.
  // e4m3: a 128-byte row is all of d; group a starts at a * 1024.
  static constexpr int GRP_B = (TM && !FP8) ? 2048 : 1024;  // between 8-row groups
  static constexpr int HSTEP_B = TM ? 1024 : HALF_B;         // bf16: between the halves
  // e4m3: q as three e4m3 parts (operand rows part * N + c) and P as two
  // (rows part * N + c); the MMA N of the logits and of P V
  static constexpr int NQP = FP8 ? 3 : 1, NPP = FP8 ? 2 : 1;
  static constexpr int NS = N * NQP, NO = N * NPP;
  static constexpr int QTILE_B = FP8 ? NS * 128 : N * D * 2;
  static constexpr int NQBUF = FP8 ? 2 : 1;   // q tiles (e4m3: written by the q warp)
  static constexpr int QHALF_B = N * 128;
  static constexpr int PTILE_B = FP8 ? NO * 128 : N * 128 * 2;  // P^T: rows of 128 tile rows
  static constexpr int PHALF_B = N * 128;
  // TMEM: S[2] of NS columns, then O[2] of NO
  static constexpr int TMEM_NEED = 2 * (NS + NO);
  static constexpr int TMEM_COLS =
      TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
  static constexpr int O_COL = 2 * NS;
  static constexpr int NTHREADS = 256;
  // rescale-factor buffers: three when the factors are published before the
  // per-chunk barrier (head-major), two when after it (token-major)
  static constexpr int NALPHA = TM ? 2 : 3;
  static constexpr int TAB_IDS = TM ? TT : 1;  // block ids per chunk in the id ring
  // e4m3 token-major tiles of 8 heads are loaded by row gathers (see the
  // producer): a token's 8 heads land as one unswizzled 1 KiB group, which
  // the MMAs read through their 128-byte-swizzle descriptors, so row hh of
  // the group sees its 16-byte pieces of d in the order j ^ hh.  The q warp
  // stores the columns of head hh with the same order, and every output
  // element of column c is written back to d ^ (16 * (c / G)).
  static constexpr bool G4 = FP8 && TM && HB == 8;

  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NST * TILE_B;
  static constexpr int OFF_Q = OFF_V + NST * TILE_B;
  static constexpr int OFF_P = OFF_Q + NQBUF * QTILE_B;
  static constexpr int OFF_BAR = OFF_P + 2 * PTILE_B;
  static constexpr int B_FULL_K = 0, B_FULL_V = NST, B_EMPTY = 2 * NST, B_S_FULL = 3 * NST,
                       B_S_EMPTY = B_S_FULL + 2, B_P_FULL = B_S_EMPTY + 2,
                       B_P_EMPTY = B_P_FULL + 2, B_O_FULL = B_P_EMPTY + 2,
                       B_O_EMPTY = B_O_FULL + 2, B_Q_FULL = B_O_EMPTY + 2,
                       B_Q_EMPTY = B_Q_FULL + NQBUF, B_EPI = B_Q_EMPTY + NQBUF,
                       NBARS = B_EPI + 2;
  static constexpr int OFF_TMEM = OFF_BAR + NBARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEM + 4;
  static constexpr int OFF_SQ = OFF_ABORT + 4;      // [3] ints: sequences of the range's ends, first
  static constexpr int OFF_FLAG = OFF_SQ + 12;      // softmax warps' broadcast word
  static constexpr int OFF_QEXP = OFF_FLAG + 4;     // e4m3: [2] floats, 2^-e of each q tile
  static constexpr int OFF_ALPHA = (OFF_QEXP + 8 + 15) / 16 * 16;  // [NALPHA][N] floats: rescale factors
  static constexpr int OFF_ML = OFF_ALPHA + NALPHA * N * 4;  // [N] float2: a piece's (m, l)
  // token-major: [2][4 warps][N] floats, each warp's chunk maxima (and, in
  // an epilogue, its share of the column sums)
  static constexpr int OFF_CMX = OFF_ML + N * 8;
  static constexpr int OFF_CP = OFF_CMX + (TM ? 2 * 4 * N * 4 : 0);  // chunk prefix per sequence, [S+1]
  static constexpr int OFF_NLEN = OFF_CP + (kMaxSeqs + 1) * 4;  // clamped context lengths
  static constexpr int OFF_TAB = OFF_NLEN + kMaxSeqs * 4;       // block-id ring
  static constexpr int SMEM_BYTES = OFF_TAB + TAB_SLOTS * TAB_IDS * 4 + 1024;  // + alignment slack
  static_assert(N % 16 == 0 && N <= 32, "MMA N");
  static_assert(NS <= 256 && NS % 16 == 0 && NO % 16 == 0, "MMA N");
  static_assert(TMEM_NEED <= 512, "tensor memory columns");
  static_assert(TT <= 32, "a KV head's rows stay in one warp");
  static_assert(OFF_BAR % 1024 == 0 && PHALF_B % 1024 == 0 && QHALF_B % 1024 == 0 &&
                    QTILE_B % 1024 == 0 && PTILE_B % 1024 == 0 && TILE_B % 1024 == 0,
                "swizzled tiles stay 1024-byte aligned");
  static_assert(OFF_ALPHA % 16 == 0 && OFF_ML % 8 == 0 && OFF_CMX % 16 == 0, "alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

struct Params {
  void* out;                     // [S, H, D] bf16
  const int32_t* block_tables;
  const int32_t* context_lens;
  int* err;                      // workspace word 0: nonzero if a wait expired / bad id
  unsigned long long* counters;  // [units] (epoch << 16) | arrivals of finished pieces
  float2* ws_ml;                 // [num_ctas][2][N] (m, l) of a piece
  float* ws_o;                   // [num_ctas][2][N][D] unnormalised o of a piece
  float* lse;                    // optional [S * H]: log2-sum-exp of each output row
  const void* q;                 // e4m3: [S * H, D] bf16 q, read by the q warp
  const float* k_scale;          // e4m3: device scalars
  const float* v_scale;
  int num_seqs, num_heads, num_groups, max_blocks, num_blocks, block_size, log2_bs;
  int num_ctas;
  float scale_log2;
  unsigned long long epoch;      // 48-bit tag of this call
  int early_meta;                // previous kernel wrote only the cache
};

// The merge of a split unit's pieces (m_p, l_p, o_p), p in CTA order:
//   M = max_p m_p,  w_p = 2^(m_p - M),  L = sum_p w_p l_p,  a = sum_p w_p o_p,
//   out = a * (1 / L),
// each sum in CTA order with explicit roundings.  Both merge paths (merge
// warp, softmax warps) use exactly these, so a unit's output does not depend
// on which CTA merges it.  A piece may hold no visible key for a column
// (m = -inf, w = 0).
__device__ __forceinline__ float merge_ref(float M) { return M == -INFINITY ? 0.f : M; }
__device__ __forceinline__ float merge_w(float m, float mref) { return fast_exp2(m - mref); }
__device__ __forceinline__ float merge_fold(float a, float w, float o) { return __fmaf_rn(w, o, a); }

template <int G, bool TM, bool FP8>
__global__ void __launch_bounds__(Cfg<G, TM, FP8>::NTHREADS, 1)
    decode_hp_kernel(const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_q, const Params p) {
  using Cf = Cfg<G, TM, FP8>;
  constexpr int HB = Cf::HB, TT = Cf::TT, N = Cf::N, NW = Cf::NW, NST = Cf::NST;
  constexpr int NALPHA = Cf::NALPHA, TAB_IDS = Cf::TAB_IDS, GRP_B = Cf::GRP_B,
                HSTEP_B = Cf::HSTEP_B, NS = Cf::NS, NO = Cf::NO, O_COL = Cf::O_COL,
                NQBUF = Cf::NQBUF, OFF_QEXP = Cf::OFF_QEXP;
  constexpr int TILE_B = Cf::TILE_B, HALF_B = Cf::HALF_B, QTILE_B = Cf::QTILE_B,
                QHALF_B = Cf::QHALF_B, PTILE_B = Cf::PTILE_B, PHALF_B = Cf::PHALF_B,
                TMEM_COLS = Cf::TMEM_COLS, NTHREADS = Cf::NTHREADS;
  constexpr int OFF_K = Cf::OFF_K, OFF_V = Cf::OFF_V, OFF_Q = Cf::OFF_Q, OFF_P = Cf::OFF_P,
                OFF_TMEM = Cf::OFF_TMEM, OFF_SQ = Cf::OFF_SQ, OFF_FLAG = Cf::OFF_FLAG,
                OFF_ALPHA = Cf::OFF_ALPHA, OFF_ML = Cf::OFF_ML, OFF_CP = Cf::OFF_CP,
                OFF_NLEN = Cf::OFF_NLEN, OFF_TAB = Cf::OFF_TAB, OFF_CMX = Cf::OFF_CMX;
  constexpr int B_FULL_K = Cf::B_FULL_K, B_FULL_V = Cf::B_FULL_V, B_EMPTY = Cf::B_EMPTY,
                B_S_FULL = Cf::B_S_FULL, B_S_EMPTY = Cf::B_S_EMPTY, B_P_FULL = Cf::B_P_FULL,
                B_P_EMPTY = Cf::B_P_EMPTY, B_O_FULL = Cf::B_O_FULL, B_O_EMPTY = Cf::B_O_EMPTY,
                B_Q_FULL = Cf::B_Q_FULL, B_Q_EMPTY = Cf::B_Q_EMPTY, B_EPI = Cf::B_EPI,
                NBARS = Cf::NBARS;
  using Walk = ChunkWalk<TT>;
  extern __shared__ unsigned char smem_raw[];
  Smem sm;
  {
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t aligned = (raw + 1023u) & ~1023u;
    sm.base = smem_raw + (aligned - raw);
    sm.base_u32 = aligned;
    sm.off_bar = Cf::OFF_BAR;
    sm.off_abort = Cf::OFF_ABORT;
  }
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = p.num_seqs, H = p.num_heads, HG = p.num_groups;
  const int cap = p.max_blocks << p.log2_bs;
  int* cp = reinterpret_cast<int*>(sm.base + OFF_CP);
  int* nl = reinterpret_cast<int*>(sm.base + OFF_NLEN);

  // ---------------- prologue ----------------
  // Inputs may come from the previous kernel in the stream.  When that kernel
  // is known to write only the KV cache, only the producer waits, right
  // before its first cache load; lengths, tables and q are read at once.
  if (!p.early_meta) ptx::grid_dependency_wait();
  const int n_own = tid < S ? min(__ldg(&p.context_lens[tid]), cap) : 0;
  if (warp == 5) {
    ptx::tmem_alloc(sm.base_u32 + OFF_TMEM, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < NBARS; ++i) {
      uint32_t cnt = 1;
      if ((i >= B_S_EMPTY && i < B_S_EMPTY + 2) || (i >= B_P_FULL && i < B_P_FULL + 2) ||
          (i >= B_O_EMPTY && i < B_O_EMPTY + 2) || (i >= B_EPI && i < B_EPI + 2))
        cnt = 128;
      // e4m3: the q warp's lanes fill a q tile; the segment's last logits
      // MMA and the softmax threads (which read its scale) release it
      if (FP8 && i >= B_Q_FULL && i < B_Q_FULL + NQBUF) cnt = 32;
      if (FP8 && i >= B_Q_EMPTY && i < B_Q_EMPTY + NQBUF) cnt = 1 + 128;
      ptx::mbar_init(sm.bar(i), cnt);
    }
    *sm.abort_flag() = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
  }
  if (!FP8 && warp == 5 && lane == 0) ptx::prefetch_tmap(&tm_q);
  if (warp < 4) {
    // zero both P tiles once: a thread only ever writes its own KV head's
    // columns of its own row, so the off-diagonal blocks stay zero
    uint4* pz = reinterpret_cast<uint4*>(sm.base + OFF_P);
    for (int i = tid; i < 2 * PTILE_B / 16; i += 128) pz[i] = make_uint4(0, 0, 0, 0);
    ptx::fence_proxy_async_smem();
  }
  for (int i = tid; i < S; i += NTHREADS) {
    const int n = i == tid ? n_own : min(__ldg(&p.context_lens[i]), cap);
    nl[i] = n;
    cp[i] = n > 0 ? (n + TT - 1) / TT : 0;
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive prefix in place: cp[i] = sum_{i' < i} ceil(n_i' / TT)
    int carry = 0;
    for (int base = 0; base < S; base += 32) {
      const int i = base + lane;
      const int v = i < S ? cp[i] : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (i < S) cp[i] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) cp[S] = carry;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm.base + OFF_TMEM);
  const long long Ctot = cp[S];  // chunks of one head group
  const long long Ktot = Ctot * HG;
  const int C = (int)(Ktot < p.num_ctas ? Ktot : p.num_ctas);
  const long long lo = (int)blockIdx.x < C ? range_lo(blockIdx.x, Ktot, C) : 0;
  const long long hi = (int)blockIdx.x < C ? range_lo(blockIdx.x + 1, Ktot, C) : 0;
  int* sq = reinterpret_cast<int*>(sm.base + OFF_SQ);
  if (lo < hi) {
    const long long r_lo = lo % Ctot, r_hi = (hi - 1) % Ctot;
    for (int i = tid; i < S; i += NTHREADS) {
      const int a = cp[i], b = cp[i + 1];
      if (a <= r_lo && r_lo < b) sq[0] = i;
      if (a <= r_hi && r_hi < b) sq[1] = i;
      if (a == 0 && b > 0) sq[2] = i;
    }
  }
  __syncthreads();
  const int seq_lo = lo < hi ? sq[0] : 0, seq_hi = lo < hi ? sq[1] : 0;
  const int first_ne = lo < hi ? sq[2] : 0;
  if (warp < 4) {
    // empty sequences get zero rows (spread over the CTAs)
    for (int i = blockIdx.x; i < S; i += gridDim.x) {
      if (nl[i] <= 0) {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + (int64_t)i * H * D;
        for (int e = tid; e < H * D; e += 128) o[e] = __float2bfloat16_rn(0.f);
        if (p.lse)
          for (int r = tid; r < H; r += 128) p.lse[(int64_t)i * H + r] = -INFINITY;
      }
    }
  }

  Walk walk;
  walk.cp = cp;
  walk.S = S;
  walk.Hkv = HG;
  walk.nl = nl;
  walk.Ctot = Ctot;
  walk.first_ne = first_ne;

  if (warp == 4) {
    // ================= producer =================
    // Head-major: one block id per chunk (lane 0) and four copies, each a
    // box {64 of d, TT tokens, HB heads} of one block.  Token-major: a chunk
    // spans TT / block_size blocks; lane i fetches the id of the chunk's
    // block i and copies that block's rows of the HB heads, both halves of
    // d, as one box {64 of d, 8 heads, 2 halves, HB / 8, block_size tokens},
    // for K and for V.  Blocks wholly past the context end are not copied.
    const uint32_t tab = sm.base_u32 + OFF_TAB;
    const int* tab_s = reinterpret_cast<const int*>(sm.base + OFF_TAB);
    const int bs = p.block_size;
    // boxes (blocks) of chunk w that hold context tokens
    auto nboxes = [&](const Walk& w) { return TM ? (w.valid() + bs - 1) >> p.log2_bs : 1; };
    // lanes copy the block ids of a chunk TAB_AHEAD chunks ahead
    auto fetch_id = [&](const Walk& w, int slot) {
      if (lane < nboxes(w))
        cp_async_4(tab + (slot * TAB_IDS + lane) * 4,
                   p.block_tables + (int64_t)w.seq * p.max_blocks + ((w.j * TT) >> p.log2_bs) +
                       lane);
    };
    walk.init(lo, hi, seq_lo, seq_hi);
    Walk ahead = walk;
#pragma unroll 1  // one copy of cold code: its first run pays instruction-fetch misses
    for (int d = 0; d < TAB_AHEAD; ++d) {
      if (!ahead.done()) {
        fetch_id(ahead, d);
        ahead.next();
      }
      cp_async_commit();
    }
    int local = 0;
    for (; !walk.done(); walk.next(), ++local) {
      const int s = local % NST;
      const uint32_t ph = (local / NST) & 1;
      cp_async_wait<TAB_AHEAD - 1>();  // this chunk's ids have landed (each lane's own copy)
      const int nb = nboxes(walk);
      int phys = lane < nb ? tab_s[(local % TAB_SLOTS) * TAB_IDS + lane] : 0;
      if (!TM) phys = __shfl_sync(0xffffffffu, phys, 0);
      if (!wait_bar(sm, sm.bar(B_EMPTY + s), ph ^ 1, p.err, 1)) break;
      if (p.early_meta && local == 0) ptx::grid_dependency_wait();
      if ((!TM || lane < nb) && (unsigned)phys >= (unsigned)p.num_blocks) {
        if (TM || lane == 0) atomicExch(p.err, 3);  // bad block id: load block 0 instead of faulting
        phys = 0;
      }
      if constexpr (TM) {
        // one block's rows of the HB heads (gathers: always the whole tile)
        const uint32_t box_b = (uint32_t)bs * HB * D * Cf::ELT;
        const uint32_t tile_tx = Cf::G4 ? (uint32_t)TILE_B : (uint32_t)nb * box_b;
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(sm.bar(B_FULL_K + s), tile_tx);
          ptx::mbar_arrive_expect_tx(sm.bar(B_FULL_V + s), tile_tx);
        }
        __syncwarp();
        if constexpr (Cf::G4) {
          // Four gathers of four tokens each, for K and for V: a token's rows
          // of the 8 heads are one 1 KiB row of the cache seen as (slot, d of
          // all heads).  Token tk's slot is the id of block tk / B (held by
          // lane tk / B) times B plus tk % B; tokens past the context end
          // repeat the chunk's first token and are masked later.
          int sl[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tk = 4 * (lane & 3) + i;
            const int tkc = tk < walk.valid() ? tk : 0;
            const int pb = __shfl_sync(0xffffffffu, phys, tkc >> p.log2_bs);
            sl[i] = (pb << p.log2_bs) + (tkc & (bs - 1));
          }
          if (lane < 4) {
            const uint32_t off = s * TILE_B + lane * 4096;
            const int col = walk.g * (HB * D / 4);
            ptx::tma_gather4(sm.base_u32 + OFF_K + off, &tm_k, sm.bar(B_FULL_K + s), col, sl[0],
                             sl[1], sl[2], sl[3]);
            ptx::tma_gather4(sm.base_u32 + OFF_V + off, &tm_v, sm.bar(B_FULL_V + s), col, sl[0],
                             sl[1], sl[2], sl[3]);
          }
        } else if (lane < nb) {
          const uint32_t off = s * TILE_B + lane * box_b;
          const int slot0 = phys << p.log2_bs;  // < num_blocks * block_size <= 2^31 - 1
          if constexpr (FP8) {
            // box {128 bytes of d, 8 heads, HB / 8, block_size tokens}
            ptx::tma_load_4d(sm.base_u32 + OFF_K + off, &tm_k, sm.bar(B_FULL_K + s), 0, 0,
                             walk.g * (HB / 8), slot0);
            ptx::tma_load_4d(sm.base_u32 + OFF_V + off, &tm_v, sm.bar(B_FULL_V + s), 0, 0,
                             walk.g * (HB / 8), slot0);
          } else {
            ptx::tma_load_5d(sm.base_u32 + OFF_K + off, &tm_k, sm.bar(B_FULL_K + s), 0, 0, 0,
                             walk.g * (HB / 8), slot0);
            ptx::tma_load_5d(sm.base_u32 + OFF_V + off, &tm_v, sm.bar(B_FULL_V + s), 0, 0, 0,
                             walk.g * (HB / 8), slot0);
          }
        }
      } else if constexpr (FP8) {
        // lane 0: K, lane 1: V; box {128 bytes of d, TT tokens, HB heads}
        const int tok = (walk.j * TT) & (bs - 1);
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(sm.bar(B_FULL_K + s), (uint32_t)TILE_B);
          ptx::mbar_arrive_expect_tx(sm.bar(B_FULL_V + s), (uint32_t)TILE_B);
        }
        __syncwarp();
        if (lane < 2)
          ptx::tma_load_4d(sm.base_u32 + (lane == 0 ? OFF_K : OFF_V) + s * TILE_B,
                           lane == 0 ? (const void*)&tm_k : (const void*)&tm_v,
                           sm.bar((lane == 0 ? B_FULL_K : B_FULL_V) + s), 0, tok, walk.g * HB,
                           phys);
      } else {
        const int tok = (walk.j * TT) & (bs - 1);
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(sm.bar(B_FULL_K + s), (uint32_t)TILE_B);
          ptx::mbar_arrive_expect_tx(sm.bar(B_FULL_V + s), (uint32_t)TILE_B);
        }
        __syncwarp();
        if (lane < 4) {
          // lanes 0, 1: K halves; lanes 2, 3: V halves.  Box {64 of d, TT
          // tokens, HB heads} at (d, token in block, first head, block).
          const bool isk = lane < 2;
          const int hf = lane & 1;
          const uint32_t dst = sm.base_u32 + (isk ? OFF_K : OFF_V) + s * TILE_B + hf * HALF_B;
          ptx::tma_load_4d(dst, isk ? (const void*)&tm_k : (const void*)&tm_v,
                           sm.bar((isk ? B_FULL_K : B_FULL_V) + s), hf * 64, tok, walk.g * HB,
                           phys);
        }
      }
      if (!ahead.done()) {
        fetch_id(ahead, (local + TAB_AHEAD) % TAB_SLOTS);
        ahead.next();
      }
      cp_async_commit();
    }
    cp_async_wait<0>();
    // drain: the last loads issued must land before the CTA can exit
    __syncwarp();
    if (lane == 0) {
      for (int l = max(0, local - NST); l < local; ++l) {
        drain_bar(sm.bar(B_FULL_K + l % NST), (l / NST) & 1);
        drain_bar(sm.bar(B_FULL_V + l % NST), (l / NST) & 1);
      }
    }
  } else if (warp == 5) {
    // ================= MMA issuer (and the q tile) =================
    // Two cursors as in the per-head kernel: the logits MMA of chunk nq and
    // the PV MMA of chunk npv < nq, each issued as soon as its inputs are
    // ready.  The q tile has one buffer: when a segment (a unit's piece)
    // starts, its load is issued once the previous segment's last logits
    // MMA has completed, and that segment's first logits MMA waits for it.
    // e4m3: the q warp fills two q tiles in turn; the MMA thread waits for
    // the segment's tile and releases it after the segment's last logits MMA.
    if (lane == 0) {
      constexpr uint32_t IDESC_QK =
          FP8 ? ptx::idesc_e4m3_f32(128, NS, false) : ptx::idesc_bf16_f32(128, N, false);
      constexpr uint32_t IDESC_PV =
          FP8 ? ptx::idesc_e4m3_f32(128, NO, true) : ptx::idesc_bf16_f32(128, N, true);
      walk.init(lo, hi, seq_lo, seq_hi);
      int nq = 0, npv = 0, seg = 0, cur_q = 0;
      bool q_loading = false, q_ready = false;
      long long t_idle = clock64();
      while (true) {
        bool progress = false;
        if (!walk.done()) {
          const bool first = walk.first_of_segment();
          if (FP8 && first && !q_ready) {
            if (ptx::mbar_test_wait(sm.bar(B_Q_FULL + (seg & 1)), (seg >> 1) & 1)) {
              q_ready = true;
              cur_q = seg & 1;
              progress = true;
            }
          } else if (!FP8 && first && !q_ready) {
            const uint32_t qbase = sm.base_u32 + OFF_Q;
            if (!q_loading) {
              if (seg == 0 || ptx::mbar_test_wait(sm.bar(B_Q_EMPTY), (seg - 1) & 1)) {
                // the unit's query heads g*N .. g*N+N-1: rows of q as [S*H, d]
                const int row = walk.seq * H + walk.g * N;
                ptx::mbar_arrive_expect_tx(sm.bar(B_Q_FULL), (uint32_t)QTILE_B);
                ptx::tma_load_2d(qbase, &tm_q, sm.bar(B_Q_FULL), 0, row);
                ptx::tma_load_2d(qbase + QHALF_B, &tm_q, sm.bar(B_Q_FULL), 64, row);
                q_loading = true;
                progress = true;
              }
            } else if (ptx::mbar_test_wait(sm.bar(B_Q_FULL), seg & 1)) {
              q_loading = false;
              q_ready = true;
              progress = true;
            }
          }
          const int s = nq % NST;
          const int b = nq & 1;
          if ((!first || q_ready) && ptx::mbar_test_wait(sm.bar(B_FULL_K + s), (nq / NST) & 1) &&
              ptx::mbar_test_wait(sm.bar(B_S_EMPTY + b), ((nq >> 1) & 1) ^ 1)) {
            ptx::tc_fence_after();
            const uint32_t kbase = sm.base_u32 + OFF_K + s * TILE_B;
            const uint32_t qbase = sm.base_u32 + OFF_Q + cur_q * QTILE_B;
            if constexpr (FP8) {
              // K and q-part rows are 128 bytes (all of d), 32 per MMA
#pragma unroll
              for (int kk = 0; kk < D / 32; ++kk) {
                const uint64_t da = ptx::smem_desc_sw128(kbase + kk * 32, 16, 1024);
                const uint64_t db = ptx::smem_desc_sw128(qbase + kk * 32, 16, 1024);
                ptx::tc_mma_f8(tmem + NS * b, da, db, IDESC_QK, kk > 0);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t da =
                    ptx::smem_desc_sw128(kbase + (kk >> 2) * HSTEP_B + (kk & 3) * 32, 16, GRP_B);
                const uint64_t db =
                    ptx::smem_desc_sw128(qbase + (kk >> 2) * QHALF_B + (kk & 3) * 32, 16, 1024);
                ptx::tc_mma_f16(tmem + NS * b, da, db, IDESC_QK, kk > 0);
              }
            }
            ptx::tc_commit(sm.bar(B_S_FULL + b));
            if (walk.last_of_segment()) {
              ptx::tc_commit(sm.bar(B_Q_EMPTY + cur_q));
              ++seg;
              q_ready = false;
            }
            walk.next();
            ++nq;
            progress = true;
          }
        }
        if (npv < nq) {
          const int s = npv % NST;
          const int b = npv & 1;
          const uint32_t bph = (npv >> 1) & 1;
          if (ptx::mbar_test_wait(sm.bar(B_P_FULL + b), bph) &&
              ptx::mbar_test_wait(sm.bar(B_O_EMPTY + b), bph ^ 1) &&
              ptx::mbar_test_wait(sm.bar(B_FULL_V + s), (npv / NST) & 1)) {
            ptx::tc_fence_after();
            const uint32_t vbase = sm.base_u32 + OFF_V + s * TILE_B;
            const uint32_t pbase = sm.base_u32 + OFF_P + b * PTILE_B;
            if constexpr (FP8) {
              // A = V^T MN-major: a 128-byte row is all of d for one tile
              // row, so one swizzle atom spans M; 32 rows (4 groups) per MMA.
              // B = P^T, K-major: rows of 128 tile rows, 32 per MMA.
#pragma unroll
              for (int kk = 0; kk < 128 / 32; ++kk) {
                const uint64_t da = ptx::smem_desc_sw128(vbase + kk * 4 * GRP_B, TILE_B, GRP_B);
                const uint64_t db = ptx::smem_desc_sw128(pbase + kk * 32, 16, 1024);
                ptx::tc_mma_f8(tmem + O_COL + NO * b, da, db, IDESC_PV, kk > 0);
              }
            } else {
              // A = V^T read MN-major from the TMA layout (16 rows, two 8-row
              // groups, per MMA; the halves of d HSTEP_B apart);
              // B = P^T, K-major, 64 rows per 128-byte swizzled half
#pragma unroll
              for (int kk = 0; kk < 128 / 16; ++kk) {
                const uint64_t da = ptx::smem_desc_sw128(vbase + kk * 2 * GRP_B, HSTEP_B, GRP_B);
                const uint64_t db =
                    ptx::smem_desc_sw128(pbase + (kk >> 2) * PHALF_B + (kk & 3) * 32, 16, 1024);
                ptx::tc_mma_f16(tmem + O_COL + NO * b, da, db, IDESC_PV, kk > 0);
              }
            }
            ptx::tc_commit(sm.bar(B_O_FULL + b));
            ptx::tc_commit(sm.bar(B_P_EMPTY + b));
            ptx::tc_commit(sm.bar(B_EMPTY + s));
            ++npv;
            progress = true;
          }
        } else if (walk.done()) {
          break;
        }
        if (progress) {
          t_idle = clock64();
        } else {
          if (*sm.abort_flag()) break;
          if (clock64() - t_idle > kWaitClocks) {
            *sm.abort_flag() = 1;
            atomicExch(p.err, 8);
            break;
          }
        }
      }
      // drain: every copy and commit this thread issued must land before exit
      if (q_loading) drain_bar(sm.bar(B_Q_FULL), seg & 1);
      if (seg > 0) {
        if (FP8) drain_bar(sm.bar(B_Q_EMPTY + ((seg - 1) & 1)), ((seg - 1) >> 1) & 1);
        else drain_bar(sm.bar(B_Q_EMPTY), (seg - 1) & 1);
      }
      if (nq > 0) drain_bar(sm.bar(B_S_FULL + ((nq - 1) & 1)), ((nq - 1) >> 1) & 1);
      if (npv > 0) {
        const int L = npv - 1;
        drain_bar(sm.bar(B_EMPTY + L % NST), (L / NST) & 1);
        drain_bar(sm.bar(B_P_EMPTY + (L & 1)), (L >> 1) & 1);
        drain_bar(sm.bar(B_O_FULL + (L & 1)), (L >> 1) & 1);
      }
    }
  } else if (warp == 6) {
    // ================= merge warp =================
    // Follows the same walk; for each split piece other than the CTA's final
    // one it waits for the softmax warps' partial, counts the arrival, and if
    // this was the unit's last piece merges all pieces into the output.
    // Lane l holds d = 4l .. 4l+3 of 8 columns at a time.
    walk.init(lo, hi, seq_lo, seq_hi);
    int e = 0;
    for (; !walk.done(); walk.next()) {
      if (!walk.last_of_segment()) continue;
      {
        Walk nx = walk;
        nx.next();
        if (nx.done()) break;  // the final piece: merged by the softmax warps
      }
      const long long first = walk.k - walk.j;
      const long long last = first + walk.nch - 1;
      const int c0 = cta_of(first, Ktot, C);
      const int c1 = cta_of(last, Ktot, C);
      if (c0 == c1) continue;  // whole unit: the softmax warps wrote the output
      const bool good = wait_bar(sm, sm.bar(B_EPI + (e++ & 1)), 0, p.err, 14);
      if (!good) continue;
      const int u = walk.seq * HG + walk.g;
      int lst = 0;
      if (lane == 0) {
        ptx::fence_acq_rel_gpu();  // the partial the softmax warps wrote precedes the count
        lst = (arrive(&p.counters[u], p.epoch) == c1 - c0 + 1);
        if (lst) ptx::fence_acq_rel_gpu();  // every other piece's partial is visible
      }
      lst = __shfl_sync(0xffffffffu, lst, 0);
      __syncwarp();
      if (!lst) continue;
      const int64_t row0 = (int64_t)walk.seq * H + (int64_t)walk.g * N;
#pragma unroll 1
      for (int cb = 0; cb < N; cb += 8) {
        float M[8], Ls[8];
        float4 a[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          M[k] = -INFINITY;
          Ls[k] = 0.f;
          a[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll 4
        for (int cc = c0; cc <= c1; ++cc) {
          const int64_t base = ((int64_t)cc * 2 + piece_slot(cc, last, Ktot, C)) * N + cb;
#pragma unroll
          for (int k = 0; k < 8; ++k) M[k] = fmaxf(M[k], __ldcg(&p.ws_ml[base + k]).x);
        }
#pragma unroll 2
        for (int cc = c0; cc <= c1; ++cc) {
          const int64_t base = ((int64_t)cc * 2 + piece_slot(cc, last, Ktot, C)) * N + cb;
          float2 ml[8];
          float4 ov[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            ml[k] = __ldcg(&p.ws_ml[base + k]);
            ov[k] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + (base + k) * D) + lane);
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float w = merge_w(ml[k].x, merge_ref(M[k]));
            Ls[k] = merge_fold(Ls[k], w, ml[k].y);
            a[k].x = merge_fold(a[k].x, w, ov[k].x);
            a[k].y = merge_fold(a[k].y, w, ov[k].y);
            a[k].z = merge_fold(a[k].z, w, ov[k].z);
            a[k].w = merge_fold(a[k].w, w, ov[k].w);
          }
        }
        // e4m3: o and l carry the factor 256 of P's encoding (it cancels);
        // v_scale multiplies the output and the log-sum-exp drops the 2^8
        const float vsc = FP8 ? __ldg(p.v_scale) : 1.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float inv = FP8 ? __frcp_rn(Ls[k]) * vsc : __frcp_rn(Ls[k]);
          __nv_bfloat162 lo2 = __floats2bfloat162_rn(a[k].x * inv, a[k].y * inv);
          __nv_bfloat162 hi2 = __floats2bfloat162_rn(a[k].z * inv, a[k].w * inv);
          uint2 w2;
          w2.x = *reinterpret_cast<uint32_t*>(&lo2);
          w2.y = *reinterpret_cast<uint32_t*>(&hi2);
          const int dq = Cf::G4 ? ((4 * lane) ^ (((cb + k) / G) << 4)) : 4 * lane;
          *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                    (row0 + cb + k) * D + dq) = w2;
          if (p.lse && lane == k) p.lse[row0 + cb + k] = M[k] + __log2f(Ls[k]) - (FP8 ? 8.f : 0.f);
        }
      }
      if (lane == 0) p.counters[u] = p.epoch << 16;  // count 0: a replay starts afresh
    }
  } else if (warp == 7) {
    // ================= q warp (e4m3 cache only) =================
    // Per segment, the unit's N bf16 query rows become three e4m3 parts:
    // q * 2^e ~= hi + mid + lo, with 2^e the power of two that puts max |q|
    // in [128, 256); each part is the round-to-nearest of what the previous
    // ones leave (exact fp32 residuals), so the sum holds q to ~2^-12
    // relative.  Part pp of column c is operand row pp * N + c.
    if constexpr (FP8) {
      float* qx = reinterpret_cast<float*>(sm.base + OFF_QEXP);
      constexpr int NPIECE = N * D / 8;  // 16-byte pieces of the unit's bf16 q rows
      constexpr int NV = NPIECE / 32;    // per lane
      walk.init(lo, hi, seq_lo, seq_hi);
      int seg = 0;
      for (; !walk.done(); walk.next()) {
        if (!walk.first_of_segment()) continue;
        const int qs = seg & 1;
        if (!wait_bar(sm, sm.bar(B_Q_EMPTY + qs), ((seg >> 1) & 1) ^ 1, p.err, 2)) break;
        ++seg;
        // the unit's query heads g*N .. g*N+N-1 are consecutive rows of q
        const uint4* src = reinterpret_cast<const uint4*>(p.q) +
                           ((int64_t)walk.seq * H + (int64_t)walk.g * N) * (D / 8);
        uint4 v[NV];
        uint32_t amax = 0;  // bit pattern of max |q| (orders like the float)
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          v[i] = __ldg(src + i * 32 + lane);
          const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
          for (int c = 0; c < 4; ++c)
            amax = max(amax, max((w[c] << 16) & 0x7fffffffu, w[c] & 0x7fff0000u));
        }
        amax = __reduce_max_sync(0xffffffffu, amax);
        const int eb = (int)(amax >> 23);  // biased exponent; 0 for zero / subnormal
        int e = eb == 0 ? 0 : 134 - eb;   // max |q| * 2^e in [128, 256)
        e = max(-126, min(126, e));
        const float mul = __int_as_float((127 + e) << 23);
        if (lane == 0) qx[qs] = __int_as_float((127 - e) << 23);
        unsigned char* qt = sm.base + OFF_Q + qs * QTILE_B;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const int idx = i * 32 + lane;
          const int c = idx >> 4, d0 = (idx & 15) * 8;
          const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
          uint32_t pw[3][2] = {{0, 0}, {0, 0}, {0, 0}};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float a = bf16_lo(w[k]) * mul, b2 = bf16_hi(w[k]) * mul;
#pragma unroll
            for (int part = 0; part < 3; ++part) {
              const uint16_t code = pack_e4m3x2_rn(a, b2);
              const float2 v2 = e4m3x2_to_float2(code);
              a -= v2.x;
              b2 -= v2.y;
              pw[part][k >> 1] |= (uint32_t)code << (16 * (k & 1));
            }
          }
#pragma unroll
          for (int part = 0; part < 3; ++part) {
            // 128-byte swizzle: 16-byte piece index XOR (row & 7); gathered
            // tiles also XOR the piece index with the column's head
            const int r = part * N + c;
            const int xq = Cf::G4 ? c / G : 0;
            const int o = (r >> 3) * 1024 + (r & 7) * 128 +
                          (((((d0 >> 4) ^ xq) ^ (r & 7)) << 4) | (d0 & 8));
            *reinterpret_cast<uint2*>(qt + o) = make_uint2(pw[part][0], pw[part][1]);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(sm.bar(B_Q_FULL + qs));
      }
    }
  } else if (warp < 4) {
    // ================= softmax + epilogue (warps 0-3) =================
    const int t = tid;           // TMEM lane: row (hh, tt) of S; element d of O
    const int hh = TM ? t % HB : t / TT;  // the row's KV head within the tile
    const int tt = TM ? t / HB : t % TT;  // the row's token within the chunk
    const int sel = lane / TT;   // head-major: which of this warp's heads
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float* abuf = reinterpret_cast<float*>(sm.base + OFF_ALPHA);
    float2* mlb = reinterpret_cast<float2*>(sm.base + OFF_ML);
    // token-major: [2][4][N] per-warp chunk maxima, by chunk parity
    float* cmx = reinterpret_cast<float*>(sm.base + OFF_CMX);
    volatile int* flag = reinterpret_cast<volatile int*>(sm.base + OFF_FLAG);
    // e4m3: logits are (S_c + S_{N+c} + S_{2N+c}) * 2^-e * k_scale * scale *
    // log2(e), with 2^-e the q tile's prescale; P carries 256 p, which
    // cancels in o / l; v_scale multiplies the output
    const float ksc = FP8 ? __ldg(p.k_scale) : 1.f;
    const float vsc = FP8 ? __ldg(p.v_scale) : 1.f;
    const float lse_off = FP8 ? 8.f : 0.f;
    const float* qexp = reinterpret_cast<const float*>(sm.base + OFF_QEXP);
    float sscale = p.scale_log2;
    int qseg = 0;
    // running max per column (the same in all TT lanes of a head) and this
    // row's share of the column sums; dm, dl: those of a just-finished piece
    float m[G], l[G], dm[G], dl[G];
    float acc[N];  // o[column][d = t]
#pragma unroll
    for (int i = 0; i < G; ++i) {
      m[i] = -INFINITY;
      l[i] = 0.f;
      dm[i] = -INFINITY;
      dl[i] = 0.f;
    }
#pragma unroll
    for (int c = 0; c < N; ++c) acc[c] = 0.f;
    struct Info {
      int seq, g, nch, j;
      long long k;
      bool last;
    } prev{0, 0, 0, 0, 0, false};
    int split_epi = 0;  // partials handed to the merge warp

    // A piece of unit `in` is done: its (m, l) per column, then the output
    // (whole unit), a partial for the merge warp, or -- the CTA's final
    // piece of a split unit -- the merge itself.
    // lsum (token-major): [4][N] floats free during the call, for the warps'
    // shares of the column sums
    auto epilogue = [&](const Info& in, const float* ms, const float* ls, bool final_piece,
                        float* lsum) {
      float M[N], L[N];
      float2 own_ml;
      if constexpr (TM) {
        // a column's rows are spread over the four warps: each warp sums its
        // own, then the four shares are added in warp order
#pragma unroll
        for (int i = 0; i < G; ++i) {
          float v = ls[i];
#pragma unroll
          for (int off = HB; off < 32; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
          if (lane < HB) lsum[warp * N + hh * G + i] = v;
          if (t < HB) mlb[hh * G + i] = make_float2(ms[i], 0.f);
        }
        ptx::bar_sync_named(2, 128);
#pragma unroll
        for (int c = 0; c < N; ++c) {
          M[c] = mlb[c].x;
          L[c] = ((lsum[c] + lsum[N + c]) + lsum[2 * N + c]) + lsum[3 * N + c];
        }
        const int oc = t < N ? t : 0;
        own_ml = make_float2(mlb[oc].x,
                             ((lsum[oc] + lsum[N + oc]) + lsum[2 * N + oc]) + lsum[3 * N + oc]);
      } else {
#pragma unroll
        for (int i = 0; i < G; ++i) {
          float v = ls[i];
#pragma unroll
          for (int off = TT / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
          if (tt == 0) mlb[hh * G + i] = make_float2(ms[i], v);
        }
        ptx::bar_sync_named(2, 128);
#pragma unroll
        for (int c = 0; c < N; ++c) {
          const float2 v = mlb[c];
          M[c] = v.x;
          L[c] = v.y;
        }
        own_ml = mlb[t < N ? t : 0];
      }
      ptx::bar_sync_named(2, 128);  // all have read mlb (and lsum) before they are rewritten
      const long long first = in.k - in.j;
      const long long last = first + in.nch - 1;
      const int c0 = cta_of(first, Ktot, C);
      const int c1 = cta_of(last, Ktot, C);
      const int64_t row0 = (int64_t)in.seq * H + (int64_t)in.g * N;
      __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + t;
      if (c0 == c1) {
#pragma unroll
        for (int c = 0; c < N; ++c)
          o[(row0 + c) * D + (Cf::G4 ? (t ^ ((c / G) << 4)) - t : 0)] =
              __float2bfloat16_rn(acc[c] * (__fdividef(1.f, L[c]) * vsc));
        if (p.lse && t < N) p.lse[row0 + t] = own_ml.x + __log2f(own_ml.y) - lse_off;
        return;
      }
      const int u = in.seq * HG + in.g;
      const int nseg = c1 - c0 + 1;
      const int64_t mine = ((int64_t)blockIdx.x * 2 + piece_slot(blockIdx.x, last, Ktot, C)) * N;
      auto write_partial = [&]() {
#pragma unroll
        for (int c = 0; c < N; ++c) p.ws_o[(mine + c) * D + t] = acc[c];
        if (t < N) p.ws_ml[mine + t] = own_ml;
      };
      write_partial();
      if (!final_piece) {
        ptx::mbar_arrive(sm.bar(B_EPI + (split_epi++ & 1)));
        return;
      }
      // The CTA's final piece: it counts like the others (one fence for the
      // CTA, after a barrier that orders the other threads' stores) and
      // merges if it was last.  At the kernel's end each global round trip
      // costs ~1.5 us, so the count assumes it is last (one atomic) and the
      // merge fetches the pieces' partials with cp.async into the idle K/V
      // rings, KB pieces per round trip.  The fold reads the pieces in CTA
      // order with the merge warp's arithmetic, so the result does not
      // depend on which CTA merges.
      ptx::bar_sync_named(2, 128);  // every thread's partial stores precede the fence
      if (t == 0) {
        ptx::fence_acq_rel_gpu();  // this CTA's partial precedes its count
        const int f = arrive_expect_last(&p.counters[u], p.epoch, nseg) == nseg ? 1 : 0;
        if (f) ptx::fence_acq_rel_gpu();  // every other piece's partial is visible
        *flag = f;
      }
      ptx::bar_sync_named(2, 128);
      if (*flag == 0) return;
      // Staging in the idle K/V rings: every piece's (m, l), then the
      // weights w_p per column, (M, L) per column, the output tile, and KB
      // pieces' o per round trip.  One round trip brings all (m, l) and the
      // first KB pieces; threads t < N then take column t's M, weights and
      // L, and every thread folds its element d = t of every column.
      constexpr int PMAX = kMaxPieces;
      constexpr int OFF_SML = 0;                              // [PMAX][N] float2
      constexpr int OFF_SW = OFF_SML + PMAX * N * 8;          // [PMAX][N] float
      constexpr int OFF_SC = OFF_SW + PMAX * N * 4;           // [N] float2 (M, L)
      constexpr int OFF_SOT = OFF_SC + N * 8;                 // [N][D] bf16 output tile
      constexpr int OFF_SPO = (OFF_SOT + N * D * 2 + 1023) / 1024 * 1024;  // [KB][N][D] float
      constexpr int KB = (2 * NST * TILE_B - OFF_SPO) / (N * D * 4);
      static_assert(KB >= 1, "staging room for one piece");
      const uint32_t stg = sm.base_u32 + OFF_K;
      const float2* sml = reinterpret_cast<const float2*>(sm.base + OFF_K + OFF_SML);
      float* sw = reinterpret_cast<float*>(sm.base + OFF_K + OFF_SW);
      float2* sc = reinterpret_cast<float2*>(sm.base + OFF_K + OFF_SC);
      __nv_bfloat16* sot = reinterpret_cast<__nv_bfloat16*>(sm.base + OFF_K + OFF_SOT);
      const float* spo = reinterpret_cast<const float*>(sm.base + OFF_K + OFF_SPO);
      auto slot_base = [&](int q) {
        const int cc = c0 + q;
        return ((int64_t)cc * 2 + piece_slot(cc, last, Ktot, C)) * N;
      };
      // o of pieces q0 .. q0 + nb - 1: N * D floats each, 16 bytes per copy
      auto fetch_o = [&](int q0, int nb) {
#pragma unroll 1
        for (int q = 0; q < nb; ++q) {
          const char* so = reinterpret_cast<const char*>(p.ws_o + slot_base(q0 + q) * D);
#pragma unroll
          for (int i = t; i < N * D / 4; i += 128)
            cp_async_16(stg + OFF_SPO + (q * N * D + i * 4) * 4, so + i * 16, 16);
        }
      };
#pragma unroll 1
      for (int i = t; i < nseg * (N / 2); i += 128) {
        const int q = i / (N / 2), j = i - q * (N / 2);
        cp_async_16(stg + OFF_SML + (q * N + 2 * j) * 8,
                    reinterpret_cast<const char*>(p.ws_ml + slot_base(q)) + j * 16, 16);
      }
      fetch_o(0, min(KB, nseg));
      cp_async_commit();
      cp_async_wait<0>();
      ptx::bar_sync_named(2, 128);  // every thread's copies have landed
      if (t < N) {
        float Mx = -INFINITY;
#pragma unroll 1
        for (int q = 0; q < nseg; ++q) Mx = fmaxf(Mx, sml[q * N + t].x);
        const float mref = merge_ref(Mx);
        float Lt = 0.f;
#pragma unroll 1
        for (int q = 0; q < nseg; ++q) {
          const float2 ml = sml[q * N + t];
          const float w = merge_w(ml.x, mref);
          sw[q * N + t] = w;
          Lt = merge_fold(Lt, w, ml.y);
        }
        sc[t] = make_float2(Mx, Lt);
      }
      ptx::bar_sync_named(2, 128);  // weights and (M, L) visible
#pragma unroll
      for (int c = 0; c < N; ++c) acc[c] = 0.f;
#pragma unroll 1
      for (int q0 = 0; q0 < nseg; q0 += KB) {
        const int nb = min(KB, nseg - q0);
        if (q0 > 0) {
          ptx::bar_sync_named(2, 128);  // the previous batch has been read
          fetch_o(q0, nb);
          cp_async_commit();
          cp_async_wait<0>();
          ptx::bar_sync_named(2, 128);
        }
#pragma unroll 1
        for (int q = 0; q < nb; ++q) {
#pragma unroll
          for (int c = 0; c < N; ++c)
            acc[c] = merge_fold(acc[c], sw[(q0 + q) * N + c], spo[(q * N + c) * D + t]);
        }
      }
      // output: element d = t of each column into the tile, then 16-byte rows
#pragma unroll
      for (int c = 0; c < N; ++c) {
        // the merge warp's rounding: a * (1 / L), times v_scale for e4m3
        const float inv = FP8 ? __frcp_rn(sc[c].y) * vsc : __frcp_rn(sc[c].y);
        sot[c * D + (Cf::G4 ? t ^ ((c / G) << 4) : t)] = __float2bfloat16_rn(acc[c] * inv);
      }
      if (p.lse && t < N) p.lse[row0 + t] = sc[t].x + __log2f(sc[t].y) - lse_off;
      ptx::bar_sync_named(2, 128);
#pragma unroll
      for (int i = t; i < N * D / 8; i += 128)
        *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + row0 * D + i * 8) =
            *reinterpret_cast<const uint4*>(sot + i * 8);
      if (t == 0) p.counters[u] = p.epoch << 16;  // count 0: a replay starts afresh
    };

    // fold chunk L's PV result into acc with that chunk's rescale factors
    auto acc_o = [&](int L, const Info& in, bool use_done, bool final_piece, float* lsum) {
      const int b = L & 1;
      const uint32_t bph = (L >> 1) & 1;
      float ov[N];
      const bool good = wait_bar(sm, sm.bar(B_O_FULL + b), bph, p.err, 10);
      ptx::tc_fence_after();
      if constexpr (N == 32) {
        ptx::tmem_ld_x32(tmem + lane_base + O_COL + NO * b, ov);
      } else {
        ptx::tmem_ld_x16(tmem + lane_base + O_COL + NO * b, ov);
      }
      if constexpr (FP8) {
        // columns N + c hold the contribution of P's low parts
        float ol[N];
        if constexpr (N == 32) {
          ptx::tmem_ld_x32(tmem + lane_base + O_COL + NO * b + N, ol);
        } else {
          ptx::tmem_ld_x16(tmem + lane_base + O_COL + NO * b + N, ol);
        }
        ptx::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < N; ++c) ov[c] += ol[c];
      }
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(sm.bar(B_O_EMPTY + b));
      const float* al = abuf + (L % NALPHA) * N;
#pragma unroll
      for (int c = 0; c < N; ++c) acc[c] = acc[c] * al[c] + (good ? ov[c] : 0.f);
      if (in.last) {
        if (use_done) epilogue(in, dm, dl, final_piece, lsum);
        else epilogue(in, m, l, final_piece, lsum);
#pragma unroll
        for (int c = 0; c < N; ++c) acc[c] = 0.f;
      }
    };

    walk.init(lo, hi, seq_lo, seq_hi);
    int local = 0;
    for (; !walk.done(); walk.next(), ++local) {
      const int s = local % NST;
      const uint32_t ph = (local / NST) & 1;
      const int b = local & 1;
      const uint32_t bph = (local >> 1) & 1;
      // ---- logits of this chunk: this warp's heads' columns ----
      // head-major: a warp's rows are whole heads, so it loads only those
      // heads' columns; token-major: every warp holds all HB heads and each
      // thread picks its head's G of the N columns
      constexpr int NL = TM ? N : NW;
      float sl[NL];
      bool good = wait_bar(sm, sm.bar(B_S_FULL + b), bph, p.err, 11);
      ptx::tc_fence_after();
      // e4m3: the logits of q's three parts, columns pp * N + c, are added
#pragma unroll
      for (int pp = 0; pp < Cf::NQP; ++pp) {
        float sp[NL];
        const uint32_t col = tmem + lane_base + NS * b + pp * N + (TM ? 0 : warp * NW);
        if constexpr (NL == 32) {
          ptx::tmem_ld_x32(col, sp);
        } else if constexpr (NL == 16) {
          ptx::tmem_ld_x16(col, sp);
        } else if constexpr (NL == 8) {
          ptx::tmem_ld_x8(col, sp);
        } else {
          ptx::tmem_ld_x4(col, sp);
        }
        ptx::tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < NL; ++k) sl[k] = pp == 0 ? sp[k] : sl[k] + sp[k];
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(sm.bar(B_S_EMPTY + b));
      if constexpr (FP8) {
        if (walk.first_of_segment()) {
          // the q tile's prescale; the q warp may refill the tile once every
          // softmax thread has read it (and the segment's last MMA is done)
          const int qs = qseg & 1;
          good = wait_bar(sm, sm.bar(B_Q_FULL + qs), (qseg >> 1) & 1, p.err, 15) && good;
          sscale = p.scale_log2 * ksc * qexp[qs];
          ptx::mbar_arrive(sm.bar(B_Q_EMPTY + qs));
          ++qseg;
        }
      }
      const int valid = walk.valid();
      float x[G];
#pragma unroll
      for (int i = 0; i < G; ++i) {
        float v = sl[i];
        if constexpr (TM) {
#pragma unroll
          for (int k = 1; k < HB; ++k)
            if (hh == k) v = sl[k * G + i];
        } else {
#pragma unroll
          for (int k = 1; k < 32 / TT; ++k)
            if (sel == k) v = sl[k * G + i];
        }
        x[i] = (good && tt < valid) ? v * sscale : -INFINITY;
      }
      // ---- chunk max per column over its head's TT rows ----
      float cm[G];
#pragma unroll
      for (int i = 0; i < G; ++i) {
        cm[i] = x[i];
        if constexpr (TM) {
#pragma unroll
          for (int off = HB; off < 32; off <<= 1)
            cm[i] = fmaxf(cm[i], __shfl_xor_sync(0xffffffffu, cm[i], off));
        } else {
#pragma unroll
          for (int off = TT / 2; off > 0; off >>= 1)
            cm[i] = fmaxf(cm[i], __shfl_xor_sync(0xffffffffu, cm[i], off));
        }
      }
      if constexpr (TM) {
        // the other warps' rows of the same heads: one exchange per chunk.
        // This barrier also publishes the previous chunk's rescale factors.
        float* cw = cmx + (local & 1) * 4 * N;
        if (lane < HB) {
#pragma unroll
          for (int i = 0; i < G; ++i) cw[warp * N + hh * G + i] = cm[i];
        }
        ptx::bar_sync_named(1, 128);
#pragma unroll
        for (int i = 0; i < G; ++i) {
          const int c = hh * G + i;
          cm[i] = fmaxf(fmaxf(cw[c], cw[N + c]), fmaxf(cw[2 * N + c], cw[3 * N + c]));
        }
      }
      if (walk.first_of_segment()) {
#pragma unroll
        for (int i = 0; i < G; ++i) {
          dm[i] = m[i];
          dl[i] = l[i];
          m[i] = -INFINITY;
          l[i] = 0.f;
        }
      }
      float alpha[G];
      __nv_bfloat16 pb[G];   // bf16: p rounded for the MMA
      uint8_t phi[G], plo[G];  // e4m3: 256 p ~= hi + lo, two e4m3 codes
      float pv[G];
#pragma unroll
      for (int i = 0; i < G; ++i) {
        const float m_new = fmaxf(m[i], cm[i]);
        const float msafe = m_new == -INFINITY ? 0.f : m_new;
        alpha[i] = fast_exp2(m[i] - msafe);
        m[i] = m_new;
        pv[i] = fast_exp2(x[i] - msafe);  // 0 for masked rows
      }
      if constexpr (FP8) {
        // 256 p in [0, 256] keeps e4m3's range; l carries the same factor,
        // so it cancels in o / l.  The residual is exact (Sterbenz).
#pragma unroll
        for (int i = 0; i < G; i += 2) {
          const float a = pv[i] * 256.f, bq = (i + 1 < G ? pv[i + 1] : 0.f) * 256.f;
          const uint16_t ch = pack_e4m3x2_rn(a, bq);
          const float2 hv = e4m3x2_to_float2(ch);
          const uint16_t cl = pack_e4m3x2_rn(a - hv.x, bq - hv.y);
          const float2 lv = e4m3x2_to_float2(cl);
          phi[i] = (uint8_t)(ch & 0xff);
          plo[i] = (uint8_t)(cl & 0xff);
          l[i] = l[i] * alpha[i] + (hv.x + lv.x);
          if (i + 1 < G) {
            phi[i + 1] = (uint8_t)(ch >> 8);
            plo[i + 1] = (uint8_t)(cl >> 8);
            l[i + 1] = l[i + 1] * alpha[i + 1] + (hv.y + lv.y);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < G; ++i) {
          pb[i] = __float2bfloat16_rn(pv[i]);
          l[i] = l[i] * alpha[i] + __bfloat162float(pb[i]);
        }
      }
      if (tt == 0) {
#pragma unroll
        for (int i = 0; i < G; ++i) abuf[(local % NALPHA) * N + hh * G + i] = alpha[i];
      }
      // ---- P tile (and the V rows past the context end) ----
      wait_bar(sm, sm.bar(B_P_EMPTY + b), bph ^ 1, p.err, 12);
      if (valid < TT) {
        wait_bar(sm, sm.bar(B_FULL_V + s), ph, p.err, 13);
        if (tt >= valid) {
          // row t (bf16: its two halves): group t / 8, row t % 8 within it
          unsigned char* vrow = sm.base + OFF_V + s * TILE_B + (t >> 3) * GRP_B + (t & 7) * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int cc = (c + t) & 7;
            *reinterpret_cast<uint4*>(vrow + cc * 16) = make_uint4(0, 0, 0, 0);
            if (!FP8) *reinterpret_cast<uint4*>(vrow + HSTEP_B + cc * 16) = make_uint4(0, 0, 0, 0);
          }
        }
      }
      if constexpr (FP8) {
        // P^T rows c (hi) and N + c (lo): 128 bytes, tile row t at byte t
        unsigned char* pt = sm.base + OFF_P + b * PTILE_B;
        const int chunk = t >> 4, byte = t & 15;
#pragma unroll
        for (int i = 0; i < G; ++i) {
          const int c = hh * G + i, cl = N + c;
          pt[(c >> 3) * 1024 + (c & 7) * 128 + (((chunk ^ (c & 7)) << 4) | byte)] = phi[i];
          pt[(cl >> 3) * 1024 + (cl & 7) * 128 + (((chunk ^ (cl & 7)) << 4) | byte)] = plo[i];
        }
      } else {
        // P^T[c][r]: row c of 128 bf16, 64 per 128-byte swizzled half
        unsigned char* pt = sm.base + OFF_P + b * PTILE_B + (t >> 6) * PHALF_B;
        const int chunk = (t & 63) >> 3;
        const int byte = (t & 7) * 2;
#pragma unroll
        for (int i = 0; i < G; ++i) {
          const int c = hh * G + i;
          *reinterpret_cast<__nv_bfloat16*>(pt + c * 128 + ((chunk ^ (c & 7)) << 4) + byte) = pb[i];
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(sm.bar(B_P_FULL + b));
      // head-major: this chunk's rescale factors are visible after this
      // barrier; token-major: the previous chunk's were at the max exchange
      if (!TM) ptx::bar_sync_named(1, 128);
      // ---- fold the previous chunk's PV result ----
      if (local > 0)
        acc_o(local - 1, prev, walk.first_of_segment(), false, cmx + ((local + 1) & 1) * 4 * N);
      prev = Info{walk.seq, walk.g, walk.nch, walk.j, walk.k, walk.last_of_segment()};
    }
    if (TM) ptx::bar_sync_named(1, 128);  // the last chunk's rescale factors
    if (local > 0) acc_o(local - 1, prev, false, true, cmx + ((local + 1) & 1) * 4 * N);
  }

  // ---------------- teardown ----------------
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------- host side ----------------

template <int G, bool TM, bool FP8>
cudaError_t launch_g(const Params& prm, const CUtensorMap& mk, const CUtensorMap& mv,
                     const CUtensorMap& mq, cudaStream_t stream) {
  using Cf = Cfg<G, TM, FP8>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_hp_kernel<G, TM, FP8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cf::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.num_ctas);
  cfg.blockDim = dim3(Cf::NTHREADS);
  cfg.dynamicSmemBytes = Cf::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  // programmatic dependent launch: the prologue may overlap the previous
  // kernel; the kernel waits for it (griddepcontrol.wait) before reading inputs
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_hp_kernel<G, TM, FP8>, mk, mv, mq, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int heads_per_tile(int group) { return group >= 2 ? 8 : 16; }

}  // namespace hp

size_t hp_workspace_bytes(int64_t num_seqs, int64_t num_heads, int num_ctas) {
  constexpr int64_t kMaxN = 32;  // columns of a tile (an upper bound over the variants)
  size_t off = 256;                                                  // error word
  off += ((size_t)num_seqs * num_heads * 8 + 255) / 256 * 256;       // merge counters (>= units)
  off += ((size_t)num_ctas * 2 * kMaxN * 8 + 255) / 256 * 256;       // (m, l) per piece slot
  off += (size_t)num_ctas * 2 * kMaxN * hp::D * 4;                   // partial o per piece slot
  return off;
}

bool hp_supported(int head_dim, int group, bool fp8, int num_seqs, int num_kv_heads,
                  int block_size, int tokens_per_seq) {
  // a tile holds HB KV heads x TT tokens: H_kv must be a multiple of HB.
  // Blocks of at least TT tokens give head-major tiles (a chunk inside one
  // block), smaller blocks token-major tiles (a chunk of whole blocks).
  (void)fp8;  // bf16 or e4m3
  if (head_dim != hp::D || tokens_per_seq != 1) return false;
  if (group != 1 && group != 2 && group != 4) return false;
  const int hb = hp::heads_per_tile(group);
  return num_kv_heads % hb == 0 && block_size >= 1 && num_seqs <= hp::kMaxSeqs &&
         tc::encode_fn() != nullptr;
}

cudaError_t launch_decode_hp(const TcLaunch& a, cudaStream_t stream) {
  using namespace hp;
  tc::EncodeTiledFn enc = tc::encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int group = a.num_heads / a.num_kv_heads;
  const int hb = heads_per_tile(group);
  const int tt = 128 / hb;
  const int ncol = hb * group;
  const bool tm = a.block_size < tt;  // token-major tiles
  const bool fp8 = a.fp8;
  if (a.num_ctas > kMaxPieces) return cudaErrorInvalidValue;  // a unit's pieces must fit the merge staging
  CUtensorMap mk, mv, mq;
  if (fp8) {
    // e4m3: a row (one token of one head) is 128 bytes, all of d.
    // Head-major: (d, token, head, block), box {128, TT, HB, 1}; token-major:
    // (d, head mod 8, head / 8, slot = block * block_size + token), box
    // {128, 8, HB / 8, block_size}: one block's rows of HB heads, 8-row
    // (1024-byte) groups per token.
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4];
    if (!tm) {
      dims[0] = D; dims[1] = a.block_size; dims[2] = a.num_kv_heads; dims[3] = a.num_blocks;
      strides[0] = (cuuint64_t)a.num_kv_heads * D;
      strides[1] = D;
      strides[2] = (cuuint64_t)a.block_size * a.num_kv_heads * D;
      box[0] = 128; box[1] = tt; box[2] = hb; box[3] = 1;
    } else {
      dims[0] = D; dims[1] = 8; dims[2] = a.num_kv_heads / 8;
      dims[3] = (cuuint64_t)a.num_blocks * a.block_size;
      strides[0] = D;
      strides[1] = 8 * (cuuint64_t)D;
      strides[2] = (cuuint64_t)a.num_kv_heads * D;
      box[0] = 128; box[1] = 8; box[2] = hb / 8; box[3] = a.block_size;
    }
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (tm && hb == 8) {
      // row gathers: the cache as (32-bit words of d over all heads, slot);
      // a gathered row is one token's 8 heads of group g (256 words, 1 KiB),
      // copied without swizzle
      cuuint64_t gd[2] = {(cuuint64_t)a.num_kv_heads * D / 4,
                          (cuuint64_t)a.num_blocks * a.block_size};
      cuuint64_t gs[1] = {(cuuint64_t)a.num_kv_heads * D};
      cuuint32_t gb[2] = {(cuuint32_t)hb * D / 4, 1};
      cuuint32_t ge[2] = {1, 1};
      if (enc(&mk, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(a.k_cache), gd, gs, gb,
              ge, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
      if (enc(&mv, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(a.v_cache), gd, gs, gb,
              ge, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    } else {
    if (enc(&mk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(a.k_cache), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (enc(&mv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(a.v_cache), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    }
  } else if (!tm) {
    // [blocks, block_size, H_kv, d] listed as (d, token, head, block) so that
    // a box {64, TT, HB, 1} lands head-major: row = head * TT + token
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)a.block_size, (cuuint64_t)a.num_kv_heads,
                          (cuuint64_t)a.num_blocks};
    cuuint64_t strides[3] = {(cuuint64_t)a.num_kv_heads * D * 2, (cuuint64_t)D * 2,
                             (cuuint64_t)a.block_size * a.num_kv_heads * D * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)tt, (cuuint32_t)hb, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.k_cache), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (enc(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.v_cache), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  } else {
    // The same cache viewed as (d in 64s, head mod 8, half of d, head / 8,
    // slot = block * block_size + token); a box {64, 8, 2, HB / 8, block_size}
    // is one block's rows of HB heads and lands token-major: for each token,
    // for each 8 heads, an 8-row (1024-byte) group per half of d.
    cuuint64_t dims[5] = {64, 8, 2, (cuuint64_t)a.num_kv_heads / 8,
                          (cuuint64_t)a.num_blocks * a.block_size};
    cuuint64_t strides[4] = {(cuuint64_t)D * 2, 128, 8 * (cuuint64_t)D * 2,
                             (cuuint64_t)a.num_kv_heads * D * 2};
    cuuint32_t box[5] = {64, 8, 2, (cuuint32_t)hb / 8, (cuuint32_t)a.block_size};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (enc(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(a.k_cache), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (enc(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(a.v_cache), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // q as [S * H rows, d]; a unit's box is {64 of d, its N query heads}
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)a.num_seqs * a.num_heads};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)ncol};
    cuuint32_t es[2] = {1, 1};
    if (enc(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.q), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  Params prm{};
  prm.out = a.out;
  prm.block_tables = a.block_tables;
  prm.context_lens = a.context_lens;
  prm.lse = a.lse;
  prm.q = a.q;
  prm.k_scale = a.k_scale;
  prm.v_scale = a.v_scale;
  char* ws = static_cast<char*>(a.workspace);
  size_t off = 0;
  prm.err = reinterpret_cast<int*>(ws + off);
  off += 256;
  prm.counters = reinterpret_cast<unsigned long long*>(ws + off);
  off += ((size_t)a.num_seqs * a.num_heads * 8 + 255) / 256 * 256;
  prm.ws_ml = reinterpret_cast<float2*>(ws + off);
  off += ((size_t)a.num_ctas * 2 * 32 * 8 + 255) / 256 * 256;
  prm.ws_o = reinterpret_cast<float*>(ws + off);
  prm.num_seqs = a.num_seqs;
  prm.num_heads = a.num_heads;
  prm.num_groups = a.num_kv_heads / hb;
  prm.max_blocks = a.max_blocks;
  prm.num_blocks = a.num_blocks;
  prm.block_size = a.block_size;
  int lb = 0;
  while ((1 << lb) < a.block_size) ++lb;
  prm.log2_bs = lb;
  prm.num_ctas = a.num_ctas;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  prm.early_meta = a.early_meta ? 1 : 0;
  prm.epoch = tc::next_call_epoch();
  switch (group * 4 + (tm ? 2 : 0) + (fp8 ? 1 : 0)) {
    case 4: return launch_g<1, false, false>(prm, mk, mv, mq, stream);
    case 5: return launch_g<1, false, true>(prm, mk, mv, mq, stream);
    case 6: return launch_g<1, true, false>(prm, mk, mv, mq, stream);
    case 7: return launch_g<1, true, true>(prm, mk, mv, mq, stream);
    case 8: return launch_g<2, false, false>(prm, mk, mv, mq, stream);
    case 9: return launch_g<2, false, true>(prm, mk, mv, mq, stream);
    case 10: return launch_g<2, true, false>(prm, mk, mv, mq, stream);
    case 11: return launch_g<2, true, true>(prm, mk, mv, mq, stream);
    case 16: return launch_g<4, false, false>(prm, mk, mv, mq, stream);
    case 17: return launch_g<4, false, true>(prm, mk, mv, mq, stream);
    case 18: return launch_g<4, true, false>(prm, mk, mv, mq, stream);
    case 19: return launch_g<4, true, true>(prm, mk, mv, mq, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
