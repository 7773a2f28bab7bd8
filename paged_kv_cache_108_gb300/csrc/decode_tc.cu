// Paged decode attention on the 5th-generation tensor cores (tcgen05) with
// TMA-staged operands, for a bf16 cache with head_dim 128.
//
// Same mathematics as the SIMT kernel ("4.6 PagedAttention & KV-Cache Memory
// Management", section "The PagedAttention Kernel": block-table gather, GQA
// head map h -> h / G, online softmax; section "Performance considerations":
// split the sequence across CTAs and merge), organised for Blackwell:
//
// Work split.  The KV of every (sequence, KV head) unit is cut into chunks
// (128 tokens for bf16, 256 for e4m3); all chunks of all units are numbered
// in (head, sequence, chunk) order and each persistent CTA (one per SM) takes
// an equal contiguous range of that numbering.  Head-major order puts the
// units of one KV head side by side, so sequences forked from a common
// prefix (adjacent in the batch) read their shared blocks within a few
// microseconds of each other, mostly from L2.  A unit whose chunks all fall in one CTA is finished
// there; otherwise each CTA writes an unnormalised partial (m, l, o) for its
// piece ("segment"), and the last of the unit's CTAs to finish merges the
// partials.  The arrival count of a unit is a 64-bit word tagged with a
// per-call epoch (48 bits) supplied by the host: a word whose tag is not the
// current epoch counts as zero, so the workspace needs no initialisation and
// may be shared by calls of different shapes; the merging CTA leaves the
// word at (epoch, 0), so replaying the same launch also starts from zero.
// Load balance is one chunk, whatever the mix of context lengths.
//
// Warp roles (256 threads):
//   warps 0-3  softmax + epilogue: thread t owns TMEM lane t (a token of the
//              logits tile, a d-element of the output tile);
//   warp 4     producer: per chunk, TMA tensor loads of each physical block's
//              K rows (and, for an e4m3 cache, V rows; 4-D tensor map
//              [blocks, block_size, H_kv, d], 128-byte swizzle, 128-byte-wide
//              boxes) into a 3-stage ring and, for bf16, each segment's q rows.
//              Blocks of fewer than 8 tokens cannot fill a 1024-byte swizzle
//              atom with one box: their rows are gathered instead, 16 bytes
//              per lane and cp.async, into the same swizzled layout;
//   warp 5     TMEM allocation and the single MMA-issuing thread;
//   warp 6     merge warp: counts finished pieces of split units and merges
//              a unit's pieces when its last piece is done;
//   warp 7     bf16: a second producer for the V rows; e4m3: the q warp.
// Per chunk c (double-buffered TMEM tiles S[c&1], O[c&1] and smem P[c&1]):
//   S = K_c q^T         tcgen05.mma M=128 tokens, N=16 (query heads padded),
//                       K=128 (d); A = K tile (K-major), B = q tile (K-major)
//   softmax             tcgen05.ld S, scale, chunk max across 128 lanes,
//                       running max m, alpha = 2^(m_old - m_new),
//                       p = 2^(s - m_new) rounded to bf16 into smem P
//   O_c = V_c^T P^T     tcgen05.mma M=128 (d), N=16, K=128 tokens;
//                       A = V tile read MN-major straight from the TMA layout
//   acc = acc*alpha + O_c   in registers after tcgen05.ld
// Tokens past a unit's end get p = 0 and their V rows are zeroed in smem, so
// stale or non-finite pool bytes never reach the output.
//
// Every mbarrier wait gives up after ~2^31 clocks: the thread records an
// error code in the workspace's first word, marks the CTA aborted (later
// waits return at once), so the kernel always terminates; copies in flight
// are drained (again with a bound) before TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <atomic>
#include <mutex>

#include "pa_device.cuh"
#include "pa_kernels.cuh"
#include "tc_ptx.cuh"
#include "tc_sched.cuh"

namespace pa {
namespace tc {

constexpr int D = 128;
constexpr int NQ = 16;                 // MMA N of PV: query heads (bf16), hi/lo rows of P (fp8)
constexpr int kMaxSeqs = 1024;
constexpr int kMaxCols = 16;           // columns of a unit (the MMA N of PV)
constexpr int TAB_SLOTS = 4, TAB_AHEAD = 3;  // block-id ring: 4 chunks, fetched 3 ahead

// Shared-memory layout and roles for a bf16 or an fp8-e4m3 cache, with K/V
// rows arriving as TMA boxes or (GATHER, block_size < 8) gathered by cp.async.
template <bool FP8, bool GATHER>
struct Cfg {
  // block ids per chunk in the ring: one per TMA box (block_size >= 8 keeps a
  // chunk within 32 boxes), or one per block of a gathered chunk (up to a
  // 256-token e4m3 chunk of 1-token blocks)
  static constexpr int TAB_W = GATHER ? 256 : 32;
  // tokens per chunk: 128 bf16 or 256 e4m3 rows, 32 KiB of K and 32 of V
  static constexpr int CH = FP8 ? 256 : 128;
  static constexpr int NHALF = CH / 128;        // 128-token halves (one logits MMA each)
  static constexpr int NST = 3;                 // K/V ring stages (192 KiB)
  static constexpr int ELT = FP8 ? 1 : 2;       // bytes per element of the K/V/q/P tiles
  static constexpr int TILE_B = CH * D * ELT;   // one K or V chunk
  // 16 KiB: one 128-byte-wide column block of a bf16 tile (64 of d for 128
  // tokens), or one 128-token half of an e4m3 tile (all of d)
  static constexpr int HALF_B = 128 * 128;
  // MMA N of QK: the query heads padded to 16 (bf16); three e4m3 parts of
  // every head, rows h, 8 + h and 16 + h, padded to 32 (fp8)
  static constexpr int NQ_S = FP8 ? 32 : 16;
  static constexpr int QTILE_B = NQ_S * D * ELT;
  // TMEM: S[2] of NHALF x NQ_S columns, then O[2] x 16 (a power of two >= 32
  // columns is allocated)
  static constexpr int S_W = NHALF * NQ_S;
  static constexpr int O_COL = 2 * S_W;
  static constexpr int TMEM_COLS = FP8 ? 256 : 64;
  static constexpr int PTILE_B = NQ * CH * ELT;
  // bf16: two producer warps issue the TMA loads, warp 4 the K rows (and
  // q) and warp 7 the V rows (measured 4 % faster on the MHA serving mix,
  // equal elsewhere).  fp8: warp 4 issues both (a second producer measured
  // slower there) and warp 7 prepares q.
  static constexpr bool TWO_PROD = !FP8;
  static constexpr int VPROD = TWO_PROD ? 7 : 4;
  static constexpr int NTHREADS = 256;

  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NST * TILE_B;
  static constexpr int OFF_Q = OFF_V + NST * TILE_B;
  static constexpr int OFF_P = OFF_Q + 2 * QTILE_B;
  static constexpr int OFF_BAR = OFF_P + 2 * PTILE_B;
  // barrier indices
  static constexpr int B_FULL_K = 0, B_FULL_V = NST, B_EMPTY = 2 * NST, B_S_FULL = 3 * NST,
                       B_S_EMPTY = B_S_FULL + 2, B_P_FULL = B_S_EMPTY + 2,
                       B_P_EMPTY = B_P_FULL + 2, B_O_FULL = B_P_EMPTY + 2,
                       B_O_EMPTY = B_O_FULL + 2, B_Q_FULL = B_O_EMPTY + 2,
                       B_Q_EMPTY = B_Q_FULL + 2, B_EPI = B_Q_EMPTY + 2, NBARS = B_EPI + 2;
  static constexpr int OFF_TMEM = OFF_BAR + NBARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEM + 4;
  static constexpr int OFF_SQ = OFF_ABORT + 4;     // [3] ints: sequences of the range's ends, first
  static constexpr int OFF_QEXP = OFF_SQ + 12;     // [2] floats: 2^-e of each q tile (fp8)
  static constexpr int OFF_RED = OFF_QEXP + 8;     // [2][4][16] floats, chunk max per column
  static constexpr int OFF_LRED = OFF_RED + 2 * 4 * 16 * 4;  // [4][16] floats, epilogue sums
  static constexpr int OFF_CP = OFF_LRED + 4 * 16 * 4;       // chunk prefix per sequence, [S+1]
  static constexpr int OFF_NLEN = OFF_CP + (kMaxSeqs + 1) * 4;  // clamped context lengths
  static constexpr int OFF_TAB = OFF_NLEN + kMaxSeqs * 4;       // block-id rings (K, V producer)
  static constexpr int SMEM_BYTES = OFF_TAB + 2 * TAB_SLOTS * TAB_W * 4 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(OFF_BAR % 1024 == 0, "tiles stay 1024-byte aligned");
};

struct Params {
  void* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int* err;        // workspace word 0: nonzero if a wait expired / bad id
  unsigned long long* counters;  // [units] (epoch << 16) | arrivals of finished segments
  float2* ws_ml;   // [num_ctas][2][G]: (m, l) of a split unit's piece (slot: piece_slot)
  float* ws_o;     // [num_ctas][2][G][D]: its unnormalised o
  int num_seqs, num_heads, num_kv_heads, max_blocks, num_blocks, block_size, log2_bs;
  int num_ctas, box_tok, log2_box;
  float scale_log2;
  // Columns of a unit: c = j * gq + i is query head g * gq + i of the
  // sequence's j-th new token (ntok tokens per sequence, the last ntok
  // positions of its context; ntok = 1 for decode).  Token j sees keys at
  // positions < n - ntok + j + 1.
  int gq, log2_gq, ntok;
  int causal;                // 0: every column sees all n keys (a shared prefix)
  float* lse;                // optional [rows]: log2-sum-exp of each output row's logits
  const void* q;             // [S * ntok, H, D] bf16 (read directly by the fp8 kernel's q warp)
  const float* k_scale;      // fp8: per-tensor dequantisation scales (device scalars)
  const float* v_scale;
  unsigned long long epoch;  // 48-bit tag of this call
  int early_meta;            // previous kernel wrote only the cache
  // the caches' base addresses, for the gathered copies (block_size < 8: a
  // TMA box of fewer than 8 rows cannot fill a whole 1024-byte swizzle atom)
  const unsigned char* kc;
  const unsigned char* vc;
};

template <int G, bool FP8, bool GATHER>
__global__ void __launch_bounds__(Cfg<FP8, GATHER>::NTHREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_q, const Params p) {
  using Cf = Cfg<FP8, GATHER>;
  constexpr int TAB_W = Cf::TAB_W;
  constexpr int CH = Cf::CH, NHALF = Cf::NHALF, NQ_S = Cf::NQ_S, S_W = Cf::S_W,
                O_COL = Cf::O_COL, TMEM_COLS = Cf::TMEM_COLS;
  using Walk = ChunkWalk<CH>;
  constexpr int NST = Cf::NST, TILE_B = Cf::TILE_B, HALF_B = Cf::HALF_B,
                QTILE_B = Cf::QTILE_B, PTILE_B = Cf::PTILE_B, NTHREADS = Cf::NTHREADS;
  constexpr int OFF_K = Cf::OFF_K, OFF_V = Cf::OFF_V, OFF_Q = Cf::OFF_Q, OFF_P = Cf::OFF_P,
                OFF_TMEM = Cf::OFF_TMEM, OFF_SQ = Cf::OFF_SQ, OFF_QEXP = Cf::OFF_QEXP,
                OFF_RED = Cf::OFF_RED, OFF_LRED = Cf::OFF_LRED, OFF_CP = Cf::OFF_CP,
                OFF_NLEN = Cf::OFF_NLEN, OFF_TAB = Cf::OFF_TAB;
  constexpr int B_FULL_K = Cf::B_FULL_K, B_FULL_V = Cf::B_FULL_V, B_EMPTY = Cf::B_EMPTY,
                B_S_FULL = Cf::B_S_FULL, B_S_EMPTY = Cf::B_S_EMPTY, B_P_FULL = Cf::B_P_FULL,
                B_P_EMPTY = Cf::B_P_EMPTY, B_O_FULL = Cf::B_O_FULL, B_O_EMPTY = Cf::B_O_EMPTY,
                B_Q_FULL = Cf::B_Q_FULL, B_Q_EMPTY = Cf::B_Q_EMPTY, B_EPI = Cf::B_EPI,
                NBARS = Cf::NBARS;
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
  const int S = p.num_seqs, Hkv = p.num_kv_heads, H = p.num_heads;
  const int cap = p.max_blocks << p.log2_bs;
  int* cp = reinterpret_cast<int*>(sm.base + OFF_CP);
  int* nl = reinterpret_cast<int*>(sm.base + OFF_NLEN);

  // ---------------- prologue ----------------
  // Inputs may come from the previous kernel in the stream.  When that kernel
  // is known to write only the KV cache, only the producer waits, right
  // before its first cache load; lengths, tables and q are read at once.
  if (!p.early_meta) ptx::grid_dependency_wait();
  // the context lengths first: their load is the prologue's longest latency
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
      if (GATHER && i < B_EMPTY) cnt = 32;  // gathered rows: every producer lane arrives
      if (FP8 && i >= B_Q_FULL && i < B_Q_FULL + 2) cnt = 32;        // the q warp's lanes
      if (FP8 && i >= B_Q_EMPTY && i < B_Q_EMPTY + 2) cnt = 1 + 128;  // MMA + softmax threads
      ptx::mbar_init(sm.bar(i), cnt);
    }
    *sm.abort_flag() = 0;
    ptx::fence_mbar_init();
  }
  if ((warp == 4 || warp == Cf::VPROD) && lane == 0) {
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    ptx::prefetch_tmap(&tm_q);
  }
  if (warp < 4) {
    // zero both q and P tiles: rows past a unit's columns stay zero
    constexpr int zoff = OFF_Q;
    constexpr int zbytes = 2 * (QTILE_B + PTILE_B);
    uint4* pz = reinterpret_cast<uint4*>(sm.base + zoff);
    for (int i = tid; i < zbytes / 16; i += 128) pz[i] = make_uint4(0, 0, 0, 0);
    ptx::fence_proxy_async_smem();
  }
  // chunk counts per sequence, loaded by all threads at once
  for (int i = tid; i < S; i += NTHREADS) {
    const int n = i == tid ? n_own : min(__ldg(&p.context_lens[i]), cap);
    nl[i] = n;
    cp[i] = n > 0 ? (n + CH - 1) / CH : 0;
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive prefix in place: cp[i] = sum_{i' < i} ceil(n_i' / CH)
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
  const long long Ctot = cp[S];         // chunks of one KV head
  const long long Ktot = Ctot * Hkv;
  // only min(CTAs, chunks) CTAs take work, so every working CTA owns at least
  // one chunk and a unit never spans more CTAs than it has chunks
  const int C = (int)(Ktot < p.num_ctas ? Ktot : p.num_ctas);
  const long long lo = (int)blockIdx.x < C ? range_lo(blockIdx.x, Ktot, C) : 0;
  const long long hi = (int)blockIdx.x < C ? range_lo(blockIdx.x + 1, Ktot, C) : 0;
  // the sequences holding chunks lo and hi - 1 and the first sequence with
  // chunks, found by all threads at once (chunk k of the (head, sequence,
  // chunk) numbering is chunk k mod Ctot of its head)
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
        // all rows of the sequence's tokens: zero output, log2-sum-exp -inf
        const int64_t rows = (int64_t)p.ntok * H;
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + (int64_t)i * rows * D;
        for (int64_t e = tid; e < rows * D; e += 128) o[e] = __float2bfloat16_rn(0.f);
        if (p.lse)
          for (int64_t r = tid; r < rows; r += 128) p.lse[(int64_t)i * rows + r] = -INFINITY;
      }
    }
  }

  Walk walk;
  walk.cp = cp;
  walk.S = S;
  walk.Hkv = Hkv;
  walk.nl = nl;
  walk.Ctot = Ctot;
  walk.first_ne = first_ne;
  // output row of column h of unit (seq, g): query head g*gq + (h mod gq) of
  // the sequence's token h / gq
  auto out_row = [&](int seq, int g, int h) -> int64_t {
    return ((int64_t)seq * p.ntok + (h >> p.log2_gq)) * H + (int64_t)g * p.gq + (h & (p.gq - 1));
  };

  if (warp == 4 || warp == Cf::VPROD) {
    // ================= producers (K: warp 4, V: warp VPROD) =================
    // Block ids travel through a shared-memory ring filled by 4-byte cp.async
    // copies TAB_AHEAD chunks ahead (TMA boxes: lane b copies and later uses
    // box b's id, block_size >= 8 keeping a chunk within 32 boxes; gathered
    // rows: up to 256 ids a chunk, read by the lanes that copy their rows),
    // so table reads overlap instead of following one another.
    const bool isk = warp == 4;                      // loads K (and q)
    const bool isv = !Cf::TWO_PROD || warp != 4;     // loads V
    const int tab_off = OFF_TAB + (isk ? 0 : TAB_SLOTS * TAB_W * 4);
    const uint32_t tab = sm.base_u32 + tab_off;
    const int* tab_s = reinterpret_cast<const int*>(sm.base + tab_off);
    auto fetch_ids = [&](const Walk& w, int slot) {
      const int nb = (w.valid() + p.box_tok - 1) >> p.log2_box;
      const int32_t* row = p.block_tables + (int64_t)w.seq * p.max_blocks;
      if constexpr (GATHER) {
        for (int e = lane; e < nb; e += 32)
          cp_async_4(tab + (slot * TAB_W + e) * 4, row + ((w.j * CH + e * p.box_tok) >> p.log2_bs));
      } else if (lane < nb) {
        cp_async_4(tab + (slot * TAB_W + lane) * 4,
                   row + ((w.j * CH + lane * p.box_tok) >> p.log2_bs));
      }
    };
    walk.init(lo, hi, seq_lo, seq_hi);
    Walk ahead = walk;
#pragma unroll 1  // one copy of cold code: its first run pays instruction-fetch misses
    for (int d = 0; d < TAB_AHEAD; ++d) {
      if (!ahead.done()) {
        fetch_ids(ahead, d);
        ahead.next();
      }
      cp_async_commit();
    }
    // Gathered rows (block_size < 8): the lanes copy 16-byte pieces and each
    // lane arrives on the chunk's FULL barrier once its own pieces have
    // landed and been made visible to the tensor cores (fence.proxy.async).
    // Commit groups per chunk i: rows(i), then ids(i + TAB_AHEAD); after
    // them, waiting until three groups remain pending completes rows(i - 1)
    // and ids(i + 1), so chunk i - 1 is published one chunk late.
    auto publish = [&](int l) {
      ptx::fence_proxy_async_smem();
      if (isk) ptx::mbar_arrive(sm.bar(B_FULL_K + l % NST));
      if (isv) ptx::mbar_arrive(sm.bar(B_FULL_V + l % NST));
    };
    int local = 0, seg = 0;
    for (; !walk.done(); walk.next(), ++local) {
      const int s = local % NST;
      const uint32_t ph = (local / NST) & 1;
      const int cs = walk.j * CH;
      const int valid = walk.valid();
      const int nbox = (valid + p.box_tok - 1) >> p.log2_box;
      if (!GATHER || local == 0) cp_async_wait<TAB_AHEAD - 1>();  // this chunk's ids have landed
      const int phys_in = lane < nbox ? tab_s[(local % TAB_SLOTS) * TAB_W + lane] : 0;
      if (!wait_bar(sm, sm.bar(B_EMPTY + s), ph ^ 1, p.err, 1)) break;
      if (!FP8 && isk && walk.first_of_segment()) {
        const int qs = seg & 1;
        const uint32_t qph = (seg >> 1) & 1;
        if (!wait_bar(sm, sm.bar(B_Q_EMPTY + qs), qph ^ 1, p.err, 2)) break;
        if (lane == 0) {
          // the unit's columns: heads g*gq .. g*gq+gq-1 of its ntok tokens
          // (3-D map [tokens, H, d], box {64, gq, ntok}; row c = j * gq + i)
          const uint32_t dst = sm.base_u32 + OFF_Q + qs * QTILE_B;
          ptx::mbar_arrive_expect_tx(sm.bar(B_Q_FULL + qs), (uint32_t)(2 * G * 128));
          ptx::tma_load_3d(dst, &tm_q, sm.bar(B_Q_FULL + qs), 0, walk.g * p.gq,
                           walk.seq * p.ntok);
          ptx::tma_load_3d(dst + QTILE_B / 2, &tm_q, sm.bar(B_Q_FULL + qs), 64, walk.g * p.gq,
                           walk.seq * p.ntok);
        }
        ++seg;
      }
      if (p.early_meta && local == 0) ptx::grid_dependency_wait();
      const uint32_t kdst = sm.base_u32 + OFF_K + s * TILE_B;
      const uint32_t vdst = sm.base_u32 + OFF_V + s * TILE_B;
      if constexpr (GATHER) {
        // Eight lanes per row, four rows per step: lane l copies 16-byte
        // piece l % 8 of row 4 * step + l / 8 (bf16: of both 128-byte column
        // blocks), so one instruction moves four whole 128-byte row pieces.
        // smem as the TMA boxes would leave it (128-byte rows, 16-byte pieces
        // XOR-swizzled by row & 7; bf16 column blocks HALF_B apart).
        const int* ids = tab_s + (local % TAB_SLOTS) * TAB_W;
        const int64_t row_bytes = (int64_t)Hkv * D * Cf::ELT;
        const int pc = lane & 7;
        const unsigned char* kg = p.kc + (int64_t)walk.g * D * Cf::ELT + pc * 16;
        const unsigned char* vg = p.vc + (int64_t)walk.g * D * Cf::ELT + pc * 16;
        const int steps = (valid + 3) >> 2;
#pragma unroll 4
        for (int st = 0; st < steps; ++st) {
          const int r = st * 4 + (lane >> 3);
          if (r < valid) {
            int phys = ids[r >> p.log2_bs];
            if ((unsigned)phys >= (unsigned)p.num_blocks) {
              atomicExch(p.err, 3);  // bad block id: load block 0 instead of faulting
              phys = 0;
            }
            const int64_t src =
                ((int64_t)phys * p.block_size + ((cs + r) & (p.block_size - 1))) * row_bytes;
            const uint32_t so = (uint32_t)(r * 128 + ((pc ^ (r & 7)) << 4));
            if (isk) {
              cp_async_16(kdst + so, kg + src, 16);
              if (!FP8) cp_async_16(kdst + HALF_B + so, kg + src + 128, 16);
            }
            if (isv) {
              cp_async_16(vdst + so, vg + src, 16);
              if (!FP8) cp_async_16(vdst + HALF_B + so, vg + src + 128, 16);
            }
          }
        }
        cp_async_commit();
      } else {
        const uint32_t bytes = (uint32_t)nbox * p.box_tok * (uint32_t)(D * Cf::ELT);
        const uint32_t row = (uint32_t)(lane * p.box_tok) * 128u;
        const int off = (cs + lane * p.box_tok) & (p.block_size - 1);
        int phys = phys_in;
        if (lane < nbox && (unsigned)phys >= (unsigned)p.num_blocks) {
          atomicExch(p.err, 3);  // bad block id: load block 0 instead of faulting
          phys = 0;
        }
        if (lane == 0) {
          if (isk) ptx::mbar_arrive_expect_tx(sm.bar(B_FULL_K + s), bytes);
          if (isv) ptx::mbar_arrive_expect_tx(sm.bar(B_FULL_V + s), bytes);
        }
        __syncwarp();
        if (lane < nbox) {
          // a token row of one head is 128 bytes in fp8 (one box) and 256 bytes
          // in bf16 (two 64-column boxes, one per 128-byte column block)
          if (isk) {
            ptx::tma_load_4d(kdst + row, &tm_k, sm.bar(B_FULL_K + s), 0, walk.g, off, phys);
            if (!FP8)
              ptx::tma_load_4d(kdst + HALF_B + row, &tm_k, sm.bar(B_FULL_K + s), 64, walk.g,
                               off, phys);
          }
          if (isv) {
            ptx::tma_load_4d(vdst + row, &tm_v, sm.bar(B_FULL_V + s), 0, walk.g, off, phys);
            if (!FP8)
              ptx::tma_load_4d(vdst + HALF_B + row, &tm_v, sm.bar(B_FULL_V + s), 64, walk.g,
                               off, phys);
          }
        }
      }
      if (!ahead.done()) {
        fetch_ids(ahead, (local + TAB_AHEAD) % TAB_SLOTS);
        ahead.next();
      }
      cp_async_commit();
      if (GATHER && local > 0) {
        cp_async_wait<3>();  // rows(local - 1) and ids(local + 1) have landed
        publish(local - 1);
      }
    }
    cp_async_wait<0>();
    if (GATHER && local > 0) publish(local - 1);
    // drain: the last loads issued must land before the CTA can exit
    // (gathered rows have landed already: every copy group is complete)
    __syncwarp();
    if (lane == 0) {
      if (!GATHER)
        for (int l = max(0, local - NST); l < local; ++l) {
          if (isk) drain_bar(sm.bar(B_FULL_K + l % NST), (l / NST) & 1);
          if (isv) drain_bar(sm.bar(B_FULL_V + l % NST), (l / NST) & 1);
        }
      if (!FP8 && isk)
        for (int sg = max(0, seg - 2); sg < seg; ++sg)
          drain_bar(sm.bar(B_Q_FULL + (sg & 1)), (sg >> 1) & 1);
    }
  } else if (warp == 5) {
    // ================= MMA issuer =================
    // Two cursors: the logits MMA of chunk nq (needs its K tile, a free S
    // buffer and, at a segment start, the q tile) and the PV MMA of chunk
    // npv < nq (needs P, a free O buffer and the V tile).  The thread polls
    // both and issues whichever is ready, so a stage is released as soon as
    // its own PV completes, never held back by a later chunk's K load.
    if (lane == 0) {
      constexpr uint32_t IDESC_QK =
          FP8 ? ptx::idesc_e4m3_f32(128, NQ_S, false) : ptx::idesc_bf16_f32(128, NQ_S, false);
      constexpr uint32_t IDESC_PV =
          FP8 ? ptx::idesc_e4m3_f32(128, NQ, true) : ptx::idesc_bf16_f32(128, NQ, true);
      walk.init(lo, hi, seq_lo, seq_hi);
      int nq = 0, npv = 0, seg = 0, cur_q = 0;
      long long t_idle = clock64();
      while (true) {
        bool progress = false;
        if (!walk.done()) {
          const int s = nq % NST;
          const int b = nq & 1;
          const bool first = walk.first_of_segment();
          bool ready = ptx::mbar_test_wait(sm.bar(B_FULL_K + s), (nq / NST) & 1) &&
                       ptx::mbar_test_wait(sm.bar(B_S_EMPTY + b), ((nq >> 1) & 1) ^ 1);
          if (ready && first) ready = ptx::mbar_test_wait(sm.bar(B_Q_FULL + (seg & 1)), (seg >> 1) & 1);
          if (ready) {
            if (first) cur_q = seg++ & 1;
            ptx::tc_fence_after();
            const uint32_t kbase = sm.base_u32 + OFF_K + s * TILE_B;
            const uint32_t qbase = sm.base_u32 + OFF_Q + cur_q * QTILE_B;
            if constexpr (FP8) {
              // K and q rows are 128 bytes (all of d); each MMA takes 32 of
              // them; one M = 128 MMA chain per 128-token half of the chunk
#pragma unroll
              for (int hf = 0; hf < NHALF; ++hf) {
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk) {
                  const uint64_t da = ptx::smem_desc_sw128(kbase + hf * HALF_B + kk * 32, 16, 1024);
                  const uint64_t db = ptx::smem_desc_sw128(qbase + kk * 32, 16, 1024);
                  ptx::tc_mma_f8(tmem + S_W * b + NQ_S * hf, da, db, IDESC_QK, kk > 0);
                }
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t da = ptx::smem_desc_sw128(kbase + (kk >> 2) * HALF_B + (kk & 3) * 32, 16, 1024);
                const uint64_t db = ptx::smem_desc_sw128(qbase + (kk >> 2) * (QTILE_B / 2) + (kk & 3) * 32, 16, 1024);
                ptx::tc_mma_f16(tmem + S_W * b, da, db, IDESC_QK, kk > 0);
              }
            }
            ptx::tc_commit(sm.bar(B_S_FULL + b));
            if (walk.last_of_segment()) ptx::tc_commit(sm.bar(B_Q_EMPTY + cur_q));
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
              // V MN-major: a 128-byte row is all of d for one token, so one
              // swizzle atom spans M; each MMA takes 32 tokens (4 atoms of 8).
              // P: one 16-row x 128-byte block per 128 tokens.
#pragma unroll
              for (int kk = 0; kk < CH / 32; ++kk) {
                const uint64_t da = ptx::smem_desc_sw128(vbase + kk * 4096, TILE_B, 1024);
                const uint64_t db = ptx::smem_desc_sw128(pbase + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024);
                ptx::tc_mma_f8(tmem + O_COL + 16 * b, da, db, IDESC_PV, kk > 0);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < CH / 16; ++kk) {
                const uint64_t da = ptx::smem_desc_sw128(vbase + kk * 2048, HALF_B, 1024);
                const uint64_t db = ptx::smem_desc_sw128(pbase + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024);
                ptx::tc_mma_f16(tmem + O_COL + 16 * b, da, db, IDESC_PV, kk > 0);
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
      // drain: every commit this thread issued must land before exit
      if (nq > 0) drain_bar(sm.bar(B_S_FULL + ((nq - 1) & 1)), ((nq - 1) >> 1) & 1);
      if (npv > 0) {
        const int L = npv - 1;
        drain_bar(sm.bar(B_EMPTY + L % NST), (L / NST) & 1);
        drain_bar(sm.bar(B_P_EMPTY + (L & 1)), (L >> 1) & 1);
      }
    }
  } else if (warp == 6) {
    // ================= merge warp =================
    // Follows the same walk; for each piece of a split unit (at most the
    // first and the last unit of this CTA's range) it waits for the softmax
    // warps' partial, counts the arrival, and if this was the unit's last
    // piece merges all pieces into the output: the merge latency stays off
    // the softmax warps' critical path.
    walk.init(lo, hi, seq_lo, seq_hi);
    int e = 0;
    for (; !walk.done(); walk.next()) {
      if (!walk.last_of_segment()) continue;
      const long long first = walk.k - walk.j;
      const long long lastc = first + walk.nch - 1;
      const int c0 = cta_of(first, Ktot, C);
      const int c1 = cta_of(lastc, Ktot, C);
      if (c0 == c1) continue;  // whole unit: the softmax warps wrote the output
      const bool good = wait_bar(sm, sm.bar(B_EPI + (e++ & 1)), 0, p.err, 14);
      if (!good) continue;
      const int u = walk.seq * Hkv + walk.g;
      const int nseg = c1 - c0 + 1;
      int last = 0;
      if (lane == 0) {
        ptx::fence_acq_rel_gpu();  // the partial the softmax warps wrote precedes the count
        last = (arrive(&p.counters[u], p.epoch) == nseg);
        if (last) ptx::fence_acq_rel_gpu();  // every other piece's partial is visible
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      __syncwarp();
      if (!last) continue;
      float M[G], Ls[G], a[G][4];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        M[h] = -INFINITY;
        Ls[h] = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) a[h][r] = 0.f;
      }
      for (int jj = 0; jj < nseg; ++jj) {
        const int64_t sj = (int64_t)(c0 + jj) * 2 + piece_slot(c0 + jj, lastc, Ktot, C);
        float2 ml[G];
        float ov[G][4];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          ml[h] = __ldcg(&p.ws_ml[sj * G + h]);
#pragma unroll
          for (int r = 0; r < 4; ++r) ov[h][r] = __ldcg(&p.ws_o[(sj * G + h) * D + lane + 32 * r]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float mn = fmaxf(M[h], ml[h].x);
          // a piece may hold no visible key for a column (multi-token units)
          const float msafe = mn == -INFINITY ? 0.f : mn;
          const float rs = fast_exp2(M[h] - msafe);  // 0 for the first piece
          const float w = fast_exp2(ml[h].x - msafe);
          Ls[h] = Ls[h] * rs + w * ml[h].y;
#pragma unroll
          for (int r = 0; r < 4; ++r) a[h][r] = a[h][r] * rs + w * ov[h][r];
          M[h] = mn;
        }
      }
      __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + lane;
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int r = 0; r < 4; ++r)
          o[out_row(walk.seq, walk.g, h) * D + 32 * r] =
              __float2bfloat16_rn(FP8 ? (a[h][r] * __ldg(p.v_scale)) / Ls[h] : a[h][r] / Ls[h]);
      if (p.lse && lane < G) {
#pragma unroll
        for (int h = 0; h < G; ++h)
          if (lane == h) p.lse[out_row(walk.seq, walk.g, h)] = M[h] + __log2f(Ls[h]) - (FP8 ? 8.f : 0.f);
      }
      if (lane == 0) p.counters[u] = p.epoch << 16;  // count 0: a replay starts afresh
    }
  } else if (warp == 7) {
    // ================= q warp (fp8 cache only) =================
    // Per segment, the group's G query rows (bf16, read from global memory)
    // become three e4m3 parts: q * 2^e ~= hi + mid + lo, with 2^e the power
    // of two that puts max |q| in [128, 256); each part is the round-to-
    // nearest of what the previous ones leave (exact fp32 residuals), so the
    // sum holds q to ~2^-12 relative.  The parts fill operand rows h, 8 + h
    // and 16 + h; logits columns h + 8 + 16 add up to 2^e q_h . k.
    if constexpr (FP8) {
      float* qexp = reinterpret_cast<float*>(sm.base + OFF_QEXP);
      constexpr int NPIECE = G * D / 8;            // 16-byte pieces of bf16 q
      constexpr int NV = (NPIECE + 31) / 32;       // per lane
      walk.init(lo, hi, seq_lo, seq_hi);
      int seg = 0;
      for (; !walk.done(); walk.next()) {
        if (!walk.first_of_segment()) continue;
        const int qs = seg & 1;
        if (!wait_bar(sm, sm.bar(B_Q_EMPTY + qs), ((seg >> 1) & 1) ^ 1, p.err, 2)) break;
        ++seg;
        const uint4* src = reinterpret_cast<const uint4*>(p.q);
        uint4 v[NV];
        uint32_t amax = 0;  // bit pattern of max |q| (orders like the float)
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const int idx = i * 32 + lane;
          const int col = idx >> 4;  // column: head g*gq + (col & (gq-1)) of token col / gq
          const int64_t row = ((int64_t)walk.seq * p.ntok + (col >> p.log2_gq)) * H +
                              (int64_t)walk.g * p.gq + (col & (p.gq - 1));
          v[i] = idx < NPIECE ? __ldg(src + row * (D / 8) + (idx & 15)) : make_uint4(0, 0, 0, 0);
          const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
          for (int c = 0; c < 4; ++c)
            amax = max(amax, max((w[c] << 16) & 0x7fffffffu, w[c] & 0x7fff0000u));
        }
        amax = __reduce_max_sync(0xffffffffu, amax);
        const int eb = (int)(amax >> 23);        // biased exponent; 0 for zero / subnormal
        int e = eb == 0 ? 0 : 134 - eb;         // max |q| * 2^e in [128, 256)
        e = max(-126, min(126, e));
        const float mul = __int_as_float((127 + e) << 23);
        if (lane == 0) qexp[qs] = __int_as_float((127 - e) << 23);
        unsigned char* qt = sm.base + OFF_Q + qs * QTILE_B;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const int idx = i * 32 + lane;
          if (idx < NPIECE) {
            const int h = idx >> 4, d0 = (idx & 15) * 8;
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            uint32_t pw[3][2] = {{0, 0}, {0, 0}, {0, 0}};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              float a = bf16_lo(w[c]) * mul, b = bf16_hi(w[c]) * mul;
#pragma unroll
              for (int part = 0; part < 3; ++part) {
                const uint16_t code = pack_e4m3x2_rn(a, b);
                const float2 v2 = e4m3x2_to_float2(code);
                a -= v2.x;
                b -= v2.y;
                pw[part][c >> 1] |= (uint32_t)code << (16 * (c & 1));
              }
            }
            // 128-byte swizzle: 16-byte piece index XOR (row & 7); row 8j + h
            // sits in the j-th 1024-byte group with (row & 7) = h
            const int o = h * 128 + ((((d0 >> 4) ^ h) << 4) | (d0 & 8));
#pragma unroll
            for (int part = 0; part < 3; ++part)
              *reinterpret_cast<uint2*>(qt + part * 1024 + o) = make_uint2(pw[part][0], pw[part][1]);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(sm.bar(B_Q_FULL + qs));
      }
    }
  } else {
    // ================= softmax + epilogue (warps 0-3) =================
    const int t = tid;  // TMEM lane: token in S, d in O
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float* red = reinterpret_cast<float*>(sm.base + OFF_RED);
    float* lred = reinterpret_cast<float*>(sm.base + OFF_LRED);
    // fp8: logits are (S_h + S_{8+h}) * 2^-e * k_scale * scale * log2(e),
    // with 2^-e the q tile's prescale; p is carried as 256 p (see below)
    const float ksc = FP8 ? __ldg(p.k_scale) : 1.f;
    const float vsc = FP8 ? __ldg(p.v_scale) : 1.f;
    const float* qexp = reinterpret_cast<const float*>(sm.base + OFF_QEXP);
    float sscale = p.scale_log2;
    int qseg = 0;
    float m[G], l[G], acc[G], alpha_prev[G], dm[G], dl[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
      acc[h] = 0.f;
      alpha_prev[h] = 0.f;
      dm[h] = -INFINITY;
      dl[h] = 0.f;
    }
    // what the O side needs to know about the chunk it lags behind
    struct Info {
      int seq, g, nch, j;
      long long k;
      bool last;
    } prev{0, 0, 0, 0, 0, false};

    int split_epi = 0;  // split-unit partials handed to the merge warp (<= 2)
    auto epilogue = [&](const Info& in, const float* ms, const float* ls) {
      float lt[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float v = ls[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) lred[warp * 16 + h] = v;
      }
      ptx::bar_sync_named(2, 128);
#pragma unroll
      for (int h = 0; h < G; ++h) lt[h] = lred[h] + lred[16 + h] + lred[32 + h] + lred[48 + h];
      ptx::bar_sync_named(2, 128);
      const long long first = in.k - in.j;            // unit's first chunk (global)
      const long long last = first + in.nch - 1;       // unit's last chunk
      const int c0 = cta_of(first, Ktot, C);
      const int c1 = cta_of(last, Ktot, C);
      const int u = in.seq * Hkv + in.g;
      __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + t;
      if (c0 == c1) {
#pragma unroll
        for (int h = 0; h < G; ++h)
          o[out_row(in.seq, in.g, h) * D] =
              __float2bfloat16_rn(FP8 ? (acc[h] * vsc) / lt[h] : acc[h] / lt[h]);
        if (p.lse) {
          // log2 of the softmax denominator (e4m3: l carries a factor 256)
#pragma unroll
          for (int h = 0; h < G; ++h)
            if (t == h) p.lse[out_row(in.seq, in.g, h)] = ms[h] + __log2f(lt[h]) - (FP8 ? 8.f : 0.f);
        }
      } else {
        // a piece of a split unit: leave the partial for the merge warp
        const int64_t slot = (int64_t)blockIdx.x * 2 + piece_slot(blockIdx.x, last, Ktot, C);
#pragma unroll
        for (int h = 0; h < G; ++h) p.ws_o[(slot * G + h) * D + t] = acc[h];
#pragma unroll
        for (int h = 0; h < G; ++h)
          if (t == h) p.ws_ml[slot * G + h] = make_float2(ms[h], lt[h]);
        ptx::mbar_arrive(sm.bar(B_EPI + (split_epi++ & 1)));
      }
    };

    auto acc_o = [&](int L, const Info& in, bool use_done) {
      const int b = L & 1;
      const uint32_t bph = (L >> 1) & 1;
      float ov[FP8 || G > 8 ? 16 : 8];
      const bool good = wait_bar(sm, sm.bar(B_O_FULL + b), bph, p.err, 10);
      ptx::tc_fence_after();
      if constexpr (FP8) {
        ptx::tmem_ld_x16(tmem + lane_base + O_COL + 16 * b, ov);
      } else {
        if constexpr (G > 8) {
          ptx::tmem_ld_x16(tmem + lane_base + O_COL + 16 * b, ov);
        } else {
          ptx::tmem_ld_x8(tmem + lane_base + O_COL + 16 * b, ov);
        }
      }
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(sm.bar(B_O_EMPTY + b));
      if (!good) {
#pragma unroll
        for (int h = 0; h < G; ++h) ov[h] = 0.f;
      }
      if constexpr (FP8) {
#pragma unroll
        for (int h = 0; h < G; ++h) ov[h] += ov[8 + h];  // hi and lo parts of P
      }
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = acc[h] * alpha_prev[h] + ov[h];
      if (in.last) {
        if (use_done) epilogue(in, dm, dl);
        else epilogue(in, m, l);
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] = 0.f;
      }
    };

    walk.init(lo, hi, seq_lo, seq_hi);
    int local = 0;
    for (; !walk.done(); walk.next(), ++local) {
      const int s = local % NST;
      const uint32_t ph = (local / NST) & 1;
      const int b = local & 1;
      const uint32_t bph = (local >> 1) & 1;
      // ---- logits of this chunk ----
      // fp8: thread t holds tokens t and 128 + t (halves 0 and 1); per half
      // the three q parts of head h are columns h, 8 + h, 16 + h
      float sv[FP8 ? 24 : (G > 8 ? 16 : 8)], sv1[FP8 ? 24 : 1];
      bool good = wait_bar(sm, sm.bar(B_S_FULL + b), bph, p.err, 11);
      ptx::tc_fence_after();
      if constexpr (FP8) {
        float a16[16], a8[8], b16[16], b8[8];
        ptx::tmem_ld_x16(tmem + lane_base + S_W * b, a16);
        ptx::tmem_ld_x8(tmem + lane_base + S_W * b + 16, a8);
        ptx::tmem_ld_x16(tmem + lane_base + S_W * b + NQ_S, b16);
        ptx::tmem_ld_x8(tmem + lane_base + S_W * b + NQ_S + 16, b8);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          sv[i] = a16[i];
          sv1[i] = b16[i];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          sv[16 + i] = a8[i];
          sv1[16 + i] = b8[i];
        }
      } else {
        if constexpr (G > 8) {
          ptx::tmem_ld_x16(tmem + lane_base + S_W * b, sv);
        } else {
          ptx::tmem_ld_x8(tmem + lane_base + S_W * b, sv);
        }
      }
      ptx::tmem_ld_wait();
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
#pragma unroll
        for (int h = 0; h < G; ++h) {
          sv[h] += sv[8 + h] + sv[16 + h];  // the parts of q
          sv1[h] += sv1[8 + h] + sv1[16 + h];
        }
      }
      const int valid = walk.valid();
      // causal limit: column h (token h / gq of the unit's ntok) sees keys at
      // positions < n - ntok + h / gq + 1, i.e. chunk rows t < tlim0 + h / gq
      // (with ntok = 1 that is t < valid)
      const int tlim0 = walk.n - (p.causal ? p.ntok - 1 : 0) - walk.j * CH;
      float x[G], x1[G];  // x1: the token of half 1 (fp8 only)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const int tl = tlim0 + (p.causal ? (h >> p.log2_gq) : 0);
        x[h] = (good && t < tl) ? sv[h] * sscale : -INFINITY;
        x1[h] = (FP8 && good && 128 + t < tl) ? sv1[FP8 ? h : 0] * sscale : -INFINITY;
      }
      // ---- chunk max per head over the 128 lanes ----
      float* rb = red + b * 64;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float v = ptx::warp_max_f32(FP8 ? fmaxf(x[h], x1[h]) : x[h]);
        if (lane == 0) rb[warp * 16 + h] = v;
      }
      ptx::bar_sync_named(1, 128);
      if (walk.first_of_segment()) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          dm[h] = m[h];
          dl[h] = l[h];
          m[h] = -INFINITY;
          l[h] = 0.f;
        }
      }
      float alpha[G];
      __nv_bfloat16 pb[G];   // bf16: p rounded for the MMA
      uint8_t p_hi[NHALF][G], p_lo[NHALF][G];  // fp8: 256 p ~= hi + lo, two e4m3 codes
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float cmax = fmaxf(fmaxf(rb[h], rb[16 + h]), fmaxf(rb[32 + h], rb[48 + h]));
        const float m_new = fmaxf(m[h], cmax);
        // a column may have seen no visible key yet (multi-token units)
        const float msafe = m_new == -INFINITY ? 0.f : m_new;
        alpha[h] = fast_exp2(m[h] - msafe);
        m[h] = m_new;
        const float pv = fast_exp2(x[h] - msafe);  // 0 for masked keys (x = -inf)
        if constexpr (FP8) {
          // 256 p in [0, 256] keeps e4m3's range; l carries the same factor,
          // so it cancels in acc / l.  The residual is exact (Sterbenz).
          const float pv1 = fast_exp2(x1[h] - msafe);
          const float ps0 = pv * 256.f, ps1 = pv1 * 256.f;
          const uint16_t ch = pack_e4m3x2_rn(ps0, ps1);
          const float2 hv = e4m3x2_to_float2(ch);
          const uint16_t cl = pack_e4m3x2_rn(ps0 - hv.x, ps1 - hv.y);
          const float2 lv = e4m3x2_to_float2(cl);
          p_hi[0][h] = (uint8_t)(ch & 0xff);
          p_hi[NHALF - 1][h] = (uint8_t)(ch >> 8);
          p_lo[0][h] = (uint8_t)(cl & 0xff);
          p_lo[NHALF - 1][h] = (uint8_t)(cl >> 8);
          l[h] = l[h] * alpha[h] + ((hv.x + lv.x) + (hv.y + lv.y));
        } else {
          pb[h] = __float2bfloat16_rn(pv);
          l[h] = l[h] * alpha[h] + __bfloat162float(pb[h]);
        }
      }
      // ---- P tile (and the V tail) for the PV MMA ----
      wait_bar(sm, sm.bar(B_P_EMPTY + b), bph ^ 1, p.err, 12);
      if (valid < CH) {
        wait_bar(sm, sm.bar(B_FULL_V + s), ph, p.err, 13);
#pragma unroll
        for (int hf = 0; hf < NHALF; ++hf) {
          // V row of token hf * 128 + t: 128 bytes (fp8) or two 128-byte
          // pieces HALF_B apart (bf16)
          if (hf * 128 + t >= valid) {
            unsigned char* vrow = sm.base + OFF_V + s * TILE_B + (hf * 128 + t) * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const int cc = (c + t) & 7;
              *reinterpret_cast<uint4*>(vrow + cc * 16) = make_uint4(0, 0, 0, 0);
              if (!FP8) *reinterpret_cast<uint4*>(vrow + HALF_B + cc * 16) = make_uint4(0, 0, 0, 0);
            }
          }
        }
      }
      if constexpr (FP8) {
        // rows h (hi) and 8 + h (lo) of the 16 x 128-token tile: one 128-byte
        // swizzled row per head, token t at byte t
        // (one 2 KiB block of 16 rows per 128-token half)
        unsigned char* pt = sm.base + OFF_P + b * PTILE_B;
        const int chunk = t >> 4;
        const int byte = t & 15;
#pragma unroll
        for (int hf = 0; hf < NHALF; ++hf)
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const int o = hf * 2048 + (h & 7) * 128 + (((chunk ^ (h & 7)) << 4) | byte);
            pt[o] = p_hi[hf][h];
            pt[1024 + o] = p_lo[hf][h];
          }
      } else {
        unsigned char* pt = sm.base + OFF_P + b * PTILE_B + (t >> 6) * 2048;
        const int chunk = (t & 63) >> 3;
        const int byte = (t & 7) * 2;
#pragma unroll
        for (int h = 0; h < G; ++h)
          *reinterpret_cast<__nv_bfloat16*>(pt + h * 128 + ((chunk ^ (h & 7)) << 4) + byte) = pb[h];
      }
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(sm.bar(B_P_FULL + b));
      // ---- fold the previous chunk's PV result ----
      if (local > 0) acc_o(local - 1, prev, walk.first_of_segment());
#pragma unroll
      for (int h = 0; h < G; ++h) alpha_prev[h] = alpha[h];
      prev = Info{walk.seq, walk.g, walk.nch, walk.j, walk.k, walk.last_of_segment()};
    }
    if (local > 0) acc_o(local - 1, prev, false);
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

unsigned long long next_call_epoch() {
  static std::atomic<unsigned long long> next_epoch{0x5eed00000000ull};
  return next_epoch.fetch_add(1, std::memory_order_relaxed) & 0xFFFFFFFFFFFFull;
}

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

template <int G, bool FP8, bool GATHER>
cudaError_t launch_g3(const Params& prm, const CUtensorMap& mk, const CUtensorMap& mv,
                      const CUtensorMap& mq, cudaStream_t stream) {
  using Cf = Cfg<FP8, GATHER>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<G, FP8, GATHER>,
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_tc_kernel<G, FP8, GATHER>, mk, mv, mq, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// block_size < 8: the instantiation that gathers rows by cp.async
template <int G, bool FP8>
cudaError_t launch_g(const TcLaunch& a, const Params& prm, const CUtensorMap& mk,
                     const CUtensorMap& mv, const CUtensorMap& mq, cudaStream_t stream) {
  return a.block_size < 8 ? launch_g3<G, FP8, true>(prm, mk, mv, mq, stream)
                          : launch_g3<G, FP8, false>(prm, mk, mv, mq, stream);
}

}  // namespace tc

size_t tc_workspace_bytes(int64_t num_seqs, int64_t num_heads, int64_t /*max_ctx*/,
                          int num_ctas, int tokens_per_seq) {
  // partials live in two slots per CTA of up to kMaxCols columns, whatever
  // the context lengths
  const int64_t rows = num_seqs * (tokens_per_seq > 0 ? tokens_per_seq : 1) * num_heads;  // >= units
  const int64_t slots = (int64_t)num_ctas * 2 * tc::kMaxCols;
  size_t off = 256;                                             // error word
  off += ((size_t)rows * 8 + 255) / 256 * 256;                  // merge counters
  off += ((size_t)slots * 8 + 255) / 256 * 256;                 // (m, l)
  off += (size_t)slots * tc::D * 4;                             // partial o
  return off;
}

bool tc_supported(int head_dim, int group, bool fp8, int num_seqs, int block_size,
                  int tokens_per_seq) {
  // Every power-of-two block size: from 8 tokens up the K/V rows arrive as
  // TMA boxes (whole 1024-byte swizzle atoms), below 8 as gathered 16-byte
  // copies.  A unit's columns (group x tokens) fill the MMA N: up to 16 for
  // bf16, 8 for e4m3 (its q takes three rows per column).
  const int t = tokens_per_seq > 0 ? tokens_per_seq : 1;
  const int cols = group * t;
  const bool pow2 = group > 0 && (group & (group - 1)) == 0 && (cols & (cols - 1)) == 0;
  return head_dim == tc::D && pow2 && group <= 8 && cols <= (fp8 ? 8 : 16) &&
         num_seqs <= tc::kMaxSeqs && block_size >= 1 &&
         (block_size & (block_size - 1)) == 0 && tc::encode_fn() != nullptr;
}

cudaError_t launch_decode_tc(const TcLaunch& a, cudaStream_t stream) {
  using namespace tc;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int box_tok = a.block_size < 128 ? a.block_size : 128;  // tokens per TMA box
  CUtensorMap mk, mv, mq;
  {
    // [blocks, block_size, H_kv, d] with d innermost; a box is one 128-byte
    // column block (64 bf16 or all 128 e4m3 of d) of box_tok tokens
    const cuuint64_t elt = a.fp8 ? 1 : 2;
    const CUtensorMapDataType dt =
        a.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)a.num_kv_heads, (cuuint64_t)a.block_size,
                          (cuuint64_t)a.num_blocks};
    cuuint64_t strides[3] = {(cuuint64_t)D * elt, (cuuint64_t)a.num_kv_heads * D * elt,
                             (cuuint64_t)a.block_size * a.num_kv_heads * D * elt};
    cuuint32_t box[4] = {(cuuint32_t)(128 / elt), 1, (cuuint32_t)box_tok, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    // L2 fills of the row's own size: a 256-byte promotion of a 128-byte e4m3
    // row also pulls the next KV head's row, read (often from DRAM again) by
    // another CTA -- measured at 35 % extra DRAM reads
    const CUtensorMapL2promotion promo =
        a.fp8 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
    if (enc(&mk, dt, 4, const_cast<void*>(a.k_cache), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (enc(&mv, dt, 4, const_cast<void*>(a.v_cache), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int ntok = a.tokens_per_seq > 0 ? a.tokens_per_seq : 1;
  const int gq = a.num_heads / a.num_kv_heads;
  {
    // q as [tokens, H, d]; a unit's box is {64 of d, its gq heads, its ntok tokens}
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.num_heads,
                          (cuuint64_t)a.num_seqs * ntok};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.num_heads * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)gq, (cuuint32_t)ntok};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  Params prm{};
  prm.out = a.out;
  prm.q = a.q;
  prm.k_scale = a.k_scale;
  prm.v_scale = a.v_scale;
  prm.block_tables = a.block_tables;
  prm.context_lens = a.context_lens;
  char* ws = static_cast<char*>(a.workspace);
  const int64_t rows = (int64_t)a.num_seqs * ntok * a.num_heads;
  prm.num_ctas = a.num_ctas;
  size_t off = 0;
  prm.err = reinterpret_cast<int*>(ws + off);
  off += 256;
  prm.counters = reinterpret_cast<unsigned long long*>(ws + off);
  off += ((size_t)rows * 8 + 255) / 256 * 256;
  prm.ws_ml = reinterpret_cast<float2*>(ws + off);
  off += ((size_t)a.num_ctas * 2 * kMaxCols * 8 + 255) / 256 * 256;
  prm.ws_o = reinterpret_cast<float*>(ws + off);
  prm.num_seqs = a.num_seqs;
  prm.num_heads = a.num_heads;
  prm.gq = gq;
  prm.ntok = ntok;
  prm.causal = a.non_causal ? 0 : 1;
  prm.lse = a.lse;
  {
    int lg = 0;
    while ((1 << lg) < gq) ++lg;
    prm.log2_gq = lg;
  }
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
  prm.early_meta = a.early_meta ? 1 : 0;
  prm.epoch = next_call_epoch();
  prm.kc = static_cast<const unsigned char*>(a.k_cache);
  prm.vc = static_cast<const unsigned char*>(a.v_cache);
  const int G = gq * ntok;  // columns of a unit
  if (a.fp8) {
    switch (G) {
      case 1: return launch_g<1, true>(a, prm, mk, mv, mq, stream);
      case 2: return launch_g<2, true>(a, prm, mk, mv, mq, stream);
      case 4: return launch_g<4, true>(a, prm, mk, mv, mq, stream);
      case 8: return launch_g<8, true>(a, prm, mk, mv, mq, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (G) {
    case 1: return launch_g<1, false>(a, prm, mk, mv, mq, stream);
    case 2: return launch_g<2, false>(a, prm, mk, mv, mq, stream);
    case 4: return launch_g<4, false>(a, prm, mk, mv, mq, stream);
    case 8: return launch_g<8, false>(a, prm, mk, mv, mq, stream);
    case 16: return launch_g<16, false>(a, prm, mk, mv, mq, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
