// Paged decode attention on the 5th-generation tensor cores (tcgen05) with
// TMA-staged operands, for a bf16 cache with head_dim 128.
//
// Same mathematics as the SIMT kernel ("4.6 PagedAttention & KV-Cache Memory
// Management", section "The PagedAttention Kernel": block-table gather, GQA
// head map h -> h / G, online softmax; section "Performance considerations":
// split the sequence across CTAs and merge), organised for Blackwell:
//
// Work split.  The KV of every (sequence, KV head) unit is cut into 128-token
// chunks; all chunks of all units are numbered in (sequence, head, chunk)
// order and each persistent CTA (one per SM) takes an equal contiguous range
// of that numbering.  A unit whose chunks all fall in one CTA is finished
// there; otherwise each CTA writes an unnormalised partial (m, l, o) for its
// piece ("segment"), and the last of the unit's CTAs to finish merges the
// partials.  The arrival count of a unit is a 64-bit word tagged with a
// per-call epoch (48 bits) supplied by the host: a word whose tag is not the
// current epoch counts as zero, so the workspace needs no initialisation and
// may be shared by calls of different shapes; the merging CTA leaves the
// word at (epoch, 0), so replaying the same launch also starts from zero.
// Load balance is one chunk, whatever the mix of context lengths.
//
// Warp roles (224 threads):
//   warps 0-3  softmax + epilogue: thread t owns TMEM lane t (a token of the
//              logits tile, a d-element of the output tile);
//   warp 4     producer: per chunk, TMA tensor loads of each physical block's
//              K and V rows (4-D tensor map [blocks, block_size, H_kv, d],
//              128-byte swizzle, two 64-column halves) into a 3-stage ring,
//              and per segment a TMA load of the group's query rows;
//   warp 5     TMEM allocation and the single MMA-issuing thread;
//   warp 6     merge warp: counts finished pieces of split units and merges
//              a unit's pieces when its last piece is done.
//
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

namespace pa {
namespace tc {

constexpr int D = 128;
constexpr int CH = 128;                // tokens per chunk
constexpr int NST = 3;                 // K/V ring stages
constexpr int NQ = 16;                 // padded query heads (MMA N)
constexpr int TILE_B = CH * D * 2;     // 32 KiB: one K or V chunk
constexpr int HALF_B = CH * 128;       // 16 KiB: one 64-column half of a tile
constexpr int QTILE_B = NQ * D * 2;    // 4 KiB
constexpr int PTILE_B = NQ * CH * 2;   // 4 KiB
constexpr int NTHREADS = 224;
constexpr int TMEM_COLS = 64;          // S[2] x 16 + O[2] x 16 columns

constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + NST * TILE_B;
constexpr int OFF_Q = OFF_V + NST * TILE_B;
constexpr int OFF_P = OFF_Q + 2 * QTILE_B;
constexpr int OFF_BAR = OFF_P + 2 * PTILE_B;
// barrier indices
constexpr int B_FULL_K = 0, B_FULL_V = 3, B_EMPTY = 6, B_S_FULL = 9, B_S_EMPTY = 11,
              B_P_FULL = 13, B_P_EMPTY = 15, B_O_FULL = 17, B_O_EMPTY = 19, B_Q_FULL = 21,
              B_Q_EMPTY = 23, B_EPI = 25, NBARS = 27;
constexpr int OFF_TMEM = OFF_BAR + NBARS * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int OFF_SQ = OFF_ABORT + 4;        // [2] ints: sequences of the range's ends
constexpr int OFF_RED = OFF_ABORT + 12;      // [2][4][8] floats, chunk max
constexpr int OFF_LRED = OFF_RED + 2 * 4 * 8 * 4;  // [4][8] floats, epilogue sums
constexpr int OFF_CP = OFF_LRED + 4 * 8 * 4;       // chunk prefix per sequence, [S+1] int
constexpr int kMaxSeqs = 1024;
constexpr int OFF_NLEN = OFF_CP + (kMaxSeqs + 1) * 4;  // clamped context length per sequence
constexpr int OFF_TAB = OFF_NLEN + kMaxSeqs * 4;  // block-id ring: 4 chunks x 16 boxes
constexpr int TAB_SLOTS = 4, TAB_AHEAD = 3;
constexpr int SMEM_BYTES = OFF_TAB + TAB_SLOTS * 16 * 4 + 1024;  // + alignment slack

constexpr long long kWaitClocks = 1LL << 31;

struct Params {
  void* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int* err;        // workspace word 0: nonzero if a wait expired / bad id
  unsigned long long* counters;  // [units] (epoch << 16) | arrivals of finished segments
  float2* ws_ml;   // [units * max_seg * G]
  float* ws_o;     // [units * max_seg * G * D]
  int num_seqs, num_heads, num_kv_heads, max_blocks, num_blocks, block_size, log2_bs;
  int num_ctas, max_seg, box_tok, log2_box;
  float scale_log2;
  unsigned long long epoch;  // 48-bit tag of this call
  int early_meta;            // previous kernel wrote only the cache
};

struct Smem {
  unsigned char* base;
  uint32_t base_u32;
  __device__ uint32_t bar(int i) const { return base_u32 + OFF_BAR + 8 * i; }
  __device__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(base + OFF_ABORT); }
};

__device__ __forceinline__ bool wait_bar(const Smem& sm, uint32_t bar, uint32_t parity,
                                         int* err, int code) {
  if (*sm.abort_flag()) return false;
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (*sm.abort_flag()) return false;
    if (clock64() - t0 > kWaitClocks) {
      *sm.abort_flag() = 1;
      atomicExch(err, code);
      return false;
    }
  }
  return true;
}

// Drain wait used while shutting down: bounded, ignores the abort flag.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > (kWaitClocks >> 2)) return;
  }
}

// Count one finished segment of a unit; returns the count including this one.
// A word tagged with another epoch (an earlier call, or stale bytes) counts as
// zero.  Lock-free: a failed exchange means another CTA's exchange succeeded.
__device__ __forceinline__ int arrive(unsigned long long* cnt, unsigned long long epoch) {
  unsigned long long v = *reinterpret_cast<volatile unsigned long long*>(cnt);
  while (true) {
    const unsigned long long nv = ((v >> 16) == epoch) ? v + 1 : ((epoch << 16) | 1ull);
    const unsigned long long old = atomicCAS(cnt, v, nv);
    if (old == v) return (int)(nv & 0xFFFFull);
    v = old;
  }
}

// First chunk index owned by CTA c when K chunks are split over C CTAs.
__device__ __forceinline__ long long range_lo(long long c, long long K, long long C) {
  return c * K / C;
}
// CTA owning chunk k.
__device__ __forceinline__ int cta_of(long long k, long long K, int C) {
  int c = (int)(k * C / K);
  while (c + 1 < C && range_lo(c + 1, K, C) <= k) ++c;
  while (c > 0 && range_lo(c, K, C) > k) --c;
  return c;
}

// Walks this CTA's chunk range; identical in every role.  The range is
// visited as up to three contiguous pieces: the unit it ends in (shared with
// the next CTA), then the unit it starts in (shared with the previous CTA),
// then the whole units in between.  Both pieces of every split unit are thus
// finished early in their CTAs, so the merge of a split unit happens while
// the pipeline still has work to hide it, and every CTA ends on whole units.
struct ChunkWalk {
  const int* cp;   // smem chunk prefix: cp[i] = chunks of sequences < i (all heads)
  const int* nl;   // smem clamped context lengths
  int S, Hkv;
  long long k;                 // current global chunk index
  long long lo0, hi0, lo1, hi1, lo2, hi2;  // the pieces, in visiting order
  long long cur_lo, cur_hi;    // the piece being visited
  int nsub, si;
  int seq, g, j, nch, n;

  int sq1, g1, j1, sq2, g2;    // where pieces 1 and 2 start (piece 2 starts a unit)

  __device__ void load_unit() {
    nch = (cp[seq + 1] - cp[seq]) / Hkv;
    n = nl[seq];
  }
  // position (seq, g, j) of chunk kk, given the sequence s holding it
  __device__ void seek_in(int s, long long kk) {
    k = kk;
    seq = s;
    load_unit();
    const int r = (int)(kk - cp[s]);
    g = r / nch;
    j = r - g * nch;
  }
  // seq_lo / seq_hi: the sequences holding chunks lo and hi - 1
  __device__ void init(long long lo, long long hi, int seq_lo, int seq_hi) {
    nsub = 0;
    si = 0;
    if (lo >= hi) {
      k = 0;
      return;
    }
    seek_in(seq_lo, lo);
    const long long head_hi = min(hi, k - j + nch);  // end of the first unit
    if (head_hi >= hi) {
      lo0 = lo; hi0 = hi; nsub = 1;
      cur_lo = lo0;
      cur_hi = hi0;
      return;
    }
    sq1 = seq; g1 = g; j1 = j;
    // the unit after the first one (a chunk exists there: head_hi < hi)
    sq2 = seq;
    g2 = g + 1;
    if (g2 == Hkv) {
      g2 = 0;
      do { ++sq2; } while (cp[sq2 + 1] == cp[sq2]);
    }
    seek_in(seq_hi, hi - 1);
    const long long tail_lo = k - j;  // first chunk of the last unit (>= head_hi)
    lo0 = tail_lo; hi0 = hi;
    lo1 = lo; hi1 = head_hi;
    lo2 = hi2 = 0;
    nsub = 2;
    if (head_hi < tail_lo) {
      lo2 = head_hi; hi2 = tail_lo;
      nsub = 3;
    }
    cur_lo = lo0;
    cur_hi = hi0;
    k = tail_lo;
    j = 0;
  }
  __device__ bool done() const { return si >= nsub; }
  __device__ void next() {
    if (++k >= cur_hi) {
      if (++si < nsub) {
        if (si == 1) {
          cur_lo = lo1; cur_hi = hi1;
          seq = sq1; g = g1; j = j1;
        } else {
          cur_lo = lo2; cur_hi = hi2;
          seq = sq2; g = g2; j = 0;
        }
        k = cur_lo;
        load_unit();
      }
      return;
    }
    if (++j == nch) {
      j = 0;
      if (++g == Hkv) {
        g = 0;
        do { ++seq; } while (cp[seq + 1] == cp[seq]);
        load_unit();
      }
    }
  }
  __device__ bool first_of_segment() const { return j == 0 || k == cur_lo; }
  __device__ bool last_of_segment() const { return j == nch - 1 || k == cur_hi - 1; }
  __device__ int valid() const { return min(CH, n - j * CH); }
};

template <int G>
__global__ void __launch_bounds__(NTHREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_q, const Params p) {
  extern __shared__ unsigned char smem_raw[];
  Smem sm;
  {
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t aligned = (raw + 1023u) & ~1023u;
    sm.base = smem_raw + (aligned - raw);
    sm.base_u32 = aligned;
  }
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = p.num_seqs, Hkv = p.num_kv_heads, H = p.num_heads;
  const int cap = p.max_blocks << p.log2_bs;
  int* cp = reinterpret_cast<int*>(sm.base + OFF_CP);
  int* nl = reinterpret_cast<int*>(sm.base + OFF_NLEN);

  // ---------------- prologue ----------------
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
      ptx::mbar_init(sm.bar(i), cnt);
    }
    *sm.abort_flag() = 0;
    ptx::fence_mbar_init();
  }
  // Inputs may come from the previous kernel in the stream.  When that kernel
  // is known to write only the KV cache, only the producer waits, right
  // before its first cache load; lengths, tables and q are read at once.
  if (!p.early_meta) ptx::grid_dependency_wait();
  if (warp == 4 && lane == 0) {
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    ptx::prefetch_tmap(&tm_q);
  }
  if (warp < 4) {
    // zero both P tiles (rows >= G stay zero for the whole kernel)
    uint4* pz = reinterpret_cast<uint4*>(sm.base + OFF_P);
    for (int i = tid; i < 2 * PTILE_B / 16; i += 128) pz[i] = make_uint4(0, 0, 0, 0);
    ptx::fence_proxy_async_smem();
    // empty sequences get zero rows (spread over the CTAs)
    for (int i = blockIdx.x; i < S; i += gridDim.x) {
      if (min(p.context_lens[i], cap) <= 0) {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + (int64_t)i * H * D;
        for (int e = tid; e < H * D; e += 128) o[e] = __float2bfloat16_rn(0.f);
      }
    }
  }
  // chunk counts per sequence, loaded by all threads at once
  for (int i = tid; i < S; i += NTHREADS) {
    const int n = min(p.context_lens[i], cap);
    nl[i] = n;
    cp[i] = n > 0 ? Hkv * ((n + CH - 1) / CH) : 0;
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive prefix in place: cp[i] = sum_{i' < i} H_kv * ceil(n_i' / CH)
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
  const long long Ktot = cp[S];
  // only min(CTAs, chunks) CTAs take work, so every working CTA owns at least
  // one chunk and a unit never spans more CTAs than it has chunks
  const int C = (int)(Ktot < p.num_ctas ? Ktot : p.num_ctas);
  const long long lo = (int)blockIdx.x < C ? range_lo(blockIdx.x, Ktot, C) : 0;
  const long long hi = (int)blockIdx.x < C ? range_lo(blockIdx.x + 1, Ktot, C) : 0;
  // the sequences holding chunks lo and hi - 1, found by all threads at once
  int* sq = reinterpret_cast<int*>(sm.base + OFF_SQ);
  if (lo < hi) {
    for (int i = tid; i < S; i += NTHREADS) {
      const int a = cp[i], b = cp[i + 1];
      if (a <= lo && lo < b) sq[0] = i;
      if (a < hi && hi <= b) sq[1] = i;
    }
  }
  __syncthreads();
  const int seq_lo = lo < hi ? sq[0] : 0, seq_hi = lo < hi ? sq[1] : 0;

  ChunkWalk walk;
  walk.cp = cp;
  walk.S = S;
  walk.Hkv = Hkv;
  walk.nl = nl;

  if (warp == 4) {
    // ================= producer =================
    // Block ids travel through a shared-memory ring filled by 4-byte cp.async
    // copies TAB_AHEAD chunks ahead (lane b copies and later uses box b's id;
    // block_size >= 8 keeps a chunk within 16 boxes), so table reads overlap
    // instead of following one another.
    const uint32_t tab = sm.base_u32 + OFF_TAB;
    const int* tab_s = reinterpret_cast<const int*>(sm.base + OFF_TAB);
    auto fetch_ids = [&](const ChunkWalk& w, int slot) {
      const int nb = (w.valid() + p.box_tok - 1) >> p.log2_box;
      if (lane < nb)
        cp_async_4(tab + (slot * 16 + lane) * 4,
                   p.block_tables + (int64_t)w.seq * p.max_blocks +
                       ((w.j * CH + lane * p.box_tok) >> p.log2_bs));
    };
    walk.init(lo, hi, seq_lo, seq_hi);
    ChunkWalk ahead = walk;
#pragma unroll
    for (int d = 0; d < TAB_AHEAD; ++d) {
      if (!ahead.done()) {
        fetch_ids(ahead, d);
        ahead.next();
      }
      cp_async_commit();
    }
    int local = 0, seg = 0;
    for (; !walk.done(); walk.next(), ++local) {
      const int s = local % NST;
      const uint32_t ph = (local / NST) & 1;
      const int cs = walk.j * CH;
      const int valid = walk.valid();
      const int nbox = (valid + p.box_tok - 1) >> p.log2_box;
      cp_async_wait<TAB_AHEAD - 1>();  // this chunk's ids have landed
      const int phys_in = lane < nbox ? tab_s[(local % TAB_SLOTS) * 16 + lane] : 0;
      if (!wait_bar(sm, sm.bar(B_EMPTY + s), ph ^ 1, p.err, 1)) break;
      if (walk.first_of_segment()) {
        const int qs = seg & 1;
        const uint32_t qph = (seg >> 1) & 1;
        if (!wait_bar(sm, sm.bar(B_Q_EMPTY + qs), qph ^ 1, p.err, 2)) break;
        if (lane == 0) {
          const uint32_t dst = sm.base_u32 + OFF_Q + qs * QTILE_B;
          const int row0 = walk.seq * H + walk.g * G;
          ptx::mbar_arrive_expect_tx(sm.bar(B_Q_FULL + qs), QTILE_B);
          ptx::tma_load_2d(dst, &tm_q, sm.bar(B_Q_FULL + qs), 0, row0);
          ptx::tma_load_2d(dst + QTILE_B / 2, &tm_q, sm.bar(B_Q_FULL + qs), 64, row0);
        }
        ++seg;
      }
      const uint32_t bytes = (uint32_t)nbox * p.box_tok * 256u;
      if (p.early_meta && local == 0) ptx::grid_dependency_wait();
      const uint32_t kdst = sm.base_u32 + OFF_K + s * TILE_B;
      const uint32_t vdst = sm.base_u32 + OFF_V + s * TILE_B;
      const uint32_t row = (uint32_t)(lane * p.box_tok) * 128u;
      const int off = (cs + lane * p.box_tok) & (p.block_size - 1);
      int phys = phys_in;
      if (lane < nbox && (unsigned)phys >= (unsigned)p.num_blocks) {
        atomicExch(p.err, 3);  // bad block id: load block 0 instead of faulting
        phys = 0;
      }
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(sm.bar(B_FULL_K + s), bytes);
        ptx::mbar_arrive_expect_tx(sm.bar(B_FULL_V + s), bytes);
      }
      __syncwarp();
      if (lane < nbox) {
        ptx::tma_load_4d(kdst + row, &tm_k, sm.bar(B_FULL_K + s), 0, walk.g, off, phys);
        ptx::tma_load_4d(kdst + HALF_B + row, &tm_k, sm.bar(B_FULL_K + s), 64, walk.g, off, phys);
        ptx::tma_load_4d(vdst + row, &tm_v, sm.bar(B_FULL_V + s), 0, walk.g, off, phys);
        ptx::tma_load_4d(vdst + HALF_B + row, &tm_v, sm.bar(B_FULL_V + s), 64, walk.g, off, phys);
      }
      if (!ahead.done()) {
        fetch_ids(ahead, (local + TAB_AHEAD) % TAB_SLOTS);
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
      for (int sg = max(0, seg - 2); sg < seg; ++sg) drain_bar(sm.bar(B_Q_FULL + (sg & 1)), (sg >> 1) & 1);
    }
  } else if (warp == 5) {
    // ================= MMA issuer =================
    // Two cursors: the logits MMA of chunk nq (needs its K tile, a free S
    // buffer and, at a segment start, the q tile) and the PV MMA of chunk
    // npv < nq (needs P, a free O buffer and the V tile).  The thread polls
    // both and issues whichever is ready, so a stage is released as soon as
    // its own PV completes, never held back by a later chunk's K load.
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = ptx::idesc_bf16_f32(128, NQ, false);
      constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32(128, NQ, true);
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
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t da = ptx::smem_desc_sw128(kbase + (kk >> 2) * HALF_B + (kk & 3) * 32, 16, 1024);
              const uint64_t db = ptx::smem_desc_sw128(qbase + (kk >> 2) * (QTILE_B / 2) + (kk & 3) * 32, 16, 1024);
              ptx::tc_mma_f16(tmem + 16 * b, da, db, IDESC_QK, kk > 0);
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
#pragma unroll
            for (int kk = 0; kk < CH / 16; ++kk) {
              const uint64_t da = ptx::smem_desc_sw128(vbase + kk * 2048, HALF_B, 1024);
              const uint64_t db = ptx::smem_desc_sw128(pbase + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024);
              ptx::tc_mma_f16(tmem + 32 + 16 * b, da, db, IDESC_PV, kk > 0);
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
      const int c0 = cta_of(first, Ktot, C);
      const int c1 = cta_of(first + walk.nch - 1, Ktot, C);
      if (c0 == c1) continue;  // whole unit: the softmax warps wrote the output
      const bool good = wait_bar(sm, sm.bar(B_EPI + (e++ & 1)), 0, p.err, 14);
      if (!good) continue;
      __threadfence();  // the partial written by this CTA is visible before the count
      const int u = walk.seq * Hkv + walk.g;
      const int nseg = c1 - c0 + 1;
      int last = 0;
      if (lane == 0) last = (arrive(&p.counters[u], p.epoch) == nseg);
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) continue;
      __threadfence();  // see every other piece's partial
      const int64_t slot0 = (int64_t)u * p.max_seg;
      float M[G], Ls[G], a[G][4];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        M[h] = -INFINITY;
        Ls[h] = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) a[h][r] = 0.f;
      }
      for (int jj = 0; jj < nseg; ++jj) {
        float2 ml[G];
        float ov[G][4];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          ml[h] = __ldcg(&p.ws_ml[(slot0 + jj) * G + h]);
#pragma unroll
          for (int r = 0; r < 4; ++r) ov[h][r] = __ldcg(&p.ws_o[((slot0 + jj) * G + h) * D + lane + 32 * r]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float mn = fmaxf(M[h], ml[h].x);
          const float rs = fast_exp2(M[h] - mn);  // 0 for the first piece
          const float w = fast_exp2(ml[h].x - mn);
          Ls[h] = Ls[h] * rs + w * ml[h].y;
#pragma unroll
          for (int r = 0; r < 4; ++r) a[h][r] = a[h][r] * rs + w * ov[h][r];
          M[h] = mn;
        }
      }
      __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) +
                         ((int64_t)walk.seq * H + (int64_t)walk.g * G) * D + lane;
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int r = 0; r < 4; ++r)
          o[(int64_t)h * D + 32 * r] = __float2bfloat16_rn(a[h][r] / Ls[h]);
      if (lane == 0) p.counters[u] = p.epoch << 16;  // count 0: a replay starts afresh
    }
  } else {
    // ================= softmax + epilogue (warps 0-3) =================
    const int t = tid;  // TMEM lane: token in S, d in O
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float* red = reinterpret_cast<float*>(sm.base + OFF_RED);
    float* lred = reinterpret_cast<float*>(sm.base + OFF_LRED);
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
        if (lane == 0) lred[warp * 8 + h] = v;
      }
      ptx::bar_sync_named(2, 128);
#pragma unroll
      for (int h = 0; h < G; ++h) lt[h] = lred[h] + lred[8 + h] + lred[16 + h] + lred[24 + h];
      ptx::bar_sync_named(2, 128);
      const long long first = in.k - in.j;            // unit's first chunk (global)
      const long long last = first + in.nch - 1;       // unit's last chunk
      const int c0 = cta_of(first, Ktot, C);
      const int c1 = cta_of(last, Ktot, C);
      const int u = in.seq * Hkv + in.g;
      __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) +
                         ((int64_t)in.seq * H + (int64_t)in.g * G) * D + t;
      if (c0 == c1) {
#pragma unroll
        for (int h = 0; h < G; ++h) o[(int64_t)h * D] = __float2bfloat16_rn(acc[h] / lt[h]);
      } else {
        // a piece of a split unit: leave the partial for the merge warp
        const int64_t slot = (int64_t)u * p.max_seg + ((int)blockIdx.x - c0);
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
      float ov[8];
      const bool good = wait_bar(sm, sm.bar(B_O_FULL + b), bph, p.err, 10);
      ptx::tc_fence_after();
      ptx::tmem_ld_x8(tmem + lane_base + 32 + 16 * b, ov);
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(sm.bar(B_O_EMPTY + b));
      if (!good) {
#pragma unroll
        for (int h = 0; h < G; ++h) ov[h] = 0.f;
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
      float sv[8];
      const bool good = wait_bar(sm, sm.bar(B_S_FULL + b), bph, p.err, 11);
      ptx::tc_fence_after();
      ptx::tmem_ld_x8(tmem + lane_base + 16 * b, sv);
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(sm.bar(B_S_EMPTY + b));
      const int valid = walk.valid();
      float x[G];
#pragma unroll
      for (int h = 0; h < G; ++h) x[h] = (good && t < valid) ? sv[h] * p.scale_log2 : -INFINITY;
      // ---- chunk max per head over the 128 lanes ----
      float* rb = red + b * 32;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float v = ptx::warp_max_f32(x[h]);
        if (lane == 0) rb[warp * 8 + h] = v;
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
      __nv_bfloat16 pb[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float cmax = fmaxf(fmaxf(rb[h], rb[8 + h]), fmaxf(rb[16 + h], rb[24 + h]));
        const float m_new = fmaxf(m[h], cmax);
        alpha[h] = fast_exp2(m[h] - m_new);
        m[h] = m_new;
        const float pv = (t < valid) ? fast_exp2(x[h] - m_new) : 0.f;
        pb[h] = __float2bfloat16_rn(pv);
        l[h] = l[h] * alpha[h] + __bfloat162float(pb[h]);
      }
      // ---- P tile (and the V tail) for the PV MMA ----
      wait_bar(sm, sm.bar(B_P_EMPTY + b), bph ^ 1, p.err, 12);
      if (valid < CH) {
        wait_bar(sm, sm.bar(B_FULL_V + s), ph, p.err, 13);
        if (t >= valid) {
          unsigned char* vrow = sm.base + OFF_V + s * TILE_B + t * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int cc = (c + t) & 7;
            *reinterpret_cast<uint4*>(vrow + cc * 16) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(vrow + HALF_B + cc * 16) = make_uint4(0, 0, 0, 0);
          }
        }
      }
      {
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

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

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

template <int G>
cudaError_t launch_g(const TcLaunch& a, const Params& prm, const CUtensorMap& mk,
                     const CUtensorMap& mv, const CUtensorMap& mq, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.num_ctas);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  // programmatic dependent launch: the prologue may overlap the previous
  // kernel; the kernel waits for it (griddepcontrol.wait) before reading inputs
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_tc_kernel<G>, mk, mv, mq, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace tc

size_t tc_workspace_bytes(int64_t num_seqs, int64_t num_heads, int64_t max_ctx, int num_ctas) {
  const int64_t max_chunks = (max_ctx + tc::CH - 1) / tc::CH;
  const int64_t max_seg = max_chunks < num_ctas ? max_chunks : num_ctas;
  const int64_t rows = num_seqs * num_heads;  // >= units * G
  size_t off = 256;                                             // error word
  off += ((size_t)rows * 8 + 255) / 256 * 256;                  // merge counters
  off += ((size_t)rows * max_seg * 8 + 255) / 256 * 256;        // (m, l)
  off += (size_t)rows * max_seg * tc::D * 4;                    // partial o
  return off;
}

bool tc_supported(int head_dim, int group, bool fp8, int num_seqs, int block_size) {
  // block_size >= 8 keeps every TMA destination 1024-byte aligned (whole
  // 128-byte-swizzle atoms)
  return head_dim == tc::D && !fp8 && (group == 1 || group == 2 || group == 4 || group == 8) &&
         num_seqs <= tc::kMaxSeqs && block_size >= 8 && tc::encode_fn() != nullptr;
}

cudaError_t launch_decode_tc(const TcLaunch& a, cudaStream_t stream) {
  using namespace tc;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int box_tok = a.block_size < CH ? a.block_size : CH;
  CUtensorMap mk, mv, mq;
  {
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)a.num_kv_heads, (cuuint64_t)a.block_size,
                          (cuuint64_t)a.num_blocks};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)a.num_kv_heads * D * 2,
                             (cuuint64_t)a.block_size * a.num_kv_heads * D * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)box_tok, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.k_cache), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (enc(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.v_cache), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)a.num_seqs * a.num_heads};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, NQ};
    cuuint32_t es[2] = {1, 1};
    if (enc(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.q), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int64_t max_ctx = (int64_t)a.max_blocks * a.block_size;
  const int64_t max_chunks = (max_ctx + CH - 1) / CH;
  Params prm{};
  prm.out = a.out;
  prm.block_tables = a.block_tables;
  prm.context_lens = a.context_lens;
  char* ws = static_cast<char*>(a.workspace);
  const int64_t rows = (int64_t)a.num_seqs * a.num_heads;
  prm.num_ctas = a.num_ctas;
  prm.max_seg = (int)(max_chunks < a.num_ctas ? max_chunks : a.num_ctas);
  size_t off = 0;
  prm.err = reinterpret_cast<int*>(ws + off);
  off += 256;
  prm.counters = reinterpret_cast<unsigned long long*>(ws + off);
  off += ((size_t)rows * 8 + 255) / 256 * 256;
  prm.ws_ml = reinterpret_cast<float2*>(ws + off);
  off += ((size_t)rows * prm.max_seg * 8 + 255) / 256 * 256;
  prm.ws_o = reinterpret_cast<float*>(ws + off);
  prm.num_seqs = a.num_seqs;
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
  prm.early_meta = a.early_meta ? 1 : 0;
  {
    // a distinct 48-bit tag per call (the merge counters' epoch)
    static std::atomic<unsigned long long> next_epoch{0x5eed00000000ull};
    prm.epoch = next_epoch.fetch_add(1, std::memory_order_relaxed) & 0xFFFFFFFFFFFFull;
  }
  const int G = a.num_heads / a.num_kv_heads;
  switch (G) {
    case 1: return launch_g<1>(a, prm, mk, mv, mq, stream);
    case 2: return launch_g<2>(a, prm, mk, mv, mq, stream);
    case 4: return launch_g<4>(a, prm, mk, mv, mq, stream);
    case 8: return launch_g<8>(a, prm, mk, mv, mq, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
