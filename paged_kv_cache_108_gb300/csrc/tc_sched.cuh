// Scheduling and synchronisation pieces shared by the tensor-core decode
// kernels: bounded mbarrier waits, the per-unit arrival counter of split
// units, the equal split of a chunk numbering over persistent CTAs, and the
// walk over one CTA's chunk range.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "tc_ptx.cuh"

namespace pa {
namespace tc {

// a wait that has not completed after this many clocks (~1 s) gives up
constexpr long long kWaitClocks = 1LL << 31;

struct Smem {
  unsigned char* base;
  uint32_t base_u32;
  int off_bar, off_abort;
  __device__ uint32_t bar(int i) const { return base_u32 + off_bar + 8 * i; }
  __device__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(base + off_abort); }
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

// arrive() for a piece that expects to be its unit's last: the first
// exchange assumes the other nseg - 1 pieces have counted, so the usual
// last arrival costs one atomic round trip instead of a read and an atomic.
__device__ __forceinline__ int arrive_expect_last(unsigned long long* cnt, unsigned long long epoch,
                                                  int nseg) {
  const unsigned long long guess = (epoch << 16) | (unsigned long long)(nseg - 1);
  unsigned long long v = atomicCAS(cnt, guess, guess + 1);
  if (v == guess) return nseg;
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

// Slot of CTA c's partial for the split unit whose last chunk is `last`: 0
// if the unit holds the CTA's last chunk, else 1 (the unit its range starts
// in).  A CTA's range has at most these two split units, so partials live in
// two slots per CTA whatever the batch's shape.
__device__ __forceinline__ int piece_slot(int c, long long last, long long K, int C) {
  return range_lo(c + 1, K, C) - 1 <= last ? 0 : 1;
}

// Walks this CTA's chunk range; identical in every role.  The range is
// visited as up to three contiguous pieces: the unit it ends in (shared with
// the next CTA), then the unit it starts in (shared with the previous CTA),
// then the whole units in between.  Both pieces of every split unit are thus
// finished early in their CTAs, so the merge of a split unit happens while
// the pipeline still has work to hide it, and every CTA ends on whole units.
template <int CH>
struct ChunkWalk {
  const int* cp;   // smem chunk prefix: cp[i] = chunks of sequences < i (one head)
  const int* nl;   // smem clamped context lengths
  int S, Hkv;
  long long Ctot;  // chunks of one head over all sequences (cp[S])
  int first_ne;    // first sequence with a chunk
  long long k;                 // current global chunk index
  long long lo0, hi0, lo1, hi1, lo2, hi2;  // the pieces, in visiting order
  long long cur_lo, cur_hi;    // the piece being visited
  int nsub, si;
  int seq, g, j, nch, n;

  int sq1, g1, j1, sq2, g2;    // where pieces 1 and 2 start (piece 2 starts a unit)

  __device__ void load_unit() {
    nch = cp[seq + 1] - cp[seq];
    n = nl[seq];
  }
  // position (seq, g, j) of chunk kk, given the sequence s holding it
  __device__ void seek_in(int s, long long kk) {
    k = kk;
    seq = s;
    load_unit();
    g = (int)(kk / Ctot);
    j = (int)(kk - g * Ctot - cp[s]);
  }
  // the unit after (q, h): the next sequence with chunks, or the next head
  __device__ void next_unit(int& q, int& h) const {
    do { ++q; } while (q < S && cp[q + 1] == cp[q]);
    if (q == S) {
      q = first_ne;
      ++h;
    }
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
    g2 = g;
    next_unit(sq2, g2);
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
      next_unit(seq, g);
      load_unit();
    }
  }
  __device__ bool first_of_segment() const { return j == 0 || k == cur_lo; }
  __device__ bool last_of_segment() const { return j == nch - 1 || k == cur_hi - 1; }
  __device__ int valid() const { return min(CH, n - j * CH); }
};

// ---- host side (defined in decode_tc.cu) ----
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// cuTensorMapEncodeTiled from the driver, or nullptr
EncodeTiledFn encode_fn();
// a distinct 48-bit tag per call of either tensor-core kernel (the epoch of
// the split-unit arrival counters, which both kernels keep at the same
// workspace offset)
unsigned long long next_call_epoch();

}  // namespace tc
}  // namespace pa
