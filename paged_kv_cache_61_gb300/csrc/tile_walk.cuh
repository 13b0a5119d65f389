// Shared device helpers of the decode kernels: the walk over a CTA's range of the
// flattened (sequence, segment, page) tile list, bounded pipeline waits and the
// write-out of the split pieces.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace pda {

constexpr unsigned kFullMask = 0xffffffffu;

// Query rows of a segment: the S query tokens of each of its G heads, row r = i*G + g
// for query token i and head seg*G + g (FlashMLA-ETAP "Usage": s_q * h_q / h_kv query
// rows per KV head). q and out rows are laid out [B][S][Hq], lse [B][Hq][S]; with S = 1
// these are the single-token layouts [B][Hq].
struct RowIndex {
  int64_t out_row;  // row of q and out
  int64_t lse;      // element of lse
};
__device__ __forceinline__ RowIndex seg_row(int b, int seg, int r, int G, int S, int Hq) {
  const int i = r / G;
  const int h = seg * G + (r - i * G);
  return {(int64_t(b) * S + i) * Hq + h, (int64_t(b) * Hq + h) * S + i};
}

// What the walk needs to know about the batch. A segment is one (sequence, KV
// head) for GQA or one (sequence, head group) for MLA.
struct WalkSpec {
  const int32_t* context_lens;
  int32_t batch;
  int32_t segs_per_seq;
  int32_t page;
};

struct Walker {
  int b;
  int np;           // pages of sequence b
  int64_t start_b;  // flattened index of sequence b's first tile
  int64_t g;        // next tile to visit
};

// A maximal run of the CTA's tiles inside one segment: pages [p0, p1) of
// segment `seg` of sequence b, whose first tile has flattened index seg_start.
struct Portion {
  int b, seg, p0, p1, np;
  int64_t seg_start;
};

__device__ __forceinline__ int pages_of(int ctx, int page) { return (ctx + page - 1) / page; }

// Warp-collective: position the walker on flattened tile g (prefix sums over the
// sequences' tile counts, 32 sequences per step).
__device__ __forceinline__ void walker_init(Walker& w, const WalkSpec& s, int64_t g, int lane) {
  int64_t base = 0;
  w.b = s.batch;
  w.start_b = 0;
  w.np = 1;
  w.g = g;
  for (int b0 = 0; b0 < s.batch; b0 += 32) {
    const int b = b0 + lane;
    const int np = b < s.batch ? pages_of(__ldg(s.context_lens + b), s.page) : 0;
    const int64_t width = int64_t(np) * s.segs_per_seq;
    int64_t incl = width;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t t = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += t;
    }
    const int64_t excl = incl - width;
    const unsigned hit =
        __ballot_sync(kFullMask, b < s.batch && base + excl <= g && g < base + incl);
    if (hit) {
      const int src = __ffs(hit) - 1;
      w.b = b0 + src;
      w.start_b = base + __shfl_sync(kFullMask, excl, src);
      w.np = __shfl_sync(kFullMask, np, src);
      return;
    }
    base += __shfl_sync(kFullMask, incl, 31);
  }
}

// Next portion of the range ending at g_hi (uniform across the calling warp).
__device__ __forceinline__ Portion walker_next(Walker& w, const WalkSpec& s, int64_t g_hi) {
  const int64_t off = w.g - w.start_b;
  const int seg = int(off / w.np);
  const int p0 = int(off - int64_t(seg) * w.np);
  const int p1 = int(min(int64_t(w.np), int64_t(p0) + (g_hi - w.g)));
  Portion pt{w.b, seg, p0, p1, w.np, w.start_b + int64_t(seg) * w.np};
  w.g += p1 - p0;
  if (p1 == w.np && seg + 1 == s.segs_per_seq) {
    w.start_b += int64_t(s.segs_per_seq) * w.np;
    ++w.b;
    if (w.b < s.batch && w.g < g_hi) w.np = pages_of(__ldg(s.context_lens + w.b), s.page);
  }
  return pt;
}

// Wait for an mbarrier phase; gives up on timeout or when another warp aborted.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (ptx::globaltimer() - t0 > ptx::kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// CTA-local slot of a split piece: 0 if the piece starts this CTA's range (the
// segment began at or before the range), 1 if it ends the range.
__device__ __forceinline__ int piece_slot(int64_t seg_start, int64_t g_lo) {
  return seg_start <= g_lo ? 0 : 1;
}

}  // namespace pda
