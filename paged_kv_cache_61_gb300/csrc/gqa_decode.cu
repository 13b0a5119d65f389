// GQA / MQA / MHA paged decode attention for sm_103a.
//
// What it computes ("From MHA to MLA", sections 3-5; drill page "L2 讲解：paged
// decode attention 与 GQA", sections ③-⑤): for each sequence b and KV head kvh,
// the G = Hq/Hkv query heads kvh*G .. kvh*G+G-1 (contiguous grouping) attend to
// the ctx_b cached tokens, gathered page by page through the block table, with
// an online softmax; long sequences are split Flash-Decoding style and the
// splits merged by their log-sum-exp.
//
// How (GB300 design, not the pages' Triton/Hopper kernels):
//  * Persistent-free, equal-work CTAs: the plan gives every CTA the same number
//    of (sequence, KV head, page) tiles in one flattened list, so one wave of
//    CTAs covers any batch mix (uniform, one 32K sequence, varlen).
//  * Two producer warps walk the CTA's tiles and take the ring fills alternately;
//    each reads the block table 32 entries at a time and issues TMA tile loads
//    (maps over [block, slot, kvh, d], coordinates (d, kvh, phys): the 64-bit
//    address is formed by the TMA unit, so no 32-bit product phys*stride exists)
//    of each page's K and V into a ring of shared-memory stages with 128-byte
//    swizzle. A stage holds one page, or two (fp8 caches; 25-32 rows per segment).
//  * Four consumer warps (eight for 25-32 rows per segment) take stages round-robin
//    (by CTA-local fill index, so a ring stage always has the same consumers).
//    Each page is one m16n8k16 tile in the transposed ("keys on M") orientation
//    the FlashMLA-ETAP README describes for Hopper WGMMA, here on warp MMA:
//    S^T[16 tokens x 8 heads] = K * Q^T, so a group of 4 heads wastes half an MMA
//    instead of 3/4 of one.
//    The online softmax runs down each column (head) with three shuffles;
//    P^T is turned into the B fragment of O^T += V^T * P^T with movmatrix.
//  * Stale slots of a partial last page are removed by selects on the scores
//    and on the V^T fragments, never by multiplying, so whatever the slots
//    hold (even NaN) cannot reach the output.
//  * At the end of each (sequence, KV head) piece the warps merge their states
//    in shared memory; a complete segment is written directly, a split piece
//    writes (O_s, L_s) to its CTA's slot. A segment cut into a few pieces is
//    merged ("From MHA to MLA", section 4) by the last piece to arrive (atomic
//    counter, reset afterwards); one cut into many pieces (a single long
//    sequence, MQA) is merged by the split-merge kernel, which the decode grid
//    releases early through programmatic dependent launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>
#include <type_traits>

#include "pda_internal.h"
#include "ptx.cuh"
#include "tile_walk.cuh"

namespace pda {

namespace {

constexpr int kPage = 16;
constexpr int kConsumerWarps = 4;
// Two producer warps take the ring fills alternately: one warp's per-fill chain (barrier
// wait, expect-tx, tensor-copy issue) took longer than the consumers needed per fill.
constexpr int kProducerWarps = 2;
// Ring stages: a multiple of the consumer warps, so stage s is only ever read by
// the warps whose fills are t = s (mod consumer warps / NHT), each of which takes
// every fill of that stage in order (the parity waits rely on this).
#ifndef PDA_GQA_STAGES
#define PDA_GQA_STAGES 8
#endif
#ifndef PDA_GQA_CTAS_PER_SM
#define PDA_GQA_CTAS_PER_SM 2
#endif
#ifndef PDA_GQA_WIDE32
#define PDA_GQA_WIDE32 1
#endif
// Warp roles. Segments of 25-32 rows (four head subtiles) run eight consumer warps, two
// per subtile taking alternate stages, in one CTA per SM: with four, one warp per subtile
// walks every page of the CTA's range, and a single long sequence (MQA) then waits on that
// one warp's chain of dependent MMAs and shuffles per page. B=1, ctx 32K, MQA: a step on
// its own 26.1 -> 21.1 us with 16-bit caches, 29.1 -> 24.0 us with fp8 (back to back
// unchanged, 5.8 and 6.8 us); B=64, ctx 1K, MQA 12.06 -> 11.20 us back to back.
template <int NHT>
struct Roles {
  static constexpr int kConsumer = (PDA_GQA_WIDE32 && NHT == 4) ? 8 : kConsumerWarps;
  static constexpr int kThreads = (kConsumer + kProducerWarps) * 32;
  static constexpr int kCtasPerSm = kConsumer == 8 ? 1 : PDA_GQA_CTAS_PER_SM;
};
#ifndef PDA_GQA_STAGES_F8
#define PDA_GQA_STAGES_F8 8
#endif
constexpr int kStages16 = PDA_GQA_STAGES;     // ring stages for 16-bit caches
constexpr int kStagesF8 = PDA_GQA_STAGES_F8;  // ring stages for fp8 caches
constexpr int kBoxBytes = kPage * 128;  // one TMA box: 16 tokens x 64 dims x 16 bit
constexpr int kCtasPerSm = PDA_GQA_CTAS_PER_SM;
constexpr unsigned kFull = kFullMask;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct GqaParams {
  const void* q;
  void* out;
  float* lse;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t batch, num_q_heads, num_kv_heads, group, max_blocks;
  int32_t heads_per_kv, seq_len_q;  // G and S: a KV head's rows are r = i*G + g
  // A KV head's S*G rows form row_chunks segments of `group` rows (the last one may hold
  // fewer): segment seg is KV head seg / row_chunks, rows (seg % row_chunks) * group + j.
  int32_t row_chunks, segs_per_seq;
  int64_t num_blocks;
  float scale_log2;     // softmax scale (times k_scale for fp8 caches) times log2(e)
  float v_scale;        // fp8 caches: V dequantization scale (1 for 16-bit caches)
  // fp8 caches: 0 = separate K and V maps; 1 = one map whose last dimension (extent 2,
  // stride |v - k|) selects K then V, so one copy lands a page's K and V tiles; 2 = the
  // same with V first (v_cache below k_cache)
  int32_t kv_pair;
  int64_t total_tiles, tiles_per_cta;
  int32_t heavy_min;  // split segments with more pieces are merged by the split-merge kernel
  int32_t* err;
  int32_t* counters;
  float* part_lse;
  float* part_out;
};

// F8: E4M3 caches. A (page, kvh) tile of one tensor is then 16 rows of D bytes (one
// TMA box, 128-byte swizzle for D = 128, 64-byte for D = 64), half the bytes of the
// 16-bit tile, and a ring stage holds two consecutive pages ([K A][V A][K B][V B]), so
// a stage carries as many bytes as a 16-bit one and the per-stage costs (producer
// issue, barrier waits, the softmax reductions) are paid once per two pages.
// 16-bit caches with four head subtiles (25-32 rows per segment) take two pages per stage
// as well: a consumer warp owns one subtile and walks every other stage of the range, and
// two pages per step give its chain of dependent MMAs, shuffles and exponentials twice
// the independent work (B=1, ctx 32K, MQA with four consumer warps and four stages: 7.01
// -> 5.78 us; the eight consumer warps of Roles take eight such stages). With fewer rows
// the warps share a subtile's pages, and one page per stage is faster (B=64, ctx 1K:
// 37.98 against 38.69 us with two).
template <int D, bool F8, int NHT>
struct Layout {
  static constexpr int kDBlocks = D / 64;
  static constexpr int kPPT = (F8 || NHT == 4) ? 2 : 1;    // pages per ring fill
  static constexpr int kCW = Roles<NHT>::kConsumer;     // consumer warps
  static constexpr int kStages =
      F8 ? kStagesF8 : (kPPT == 2 && kCW == 4 ? kStages16 / 2 : kStages16);
  static constexpr int kTileBytes = F8 ? kPage * D : kDBlocks * kBoxBytes;  // page, tensor
  static constexpr int kStageBytes = 2 * kPPT * kTileBytes;
  static constexpr int kMergeStride = D + 4;  // floats per head row; +4 spreads banks
  static constexpr int kMergeWarpFloats = 8 * kMergeStride + 16;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kMergeBytes = kCW * kMergeWarpFloats * 4;
  static constexpr int kBarBytes = 2 * kStages * 8 + 16;
  static constexpr int kSmemBytes = 1024 + kRingBytes + kMergeBytes + kBarBytes;
  static_assert(kStages % kCW == 0, "each stage needs a fixed set of consumer warps");
};

// Byte offset of 16-byte chunk `ch` of row `r` in a swizzled fp8 tile of 16 rows of D
// bytes: the TMA 128-byte swizzle XORs address bits 4-6 with bits 7-9, the 64-byte
// swizzle bits 4-5 with bits 7-8 (the ring stages are 1024-byte aligned).
template <int D>
__device__ __forceinline__ uint32_t f8_tile_offset(int r, int ch) {
  if constexpr (D == 128) return uint32_t(r * 128 + ((ch ^ (r & 7)) << 4));
  else return uint32_t(r * 64 + ((ch ^ ((r >> 1) & 3)) << 4));
}

template <typename T>
__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  uint4 r;
  r.x = ptx::Mma<T>::pack(v[0], v[1]);
  r.y = ptx::Mma<T>::pack(v[2], v[3]);
  r.z = ptx::Mma<T>::pack(v[4], v[5]);
  r.w = ptx::Mma<T>::pack(v[6], v[7]);
  return r;
}

// A packed pair of q's type as a pair of the MMAs' type (the same bits when they agree).
template <typename T, typename TM>
__device__ __forceinline__ uint32_t to_mma_pair(uint32_t w) {
  if constexpr (std::is_same_v<T, TM>) {
    return w;
  } else {
    float lo, hi;
    ptx::Mma<T>::unpack(w, lo, hi);
    return ptx::Mma<TM>::pack(lo, hi);
  }
}

// ------------------------------------------------------------------ the kernel
template <int D, typename T, int NHT, bool F8>
__global__ void __launch_bounds__(Roles<NHT>::kThreads, Roles<NHT>::kCtasPerSm)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const GqaParams p) {
  using L = Layout<D, F8, NHT>;
  // the MMAs' operand type: q's type, except over E4M3 caches, whose codes convert to
  // fp16 in one instruction per pair (to bf16 it takes three more); q is then converted
  // to fp16 as it is loaded (exact for |q| in [2^-14, 65504])
  using TM = std::conditional_t<F8, __half, T>;
  constexpr int kStages = L::kStages;
  constexpr int kPPT = L::kPPT;
  constexpr int kWP = L::kCW / NHT;  // consumer warps sharing one head subtile
  constexpr int kKS = D / 16;                // k-steps of S^T and m-tiles of O^T

  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = align1024(smem_raw);
  float* merge = reinterpret_cast<float*>(ring + L::kRingBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + L::kRingBytes + L::kMergeBytes);
  uint64_t* empty = full + kStages;
  volatile int* flags = reinterpret_cast<volatile int*>(empty + kStages);  // [0] abort, [1] last

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t g_lo = int64_t(blockIdx.x) * p.tiles_per_cta;
  const int64_t g_hi = min(p.total_tiles, g_lo + p.tiles_per_cta);
  // Let the split-merge grid that may follow on this stream be scheduled early; it
  // waits for this grid's completion before it reads anything.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (g_lo >= g_hi) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], NHT);
    }
    flags[0] = 0;
    flags[1] = 0;
    ptx::fence_mbarrier_init();
  }
  __syncthreads();

  const WalkSpec spec{p.context_lens, p.batch, p.segs_per_seq, kPage};
  Walker walk;
  walker_init(walk, spec, g_lo, lane);

  if (warp >= L::kCW) {
    // ============================== producer warps ==============================
    // Both walk every fill of the CTA's range; producer pw issues the fills f with
    // f = pw (mod kProducerWarps) and skips the others.
    const int pw = warp - L::kCW;
    if (lane == 0) {
      ptx::prefetch_tensormap(&tm_k);
      ptx::prefetch_tensormap(&tm_v);
    }
    const uint64_t policy = ptx::policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t filled = 0;  // bit s: stage s was filled (by this warp) at least once
    int fill = 0;         // CTA-local fill index
    bool ok = true;
    while (ok && walk.g < g_hi) {
      const Portion pt = walker_next(walk, spec, g_hi);
      const int kvh = pt.seg / p.row_chunks;
      const int32_t* row = p.block_tables + int64_t(pt.b) * p.max_blocks;
      int32_t next = (pt.p0 + lane < pt.p1) ? __ldg(row + pt.p0 + lane) : 0;
      for (int base = pt.p0; ok && base < pt.p1; base += 32) {
        const int32_t cur = next;
        if (base + 32 < pt.p1) next = (base + 32 + lane < pt.p1) ? __ldg(row + base + 32 + lane) : 0;
        const int n = min(32, pt.p1 - base);
        // a fill takes kPPT consecutive pages; a batch starts kPPT-aligned within the
        // portion (32 is a multiple of kPPT), so a fill never spans two batches
        for (int j = 0; j < n; j += kPPT, ++fill) {
          if (fill % kProducerWarps != pw) {
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          const int32_t phys = __shfl_sync(kFull, cur, j);
          const int32_t phys2 = __shfl_sync(kFull, cur, min(j + 1, 31));
          const bool two = kPPT == 2 && j + 1 < n;
          int good = 1;
          if (lane == 0) {
            if (!wait_phase(&empty[stage], phase ^ 1, flags)) {
              good = 0;
            } else {
              // An id outside the pool is flagged; TMA fills such a tile with zeros.
              if (phys < 0 || int64_t(phys) >= p.num_blocks ||
                  (two && (phys2 < 0 || int64_t(phys2) >= p.num_blocks)))
                atomicOr(p.err, 1);
              ptx::mbar_arrive_expect_tx(&full[stage],
                                         two ? L::kStageBytes : 2 * L::kTileBytes);
            }
          }
          ok = __shfl_sync(kFull, good, 0) != 0;
          if (!ok) break;
          // The fill's copies are issued by several lanes at once (one copy per lane; a
          // single thread issuing them one after another was the producer's bottleneck):
          // lane c copies tensor c & 1 (K, V) of page c >> 1 into [K A][V A][K B][V B].
          // fp8: box (D bytes, 1 kvh, 16 slots, 1 block); 16-bit: box (64 d, 16 slots,
          // D/64 d-blocks, 1 kvh, 1 block), landing as D/64 swizzled [16][64] sub-tiles.
          if (F8 && p.kv_pair != 0) {
            // fp8, one map over both caches: lane c copies page c's K and V tiles at once
            if (lane < (two ? 2 : 1)) {
              uint8_t* dst = ring + stage * L::kStageBytes + lane * 2 * L::kTileBytes;
              ptx::tma_load_5d(dst, &tm_k, &full[stage], 0, kvh, 0, lane ? phys2 : phys, 0,
                               policy);
            }
          } else if (lane < (two ? 4 : 2)) {
            const CUtensorMap* map = (lane & 1) ? &tm_v : &tm_k;
            uint8_t* dst = ring + stage * L::kStageBytes + lane * L::kTileBytes;
            const int32_t ph = (lane >> 1) ? phys2 : phys;
            if constexpr (F8)
              ptx::tma_load_4d(dst, map, &full[stage], 0, kvh, 0, ph, policy);
            else
              ptx::tma_load_5d(dst, map, &full[stage], 0, 0, 0, kvh, ph, policy);
          }
          filled |= 1u << stage;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    if (!ok && lane == 0) {
      flags[0] = 1;
      atomicOr(p.err, 2);
    }
    // Never leave with a copy in flight: wait (bounded) for each stage's last fill.
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        if (!(filled >> s & 1)) continue;
        // stages before `stage` were last filled in `phase`, the rest in phase ^ 1
        const uint32_t par = (s < stage) ? phase : (phase ^ 1);
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(&full[s], par) && ptx::globaltimer() - t0 < ptx::kWaitLimitNs) {
        }
      }
    }
    return;
  }

  // ============================== consumer warps ==============================
  // The grid may start while the previous kernel on the stream drains (programmatic
  // dependent launch; only this library's decode and split-merge kernels allow that, and
  // any other predecessor, the caller's kernels included, has completed before this grid
  // starts). None of those kernels writes q, the caches, the tables or the lengths, so
  // the consumers read them and attend to their pages at once; they write out, lse and
  // the workspace, which the previous grid may still be reading or writing, only after
  // the griddepcontrol.wait at the end of each portion's page loop.
  const int hsub = warp % NHT;
  const int pres = warp / NHT;
  const int tid = threadIdx.x;  // 0..127 among consumers
  const T* __restrict__ qg = static_cast<const T*>(p.q);
  T* __restrict__ outg = static_cast<T*>(p.out);
  float* mw = merge + warp * L::kMergeWarpFloats;
  const int r0 = lane >> 2;            // token row (S^T) / d row (O^T) of this lane
  const int cq = 2 * (lane & 3);       // first of the two head columns of this lane
  // ldmatrix lane roles
  const int tok_k = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int chunk_k = lane >> 4;
  const int tok_v = (lane & 7) + ((lane >> 4) & 1) * 8;
  const int chunk_v = (lane >> 3) & 1;
  const uint32_t ring_s = ptx::smem_addr(ring);

  bool aborted = false;
  int64_t k = 0;  // CTA-local index of the current portion's first tile
  while (walk.g < g_hi) {
    const Portion pt = walker_next(walk, spec, g_hi);
    const int ctx = __ldg(p.context_lens + pt.b);
    const int npg = pt.p1 - pt.p0;
    // the segment's KV head, its first row and its row count
    const int kvh = pt.seg / p.row_chunks;
    const int rbase = (pt.seg - kvh * p.row_chunks) * p.group;
    const int nrows = min(p.group, p.heads_per_kv * p.seq_len_q - rbase);

    // Q^T as the B operand (k = head dim, n = head): lane holds head hsub*8 + lane/4.
    // fp8 caches: the K fragment of a lane holds 4 consecutive dims of a token (one
    // 32-bit shared-memory word) as its k indices {cq, cq+1, cq+8, cq+9}; the dot
    // product does not depend on the order of k, so q takes the same assignment:
    // dims 16ks + 2cq, +1 as k = cq, cq+1 and dims 16ks + 2cq + 2, +3 as k = cq+8, cq+9.
    const int jq = hsub * 8 + r0;
    uint32_t qf[kKS][2];
    {
      const bool hv = jq < nrows;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          qg + seg_row(pt.b, kvh, rbase + (hv ? jq : 0), p.heads_per_kv, p.seq_len_q,
                       p.num_q_heads).out_row * D);
#pragma unroll
      for (int ks = 0; ks < kKS; ++ks) {
        if constexpr (F8) {
          qf[ks][0] = hv ? to_mma_pair<T, TM>(__ldg(qrow + (ks * 16 + 2 * cq) / 2)) : 0u;
          qf[ks][1] = hv ? to_mma_pair<T, TM>(__ldg(qrow + (ks * 16 + 2 * cq + 2) / 2)) : 0u;
        } else {
          qf[ks][0] = hv ? __ldg(qrow + (ks * 16 + cq) / 2) : 0u;
          qf[ks][1] = hv ? __ldg(qrow + (ks * 16 + 8 + cq) / 2) : 0u;
        }
      }
    }

    // Causal limits of this lane's two columns (segment rows hsub*8 + cq, + 1): row
    // r = i*G + g of the KV head is query token i, which sees tokens [0, ctx - S + 1 + i)
    // (bottom-right aligned; all ctx tokens when S = 1). Padded rows take ctx.
    int lim0 = ctx, lim1 = ctx;
    if (p.seq_len_q > 1) {
      const int ra = hsub * 8 + cq;
      if (ra < nrows) lim0 = ctx - p.seq_len_q + 1 + (rbase + ra) / p.heads_per_kv;
      if (ra + 1 < nrows) lim1 = ctx - p.seq_len_q + 1 + (rbase + ra + 1) / p.heads_per_kv;
    }

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc[kKS][4];
#pragma unroll
    for (int mt = 0; mt < kKS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

    // This warp's ring fills are those with CTA-local index t = pres (mod kWP). A fill
    // holds kPPT consecutive pages of the portion (two for fp8 caches, so a stage moves
    // as many bytes as a 16-bit page; two for 16-bit caches with four head subtiles).
    const int nfill = (npg + kPPT - 1) / kPPT;
    const int first = int(((pres - k) % kWP + kWP) % kWP);
    for (int i = first; i < nfill; i += kWP) {
      const int64_t t = k + i;
      const int stage = int(t % kStages);
      const uint32_t par = uint32_t(t / kStages) & 1u;
      if (!aborted && !wait_phase(&full[stage], par, flags)) {
        aborted = true;
        if (lane == 0) {
          flags[0] = 1;
          atomicOr(p.err, 2);
        }
      }
      if (aborted) continue;
      const uint32_t kb = ring_s + stage * L::kStageBytes;
      if constexpr (F8) {
        // ---- two pages A, B (B may be absent at a portion's end: then its slots are
        // all stale, masked below exactly like the stale slots of a partial page)
        const int pg0 = (pt.p0 + i * kPPT) * kPage;  // first token of page A
        const int vld[2] = {min(kPage, ctx - pg0),
                            (i * kPPT + 1 < npg) ? min(kPage, ctx - pg0 - kPage) : 0};
        // a page's two tiles: K then V, or V then K when one map reads V first
        const uint32_t koff = p.kv_pair == 2 ? L::kTileBytes : 0;
        const uint32_t voff = p.kv_pair == 2 ? 0 : L::kTileBytes;
        const uint32_t kpg[2] = {kb + koff, kb + 2 * L::kTileBytes + koff};
        // S^T = K * Q^T for both pages: two independent accumulation chains. One
        // ldmatrix.x4 covers two k-steps: matrices (tokens 0-7 | 8-15) x (chunk ks |
        // ks+1) of 16 bytes; a lane gets 4 consecutive bytes (dims) of one token.
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < kKS; ks += 2) {
          uint32_t x[2][4];
#pragma unroll
          for (int hp = 0; hp < 2; ++hp)
            ptx::ldsm_x4(kpg[hp] + f8_tile_offset<D>(tok_k, ks + chunk_k), x[hp][0], x[hp][1],
                         x[hp][2], x[hp][3]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int hp = 0; hp < 2; ++hp) {
              uint32_t a[4];
              ptx::Mma<TM>::from_e4m3x4(x[hp][2 * h], a[0], a[2]);       // token r0
              ptx::Mma<TM>::from_e4m3x4(x[hp][2 * h + 1], a[1], a[3]);   // token r0 + 8
              ptx::Mma<TM>::run(s[hp], a, qf[ks + h][0], qf[ks + h][1]);
            }
          }
        }
        float x[2][4];
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {
#pragma unroll
          for (int e = 0; e < 4; ++e) x[hp][e] = s[hp][e] * p.scale_log2;
          // tokens of this page each column may see: present slots, then the causal limit
          const int ca = min(vld[hp], lim0 - pg0 - hp * kPage);
          const int cb = min(vld[hp], lim1 - pg0 - hp * kPage);
          if (ca < kPage || cb < kPage) {
            if (r0 >= ca) x[hp][0] = -INFINITY;
            if (r0 >= cb) x[hp][1] = -INFINITY;
            if (r0 + 8 >= ca) x[hp][2] = -INFINITY;
            if (r0 + 8 >= cb) x[hp][3] = -INFINITY;
          }
        }
        // online softmax down each head column over the 32 tokens (log2 domain)
        float c0 = fmaxf(fmaxf(x[0][0], x[0][2]), fmaxf(x[1][0], x[1][2]));
        float c1 = fmaxf(fmaxf(x[0][1], x[0][3]), fmaxf(x[1][1], x[1][3]));
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          c0 = fmaxf(c0, __shfl_xor_sync(kFull, c0, o));
          c1 = fmaxf(c1, __shfl_xor_sync(kFull, c1, o));
        }
        const float mn0 = fmaxf(m0, c0), mn1 = fmaxf(m1, c1);
        // a column that has seen no token yet (causal rows of a split piece) keeps m =
        // -inf: subtract 0 instead, so its weights stay 0 rather than NaN
        const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = ptx::exp2_approx(m0 - ms0), al1 = ptx::exp2_approx(m1 - ms1);
        float pp[2][4];
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {
          pp[hp][0] = ptx::exp2_approx(x[hp][0] - ms0);
          pp[hp][1] = ptx::exp2_approx(x[hp][1] - ms1);
          pp[hp][2] = ptx::exp2_approx(x[hp][2] - ms0);
          pp[hp][3] = ptx::exp2_approx(x[hp][3] - ms1);
        }
        l0 = l0 * al0 + ((pp[0][0] + pp[0][2]) + (pp[1][0] + pp[1][2]));
        l1 = l1 * al1 + ((pp[0][1] + pp[0][3]) + (pp[1][1] + pp[1][3]));
        m0 = mn0;
        m1 = mn1;
        if (__any_sync(kFull, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
          for (int mt = 0; mt < kKS; ++mt) {
            acc[mt][0] *= al0;
            acc[mt][1] *= al1;
            acc[mt][2] *= al0;
            acc[mt][3] *= al1;
          }
        }
        // P^T as B operands (k = token, n = head) and the token masks of the V^T
        // fragments (tokens cq, cq+1 and cq+8, cq+9 of each page)
        uint32_t pb[2][2], vm_lo[2], vm_hi[2];
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {
          pb[hp][0] = ptx::movmatrix_trans(ptx::Mma<TM>::pack(pp[hp][0], pp[hp][1]));
          pb[hp][1] = ptx::movmatrix_trans(ptx::Mma<TM>::pack(pp[hp][2], pp[hp][3]));
          const int v = vld[hp];
          vm_lo[hp] = (cq < v ? 0x0000ffffu : 0u) | (cq + 1 < v ? 0xffff0000u : 0u);
          vm_hi[hp] = (cq + 8 < v ? 0x0000ffffu : 0u) | (cq + 9 < v ? 0xffff0000u : 0u);
        }
        // O^T += V^T * P^T over both pages. ldmatrix.x4.trans over (tokens 0-7 | 8-15) x
        // (chunk mt | mt+1), 16-bit elements = dim pairs: a lane gets dims 2*r0, 2*r0+1
        // of tokens cq, cq+1. After a byte permute the pairs are (tokens cq, cq+1) of
        // dim 2*r0 and of dim 2*r0+1, so row r0 of m-tile mt is dim 16mt + 2*r0 and row
        // r0+8 is the next dim.
        const uint32_t vpg[2] = {kb + voff, kb + 2 * L::kTileBytes + voff};
#pragma unroll
        for (int mt = 0; mt < kKS; mt += 2) {
          uint32_t y[2][4];
#pragma unroll
          for (int hp = 0; hp < 2; ++hp)
            ptx::ldsm_x4_trans(vpg[hp] + f8_tile_offset<D>(tok_k, mt + chunk_k), y[hp][0],
                               y[hp][1], y[hp][2], y[hp][3]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int hp = 0; hp < 2; ++hp) {
              uint32_t a[4];
              ptx::Mma<TM>::from_e4m3x4(ptx::prmt(y[hp][2 * h], 0u, 0x3120u), a[0], a[1]);
              ptx::Mma<TM>::from_e4m3x4(ptx::prmt(y[hp][2 * h + 1], 0u, 0x3120u), a[2], a[3]);
              a[0] &= vm_lo[hp];
              a[1] &= vm_lo[hp];
              a[2] &= vm_hi[hp];
              a[3] &= vm_hi[hp];
              ptx::Mma<TM>::run(acc[mt + h], a, pb[hp][0], pb[hp][1]);
            }
          }
        }
      } else if constexpr (kPPT == 2) {
        // ---- two 16-bit pages A, B (B may be absent at a portion's end: its slots are
        // then all stale and masked like the stale slots of a partial page)
        const int pg0 = (pt.p0 + i * kPPT) * kPage;
        const int vld[2] = {min(kPage, ctx - pg0),
                            (i * kPPT + 1 < npg) ? min(kPage, ctx - pg0 - kPage) : 0};
        const uint32_t kpg[2] = {kb, kb + 2 * L::kTileBytes};
        const uint32_t vpg[2] = {kb + L::kTileBytes, kb + 3 * L::kTileBytes};
        // S^T = K * Q^T for both pages: four independent accumulation chains (page x
        // parity of the k-step)
        float s[2][2][4] = {};
#pragma unroll
        for (int ks = 0; ks < kKS; ++ks) {
          const int chunk = (ks & 3) * 2 + chunk_k;
          const uint32_t off = (ks >> 2) * kBoxBytes + tok_k * 128 + ((chunk ^ (tok_k & 7)) << 4);
#pragma unroll
          for (int hp = 0; hp < 2; ++hp) {
            uint32_t a[4];
            ptx::ldsm_x4(kpg[hp] + off, a[0], a[1], a[2], a[3]);
            ptx::Mma<T>::run(s[hp][ks & 1], a, qf[ks][0], qf[ks][1]);
          }
        }
        float x[2][4];
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {
#pragma unroll
          for (int e = 0; e < 4; ++e) x[hp][e] = (s[hp][0][e] + s[hp][1][e]) * p.scale_log2;
          const int ca = min(vld[hp], lim0 - pg0 - hp * kPage);
          const int cb = min(vld[hp], lim1 - pg0 - hp * kPage);
          if (ca < kPage || cb < kPage) {
            if (r0 >= ca) x[hp][0] = -INFINITY;
            if (r0 >= cb) x[hp][1] = -INFINITY;
            if (r0 + 8 >= ca) x[hp][2] = -INFINITY;
            if (r0 + 8 >= cb) x[hp][3] = -INFINITY;
          }
        }
        float c0 = fmaxf(fmaxf(x[0][0], x[0][2]), fmaxf(x[1][0], x[1][2]));
        float c1 = fmaxf(fmaxf(x[0][1], x[0][3]), fmaxf(x[1][1], x[1][3]));
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          c0 = fmaxf(c0, __shfl_xor_sync(kFull, c0, o));
          c1 = fmaxf(c1, __shfl_xor_sync(kFull, c1, o));
        }
        const float mn0 = fmaxf(m0, c0), mn1 = fmaxf(m1, c1);
        const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = ptx::exp2_approx(m0 - ms0), al1 = ptx::exp2_approx(m1 - ms1);
        float pp[2][4];
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {
          pp[hp][0] = ptx::exp2_approx(x[hp][0] - ms0);
          pp[hp][1] = ptx::exp2_approx(x[hp][1] - ms1);
          pp[hp][2] = ptx::exp2_approx(x[hp][2] - ms0);
          pp[hp][3] = ptx::exp2_approx(x[hp][3] - ms1);
        }
        l0 = l0 * al0 + ((pp[0][0] + pp[0][2]) + (pp[1][0] + pp[1][2]));
        l1 = l1 * al1 + ((pp[0][1] + pp[0][3]) + (pp[1][1] + pp[1][3]));
        m0 = mn0;
        m1 = mn1;
        if (__any_sync(kFull, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
          for (int mt = 0; mt < kKS; ++mt) {
            acc[mt][0] *= al0;
            acc[mt][1] *= al1;
            acc[mt][2] *= al0;
            acc[mt][3] *= al1;
          }
        }
        uint32_t pb[2][2], vm_lo[2], vm_hi[2];
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {
          pb[hp][0] = ptx::movmatrix_trans(ptx::Mma<T>::pack(pp[hp][0], pp[hp][1]));
          pb[hp][1] = ptx::movmatrix_trans(ptx::Mma<T>::pack(pp[hp][2], pp[hp][3]));
          const int v = vld[hp];
          vm_lo[hp] = (cq < v ? 0x0000ffffu : 0u) | (cq + 1 < v ? 0xffff0000u : 0u);
          vm_hi[hp] = (cq + 8 < v ? 0x0000ffffu : 0u) | (cq + 9 < v ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int mt = 0; mt < kKS; ++mt) {
          const int chunk = (mt & 3) * 2 + chunk_v;
          const uint32_t off = (mt >> 2) * kBoxBytes + tok_v * 128 + ((chunk ^ (tok_v & 7)) << 4);
#pragma unroll
          for (int hp = 0; hp < 2; ++hp) {
            uint32_t a[4];
            ptx::ldsm_x4_trans(vpg[hp] + off, a[0], a[1], a[2], a[3]);
            a[0] &= vm_lo[hp];
            a[1] &= vm_lo[hp];
            a[2] &= vm_hi[hp];
            a[3] &= vm_hi[hp];
            ptx::Mma<T>::run(acc[mt], a, pb[hp][0], pb[hp][1]);
          }
        }
      } else {
        const int valid = min(kPage, ctx - (pt.p0 + i) * kPage);
        const uint32_t vb = kb + L::kTileBytes;

        // S^T = K * Q^T  (M = 16 tokens, N = 8 heads, K = D), as two independent chains
        // over the even and odd k-steps (half the dependent MMA latency per page)
        float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < kKS; ++ks) {
          const int chunk = (ks & 3) * 2 + chunk_k;
          const uint32_t addr =
              kb + (ks >> 2) * kBoxBytes + tok_k * 128 + ((chunk ^ (tok_k & 7)) << 4);
          uint32_t a[4];
          ptx::ldsm_x4(addr, a[0], a[1], a[2], a[3]);
          ptx::Mma<T>::run((ks & 1) ? s2 : s, a, qf[ks][0], qf[ks][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) s[e] += s2[e];
        float x0 = s[0] * p.scale_log2, x1 = s[1] * p.scale_log2;
        float x2 = s[2] * p.scale_log2, x3 = s[3] * p.scale_log2;
        // tokens of this page each column may see: present slots, then the causal limit
        const int ca = min(valid, lim0 - (pt.p0 + i) * kPage);
        const int cb = min(valid, lim1 - (pt.p0 + i) * kPage);
        if (ca < kPage || cb < kPage) {
          if (r0 >= ca) x0 = -INFINITY;
          if (r0 >= cb) x1 = -INFINITY;
          if (r0 + 8 >= ca) x2 = -INFINITY;
          if (r0 + 8 >= cb) x3 = -INFINITY;
        }
        // online softmax down each head column (log2 domain)
        float c0 = fmaxf(x0, x2), c1 = fmaxf(x1, x3);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          c0 = fmaxf(c0, __shfl_xor_sync(kFull, c0, o));
          c1 = fmaxf(c1, __shfl_xor_sync(kFull, c1, o));
        }
        const float mn0 = fmaxf(m0, c0), mn1 = fmaxf(m1, c1);
        // a column that has seen no token yet keeps m = -inf (see the fp8 path)
        const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = ptx::exp2_approx(m0 - ms0), al1 = ptx::exp2_approx(m1 - ms1);
        const float p0 = ptx::exp2_approx(x0 - ms0), p1 = ptx::exp2_approx(x1 - ms1);
        const float p2 = ptx::exp2_approx(x2 - ms0), p3 = ptx::exp2_approx(x3 - ms1);
        l0 = l0 * al0 + (p0 + p2);
        l1 = l1 * al1 + (p1 + p3);
        m0 = mn0;
        m1 = mn1;
        if (__any_sync(kFull, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
          for (int mt = 0; mt < kKS; ++mt) {
            acc[mt][0] *= al0;
            acc[mt][1] *= al1;
            acc[mt][2] *= al0;
            acc[mt][3] *= al1;
          }
        }
        // P^T as the B operand (k = token, n = head)
        const uint32_t pb0 = ptx::movmatrix_trans(ptx::Mma<T>::pack(p0, p1));
        const uint32_t pb1 = ptx::movmatrix_trans(ptx::Mma<T>::pack(p2, p3));
        // token masks for the V^T fragments (tokens cq, cq+1 and cq+8, cq+9)
        uint32_t vm_lo = 0xffffffffu, vm_hi = 0xffffffffu;
        if (valid < kPage) {
          vm_lo = (cq < valid ? 0x0000ffffu : 0u) | (cq + 1 < valid ? 0xffff0000u : 0u);
          vm_hi = (cq + 8 < valid ? 0x0000ffffu : 0u) | (cq + 9 < valid ? 0xffff0000u : 0u);
        }
        // O^T += V^T * P^T  (M = D in 16-row tiles, N = 8 heads, K = 16 tokens)
#pragma unroll
        for (int mt = 0; mt < kKS; ++mt) {
          const int chunk = (mt & 3) * 2 + chunk_v;
          const uint32_t addr =
              vb + (mt >> 2) * kBoxBytes + tok_v * 128 + ((chunk ^ (tok_v & 7)) << 4);
          uint32_t a[4];
          ptx::ldsm_x4_trans(addr, a[0], a[1], a[2], a[3]);
          a[0] &= vm_lo;
          a[1] &= vm_lo;
          a[2] &= vm_hi;
          a[3] &= vm_hi;
          ptx::Mma<T>::run(acc[mt], a, pb0, pb1);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[stage]);
    }
    k += nfill;
    // the previous grid on the stream has completed from here on (returns at once after
    // the first portion)
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- this warp's state -> shared memory
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, o);
      l1 += __shfl_xor_sync(kFull, l1, o);
    }
    // rows r0 and r0 + 8 of m-tile mt are dims 16mt + r0 and + 8 (16-bit caches) or
    // 16mt + 2*r0 and + 1 (fp8 caches)
    constexpr int kRowStep = F8 ? 1 : 8;
#pragma unroll
    for (int mt = 0; mt < kKS; ++mt) {
      const int d = mt * 16 + (F8 ? 2 * r0 : r0);
      mw[cq * L::kMergeStride + d] = acc[mt][0];
      mw[(cq + 1) * L::kMergeStride + d] = acc[mt][1];
      mw[cq * L::kMergeStride + d + kRowStep] = acc[mt][2];
      mw[(cq + 1) * L::kMergeStride + d + kRowStep] = acc[mt][3];
    }
    if (lane < 4) {
      mw[8 * L::kMergeStride + cq] = m0;
      mw[8 * L::kMergeStride + cq + 1] = m1;
      mw[8 * L::kMergeStride + 8 + cq] = l0;
      mw[8 * L::kMergeStride + 8 + cq + 1] = l1;
    }
    ptx::named_barrier_sync(1, L::kCW * 32);

    // ---- merge the warps of each head subtile; write final rows or this CTA's split slot
    const bool whole = (pt.p0 == 0 && pt.p1 == pt.np);
    const int slot = piece_slot(pt.seg_start, g_lo);
    const int64_t slot_row = (int64_t(blockIdx.x) * 2 + slot) * p.group;
    constexpr int kChunks = D / 8;
    for (int idx = tid; idx < nrows * kChunks; idx += L::kCW * 32) {
      const int j = idx / kChunks;
      const int dc = idx - j * kChunks;
      const int hs = j >> 3, n = j & 7;
      float mx = -INFINITY;
#pragma unroll
      for (int r = 0; r < kWP; ++r)
        mx = fmaxf(mx, merge[(hs + r * NHT) * L::kMergeWarpFloats + 8 * L::kMergeStride + n]);
      float lsum = 0.f, o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int r = 0; r < kWP; ++r) {
        const float* w = merge + (hs + r * NHT) * L::kMergeWarpFloats;
        const float wm = w[8 * L::kMergeStride + n];
        if (wm == -INFINITY) continue;  // this warp saw no page of the portion
        const float f = ptx::exp2_approx(wm - mx);
        lsum += w[8 * L::kMergeStride + 8 + n] * f;
        const float4 a = *reinterpret_cast<const float4*>(w + n * L::kMergeStride + dc * 8);
        const float4 b = *reinterpret_cast<const float4*>(w + n * L::kMergeStride + dc * 8 + 4);
        o[0] += a.x * f; o[1] += a.y * f; o[2] += a.z * f; o[3] += a.w * f;
        o[4] += b.x * f; o[5] += b.y * f; o[6] += b.z * f; o[7] += b.w * f;
      }
      // lsum = 0 only for a causal row that saw no token of a split piece: its partial
      // is O = 0, L = -inf, which the merges skip
      const float inv = lsum > 0.f ? p.v_scale / lsum : 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] *= inv;
      const float lse_nat = lsum > 0.f ? (mx + log2f(lsum)) * kLn2 : -INFINITY;
      if (whole) {
        const RowIndex ri =
            seg_row(pt.b, kvh, rbase + j, p.heads_per_kv, p.seq_len_q, p.num_q_heads);
        *reinterpret_cast<uint4*>(outg + ri.out_row * D + dc * 8) = pack8<T>(o);
        if (dc == 0 && p.lse != nullptr) p.lse[ri.lse] = lse_nat;
      } else {
        float* po = p.part_out + (slot_row + j) * D + dc * 8;
        __stcg(reinterpret_cast<float4*>(po), make_float4(o[0], o[1], o[2], o[3]));
        __stcg(reinterpret_cast<float4*>(po + 4), make_float4(o[4], o[5], o[6], o[7]));
        if (dc == 0) __stcg(p.part_lse + slot_row + j, lse_nat);
      }
    }

    if (!whole) {
      // ---- split piece. Few pieces: count arrivals and let the last piece merge them
      // here. Many pieces: the split-merge kernel that follows merges them in parallel.
      const int64_t c0 = pt.seg_start / p.tiles_per_cta;
      const int64_t c1 = (pt.seg_start + pt.np - 1) / p.tiles_per_cta;
      const int pieces = int(c1 - c0 + 1);
      if (pieces <= p.heavy_min) {
        __threadfence();
        ptx::named_barrier_sync(1, L::kCW * 32);
        int32_t* counter = p.counters + int64_t(pt.b) * p.segs_per_seq + pt.seg;
        if (tid == 0) {
          const int prev = aborted ? -1 : atomicAdd(counter, 1);
          flags[1] = (prev == pieces - 1) ? 1 : 0;
        }
        ptx::named_barrier_sync(1, L::kCW * 32);
        if (flags[1]) {
          __threadfence();
          for (int idx = tid; idx < nrows * kChunks; idx += L::kCW * 32) {
            const int j = idx / kChunks;
            const int dc = idx - j * kChunks;
            // online merge over the pieces, four at a time with independent loads
            float mx = -INFINITY, den = 0.f, o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int64_t cb = c0; cb <= c1; cb += 4) {
              float ls[4];
              float4 va[4], vb[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int64_t c = cb + u;
                ls[u] = -INFINITY;
                va[u] = vb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (c <= c1) {
                  const int sl = (c == c0 && pt.seg_start > c * p.tiles_per_cta) ? 1 : 0;
                  const int64_t rowi = (c * 2 + sl) * p.group + j;
                  ls[u] = __ldcg(p.part_lse + rowi);
                  va[u] = __ldcg(reinterpret_cast<const float4*>(p.part_out + rowi * D + dc * 8));
                  vb[u] = __ldcg(reinterpret_cast<const float4*>(p.part_out + rowi * D + dc * 8 + 4));
                }
              }
              const float nm = fmaxf(fmaxf(mx, fmaxf(ls[0], ls[1])), fmaxf(ls[2], ls[3]));
              if (nm == -INFINITY) continue;
              const float f = ptx::exp2_approx((mx - nm) * kLog2e);
              den *= f;
#pragma unroll
              for (int e = 0; e < 8; ++e) o[e] *= f;
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float wgt = ptx::exp2_approx((ls[u] - nm) * kLog2e);
                den += wgt;
                o[0] += wgt * va[u].x; o[1] += wgt * va[u].y; o[2] += wgt * va[u].z; o[3] += wgt * va[u].w;
                o[4] += wgt * vb[u].x; o[5] += wgt * vb[u].y; o[6] += wgt * vb[u].z; o[7] += wgt * vb[u].w;
              }
              mx = nm;
            }
            const float inv = 1.f / den;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] *= inv;
            const RowIndex ri =
                seg_row(pt.b, kvh, rbase + j, p.heads_per_kv, p.seq_len_q, p.num_q_heads);
            *reinterpret_cast<uint4*>(outg + ri.out_row * D + dc * 8) = pack8<T>(o);
            if (dc == 0 && p.lse != nullptr) p.lse[ri.lse] = mx + logf(den);
          }
          if (tid == 0) atomicExch(counter, 0);
        }
      }
    }
    // the merge area is rewritten by the next portion
    ptx::named_barrier_sync(1, L::kCW * 32);
  }
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

// Map over a paged cache [num_blocks, P, Hkv, D] (16-bit), 128-byte swizzle: dims
// (d mod 64, slot, d / 64, kvh, block) with box (64, P, D/64, 1, 1), so one copy lands
// a (block, kvh) tile as D/64 swizzled [P][64] sub-tiles.
bool encode_cache_map(CUtensorMap* map, const void* base, int64_t num_blocks, int page, int hkv,
                      int d, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[5] = {64, cuuint64_t(page), cuuint64_t(d / 64), cuuint64_t(hkv),
                              cuuint64_t(num_blocks)};
  const cuuint64_t strides[4] = {cuuint64_t(hkv) * d * 2, 128, cuuint64_t(d) * 2,
                                 cuuint64_t(page) * hkv * d * 2};
  const cuuint32_t box[5] = {64, cuuint32_t(page), cuuint32_t(d / 64), 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map over an E4M3 cache [num_blocks, P, Hkv, D] bytes: dims (d, kvh, slot, block),
// box (D, 1, P, 1), so one copy lands a (block, kvh) tile as P rows of D bytes, with
// 128-byte (D = 128) or 64-byte (D = 64) swizzle. L2 promotion stays at 128 bytes: a
// row is at most 128 bytes, and a 256-byte promotion fetched the next KV head's row
// too, which only other CTAs use, often after it has left L2 (varlen batch: 1.43x the
// algorithmic DRAM bytes).
bool encode_cache_map_f8(CUtensorMap* map, const void* base, int64_t num_blocks, int page,
                         int hkv, int d) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {cuuint64_t(d), cuuint64_t(hkv), cuuint64_t(page),
                              cuuint64_t(num_blocks)};
  const cuuint64_t strides[3] = {cuuint64_t(d), cuuint64_t(hkv) * d, cuuint64_t(page) * hkv * d};
  const cuuint32_t box[4] = {cuuint32_t(d), 1, cuuint32_t(page), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One map over both E4M3 caches: dims (d, kvh, slot, block, tensor) where the tensor
// dimension (extent 2) steps from the lower of the two cache addresses to the other, so
// one copy of box (D, 1, P, 1, 2) lands a page's two tiles back to back. Only
// coordinates 0 and 1 of that dimension are ever read, i.e. the two caches themselves.
bool encode_cache_pair_f8(CUtensorMap* map, const void* k, const void* v, int64_t num_blocks,
                          int page, int hkv, int d, int32_t* order) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const uintptr_t ka = reinterpret_cast<uintptr_t>(k), va = reinterpret_cast<uintptr_t>(v);
  const uintptr_t lo = ka < va ? ka : va, gap = ka < va ? va - ka : ka - va;
  const uint64_t cache_bytes = uint64_t(num_blocks) * page * hkv * d;
  if (gap < cache_bytes || gap % 16 != 0 || gap >= (uint64_t(1) << 40)) return false;
  const cuuint64_t dims[5] = {cuuint64_t(d), cuuint64_t(hkv), cuuint64_t(page),
                              cuuint64_t(num_blocks), 2};
  const cuuint64_t strides[4] = {cuuint64_t(d), cuuint64_t(hkv) * d,
                                 cuuint64_t(page) * hkv * d, cuuint64_t(gap)};
  const cuuint32_t box[5] = {cuuint32_t(d), 1, cuuint32_t(page), 1, 2};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  if (fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, reinterpret_cast<void*>(lo), dims, strides, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  *order = ka < va ? 1 : 2;
  return true;
}

template <int D, typename T, int NHT, bool F8>
int launch_one(const CUtensorMap& tk, const CUtensorMap& tv, const GqaParams& prm, int grid,
               cudaStream_t stream) {
  auto kern = gqa_decode_kernel<D, T, NHT, F8>;
  using L = Layout<D, F8, NHT>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    L::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(Roles<NHT>::kThreads);
  cfg.dynamicSmemBytes = L::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tk, tv, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, typename T, bool F8>
int launch_d(int nht, const CUtensorMap& tk, const CUtensorMap& tv, const GqaParams& prm, int grid,
             cudaStream_t s) {
  switch (nht) {
    case 1: return launch_one<D, T, 1, F8>(tk, tv, prm, grid, s);
    case 2: return launch_one<D, T, 2, F8>(tk, tv, prm, grid, s);
    default: return launch_one<D, T, 4, F8>(tk, tv, prm, grid, s);
  }
}

template <bool F8>
int launch_dt(int d, bool bf16, int nht, const CUtensorMap& tk, const CUtensorMap& tv,
              const GqaParams& prm, int grid, cudaStream_t s) {
  if (d == 64)
    return bf16 ? launch_d<64, __nv_bfloat16, F8>(nht, tk, tv, prm, grid, s)
                : launch_d<64, __half, F8>(nht, tk, tv, prm, grid, s);
  return bf16 ? launch_d<128, __nv_bfloat16, F8>(nht, tk, tv, prm, grid, s)
              : launch_d<128, __half, F8>(nht, tk, tv, prm, grid, s);
}

}  // namespace

bool gqa_supported(const pda_problem& p, std::string* why) {
  if (p.head_dim_qk != p.head_dim_v || (p.head_dim_qk != 64 && p.head_dim_qk != 128)) {
    *why = "GQA decode supports head_dim_qk == head_dim_v in {64, 128}";
    return false;
  }
  if (p.page_size != kPage) {
    *why = "GQA decode supports page_size 16";
    return false;
  }
  const int g = p.num_q_heads / p.num_kv_heads;
  const int sq = p.seq_len_q > 1 ? p.seq_len_q : 1;
  if (int64_t(g) * sq > kMaxRowsPerKvHead) {
    *why = "GQA decode supports up to " + std::to_string(kMaxRowsPerKvHead) +
           " query rows (seq_len_q * Hq / Hkv) per KV head";
    return false;
  }
  if (int64_t(p.num_kv_heads) * ((int64_t(g) * sq + 31) / 32) > INT32_MAX) {
    *why = "Hkv times the row chunks per KV head must fit in int32";
    return false;
  }
  if (p.num_blocks > INT32_MAX) {
    *why = "num_blocks must fit in int32 (block-table entries are int32)";
    return false;
  }
  return true;
}

int gqa_ctas_per_sm(const pda_problem& p) {
  // the launcher's head-subtile count of a segment (rows in chunks of at most 32)
  const int64_t rows = int64_t(p.seq_len_q > 1 ? p.seq_len_q : 1) * (p.num_q_heads / p.num_kv_heads);
  const int64_t group = (rows + (rows + 31) / 32 - 1) / ((rows + 31) / 32);
  const bool four = (group + 7) / 8 > 2;
  return four ? Roles<4>::kCtasPerSm : kCtasPerSm;
}

int launch_gqa_decode(const Plan& plan, const GqaArgs& a, const Workspace& ws, void* stream) {
  const pda_problem& pr = plan.prob;
  const bool bf16 = pr.dtype == PDA_BF16;
  const bool f8 = pr.kv_format == PDA_KV_FP8_E4M3;
  CUtensorMap m[2];
  int32_t kv_pair = 0;
  const bool maps_ok = plan.map_cache.get(a.k_cache, a.v_cache, m, &kv_pair,
                                          [&](CUtensorMap* t, int32_t* order) {
    const bool ok =
        f8 ? encode_cache_map_f8(&t[0], a.k_cache, pr.num_blocks, pr.page_size,
                                 pr.num_kv_heads, pr.head_dim_qk) &&
                 encode_cache_map_f8(&t[1], a.v_cache, pr.num_blocks, pr.page_size,
                                     pr.num_kv_heads, pr.head_dim_v)
           : encode_cache_map(&t[0], a.k_cache, pr.num_blocks, pr.page_size, pr.num_kv_heads,
                              pr.head_dim_qk, bf16) &&
                 encode_cache_map(&t[1], a.v_cache, pr.num_blocks, pr.page_size,
                                  pr.num_kv_heads, pr.head_dim_v, bf16);
    // fp8: when one map can span both caches, a page's K and V come in one copy (the
    // producer's copy issue, not HBM, bounds the fp8 kernel)
    if (ok && f8) {
      CUtensorMap pair;
      if (encode_cache_pair_f8(&pair, a.k_cache, a.v_cache, pr.num_blocks, pr.page_size,
                               pr.num_kv_heads, pr.head_dim_qk, order))
        t[0] = pair;
    }
    return ok;
  });
  if (!maps_ok) return -1;
  const CUtensorMap& tk = m[0];
  const CUtensorMap& tv = m[1];
  GqaParams prm{};
  prm.kv_pair = kv_pair;
  prm.q = a.q;
  prm.out = a.out;
  prm.lse = a.lse;
  prm.block_tables = a.block_tables;
  prm.context_lens = a.context_lens;
  prm.batch = pr.batch;
  prm.num_q_heads = pr.num_q_heads;
  prm.num_kv_heads = pr.num_kv_heads;
  prm.group = plan.group;
  prm.heads_per_kv = plan.heads_per_seg;
  prm.row_chunks = plan.row_chunks;
  prm.segs_per_seq = plan.segs_per_seq;
  prm.seq_len_q = plan.seq_len_q;
  prm.max_blocks = pr.max_blocks_per_seq;
  prm.num_blocks = pr.num_blocks;
  prm.scale_log2 = a.scale * a.k_scale * kLog2e;
  prm.v_scale = a.v_scale;
  prm.total_tiles = plan.total_tiles;
  prm.tiles_per_cta = plan.tiles_per_cta;
  prm.heavy_min = plan.heavy_min_pieces;
  prm.err = ws.err;
  prm.counters = ws.counters;
  prm.part_lse = ws.part_lse;
  prm.part_out = ws.part_out;
  const int nht = plan.head_subtiles <= 1 ? 1 : (plan.head_subtiles <= 2 ? 2 : 4);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int e = f8 ? launch_dt<true>(pr.head_dim_qk, bf16, nht, tk, tv, prm, plan.num_ctas, s)
                  : launch_dt<false>(pr.head_dim_qk, bf16, nht, tk, tv, prm, plan.num_ctas, s);
  if (e != 0) return e;
  return launch_split_merge(plan, ws, a.out, a.lse, stream);
}

}  // namespace pda
