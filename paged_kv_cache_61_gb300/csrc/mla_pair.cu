// Absorbed-MLA paged decode for head groups of 128 query heads, one group per pair of
// CTAs (a two-CTA thread-block cluster on two SMs).
//
// What it computes is what mla_decode.cu computes ("From MHA to MLA", section 6;
// FlashMLA-ETAP README, "Usage"): every query head attends to one shared 576-wide
// record per token (512 latent + 64 rope); score = scale * <q_h, rec_j>, value =
// rec_j[:512]; output [B, Hq, 512] and the fp32 LSE.
//
// How. With 128 heads the output accumulator of a head group (128 x 512 fp32) fills a
// whole SM's tensor memory, and q for 128 heads (144 KB) most of its shared memory. The
// group is therefore split over two SMs by record dimension:
//  * CTA r of the pair holds latent dims [256r, 256r+256) and rope dims
//    [512+32r, 512+32r+32) of every page (36 KB per 64-token page) in a four-stage
//    page ring, and the same dims of q for the 128 heads in tensor memory (the score
//    MMA's A operand). Each latent byte is read from HBM once per head group.
//  * Scores with the heads on the MMA's M axis: S_r[128 x 64 tokens] = q_r * K_r^T
//    (M=128, N=64, K=288: 18 tcgen05.mma). On this part an MMA's issue cost is set by
//    N (a floor of ~46 cycles up to N=64), so 128 heads on M cost what 64 would.
//  * The two partial score tiles are swapped through distributed shared memory: each
//    CTA stages its tile in its own shared memory and one bulk copy per warp moves it
//    into the peer's buffer, counted on the peer's mbarrier. Both CTAs then hold
//    S = S_0 + S_1 bit for bit (fp32 addition commutes) and run the same online softmax,
//    one thread per head with the running maximum and sums in registers, so they take
//    the same rescaling decisions without exchanging them.
//  * P (16-bit) is written to tensor memory and is the A operand of the PV MMA:
//    O_r[128 x 256] += P[128 x 64] * V_r[64 x 256] (M=128, N=256, 4 MMAs), V_r read in
//    place from the page's latent sub-tiles. CTA r owns output dims [256r, 256r+256).
//  * Split pieces and their merge follow the other decode kernels; each CTA writes and
//    merges its half of the output dims.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "pda_internal.h"
#include "ptx.cuh"
#include "ptx_cluster.cuh"
#include "tile_walk.cuh"

namespace pda {

namespace {

constexpr int kPage = 64;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kHeads = 128;                 // query heads per pair
constexpr int kHalfDv = kDv / 2;            // output / latent dims per CTA
constexpr int kLatSubs = kHalfDv / 64;      // 128-byte-swizzled 64-dim sub-tiles per CTA
constexpr int kRopeHalf = 32;               // rope dims per CTA (64-byte swizzle)
constexpr int kStages = 4;
constexpr int kLatSubBytes = kPage * 128;                          // [64 tokens][64 dims]
constexpr int kRopeBytes = kPage * kRopeHalf * 2;                  // [64 tokens][32 dims]
constexpr int kStageBytes = kLatSubs * kLatSubBytes + kRopeBytes;  // 36 KB
constexpr int kXBytes = kHeads * kPage * 4;                        // one fp32 score tile
constexpr int kSoftmaxWarps = 4;                                   // one thread per head
constexpr int kThreads = 64 + 32 * kSoftmaxWarps;
constexpr int kTmemCols = 512;
// tensor-memory columns (32-bit): q_r as 16-bit pairs, S, P as 16-bit pairs, O_r
constexpr int kColQ = 0;     // 144 columns: latent dims in [0, 128), rope dims in [128, 144)
constexpr int kColP = 160;   // 32 columns
constexpr int kColS = 192;   // 64 columns
constexpr int kColO = 256;   // 256 columns
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;   // lazy-max slack (log2 units)

struct Layout {
  static constexpr int kKV = 0;
  static constexpr int kX = kKV + kStages * kStageBytes;   // the peer's partial scores land here
  static constexpr int kStg = kX + kXBytes;                 // this CTA's, on their way out
  static constexpr int kBar = kStg + kXBytes;
  static constexpr int kBarCount = 24;
  static constexpr int kSmem = 1024 + kBar + kBarCount * 8 + 64;
  static_assert(kStageBytes % 1024 == 0 && kX % 1024 == 0, "swizzled tiles stay 1024-byte aligned");
  static_assert(kSmem <= 227 * 1024, "fits one SM's shared memory");
};

struct PairParams {
  const void* q;
  void* out;
  float* lse;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t batch, num_q_heads, groups, max_blocks;
  int64_t num_blocks;
  float scale_log2;
  int64_t total_tiles, tiles_per_cta;
  int32_t heavy_min;
  int32_t* err;
  int32_t* counters;   // [B][groups][2]: one per output half
  float* part_lse;
  float* part_out;
};

__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                             int32_t* err) {
  if (wait_phase(bar, parity, abort)) return true;
  *abort = 1;
  atomicOr(err, 2);
  return false;
}

// Bounded wait on a phase completed by the peer CTA (acquire at cluster scope).
__device__ __forceinline__ bool bounded_wait_cluster(uint64_t* bar, uint32_t parity,
                                                     volatile int* abort, int32_t* err) {
  if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort || ptx::globaltimer() - t0 > ptx::kWaitLimitNs) break;
  }
  *abort = 1;
  atomicOr(err, 2);
  return false;
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return ptx::Mma<T>::pack(lo, hi);
}

// Sum of the two 16-bit values packed by pack2 (the weights the PV MMA really uses).
template <typename T>
__device__ __forceinline__ float sum2(uint32_t w);
template <>
__device__ __forceinline__ float sum2<__nv_bfloat16>(uint32_t w) {
  return __uint_as_float(w << 16) + __uint_as_float(w & 0xffff0000u);
}
template <>
__device__ __forceinline__ float sum2<__half>(uint32_t w) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
  return f.x + f.y;
}

template <typename T>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_pair_kernel(const __grid_constant__ CUtensorMap tm_kv_lat,
                    const __grid_constant__ CUtensorMap tm_kv_rope, const PairParams p) {
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ uint8_t smem_raw[];
  // the same offset in both CTAs of the pair (same kernel, same static layout)
  uint8_t* base = align1024(smem_raw);
  uint8_t* kv = base + Layout::kKV;
  uint8_t* xbuf = base + Layout::kX;
  uint8_t* stg_out = base + Layout::kStg;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + Layout::kBar);
  uint64_t* kv_full = bars + 0;    // [4]
  uint64_t* kv_empty = bars + 4;   // [4]
  uint64_t* q_full = bars + 8;     // q of the next piece is in tensor memory
  uint64_t* s_full = bars + 9;     // S written by the score MMA
  uint64_t* s_free = bars + 10;    // S read by the softmax warps
  uint64_t* p_full = bars + 11;    // P written
  uint64_t* pv_done = bars + 12;   // PV of a page completed
  uint64_t* x_full = bars + 13;    // the peer's partial scores are in xbuf
  uint64_t* x_free = bars + 14;    // the peer has read this CTA's partial scores
  // [0] abort, [1] last piece to arrive
  volatile int* flags = reinterpret_cast<volatile int*>(bars + 16);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int64_t pair = blockIdx.x >> 1;
  const int64_t g_lo = pair * p.tiles_per_cta;
  const int64_t g_hi = min(p.total_tiles, g_lo + p.tiles_per_cta);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // both CTAs of a pair share the range, so they leave together
  if (g_lo >= g_hi) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&kv_full[s], 1);
      ptx::mbar_init(&kv_empty[s], 1);
    }
    ptx::mbar_init(q_full, kSoftmaxWarps);
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(s_free, kSoftmaxWarps);
    ptx::mbar_init(p_full, kSoftmaxWarps);
    ptx::mbar_init(pv_done, 1);
    ptx::mbar_init(x_full, 1);
    ptx::mbar_init(x_free, kSoftmaxWarps);
    for (int i = 0; i < 8; ++i) flags[i] = 0;
    ptx::fence_mbarrier_init();
    // the first page's partial scores from the peer (its copies may land first)
    ptx::mbar_arrive_expect_tx(x_full, kXBytes);
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, kTmemCols);
  ptx::tc_fence_before();
  ptx::cluster_sync();   // both CTAs' barriers exist before any access from the peer
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const WalkSpec spec{p.context_lens, p.batch, p.groups, kPage};
  Walker walk;
  walker_init(walk, spec, g_lo, lane);

  if (warp == 0) {
    // ============================== TMA producer ==============================
    if (lane == 0) {
      ptx::prefetch_tensormap(&tm_kv_lat);
      ptx::prefetch_tensormap(&tm_kv_rope);
    }
    const uint64_t pol_stream = ptx::policy_evict_first();
    int t = 0, st = 0;
    uint32_t ph = 0;
    bool ok = true;
    while (ok && walk.g < g_hi) {
      const Portion pt = walker_next(walk, spec, g_hi);
      const int32_t* row = p.block_tables + int64_t(pt.b) * p.max_blocks;
      for (int base_pg = pt.p0; ok && base_pg < pt.p1; base_pg += 32) {
        const int32_t ids = (base_pg + lane < pt.p1) ? __ldg(row + base_pg + lane) : 0;
        const int n = min(32, pt.p1 - base_pg);
        for (int j = 0; j < n; ++j) {
          const int32_t phys = __shfl_sync(kFullMask, ids, j);
          int good = 1;
          if (lane == 0) {
            if (!bounded_wait(&kv_empty[st], ph ^ 1, flags, p.err)) {
              good = 0;
            } else {
              if (phys < 0 || int64_t(phys) >= p.num_blocks) atomicOr(p.err, 1);
              uint8_t* dst = kv + st * kStageBytes;
              ptx::mbar_arrive_expect_tx(&kv_full[st], kStageBytes);
              ptx::tma_load_4d(dst, &tm_kv_lat, &kv_full[st], 0, 0, kLatSubs * int32_t(rank), phys,
                               pol_stream);
              ptx::tma_load_3d(dst + kLatSubs * kLatSubBytes, &tm_kv_rope, &kv_full[st],
                               kDv + kRopeHalf * int32_t(rank), 0, phys, pol_stream);
            }
          }
          ok = __shfl_sync(kFullMask, good, 0) != 0;
          if (!ok) break;
          ++t;
          if (++st == kStages) {
            st = 0;
            ph ^= 1;
          }
        }
      }
    }
    // Leave no copy in flight: the last fill of each stage (bounded).
    if (lane == 0) {
      for (int k = 1; k <= kStages && t - k >= 0; ++k) {
        const int tt = t - k;
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(&kv_full[tt % kStages], (tt / kStages) & 1) &&
               ptx::globaltimer() - t0 < ptx::kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ============================== MMA issuer ==============================
    // One thread issues whichever MMA group is ready: the scores of the next page
    // (its stage, q and the S columns are ready) or the PV of the oldest page whose P
    // is in tensor memory.
    constexpr uint32_t kIdQK = ptx::umma_idesc_f16(128, 64, 0, 0, kBf16);
    constexpr uint32_t kIdPV = ptx::umma_idesc_f16(128, 256, 0, 1, kBf16);
    const uint32_t kv_s = ptx::smem_addr(kv);
    if (lane == 0) {
      int u = 0, i = 0, npg = 0;
      int t_qk = 0, t_pv = 0, st_qk = 0, st_pv = 0;
      uint32_t ph_qk = 0;
      bool have = false, need_q = false, qk_done = false;
      uint32_t first_bits = 0;   // bit (t & 31): page t is the first of its piece
      uint64_t last_progress = ptx::globaltimer();
      while (true) {
        bool progress = false;
        if (!qk_done && (!have || i == npg)) {
          if (walk.g < g_hi) {
            const Portion pt = walker_next(walk, spec, g_hi);
            npg = pt.p1 - pt.p0;
            i = 0;
            have = true;
            need_q = true;
          } else {
            qk_done = true;
          }
        }
        if (!qk_done && i < npg) {
          const bool ready = (!need_q || ptx::mbar_try_wait(q_full, u & 1)) &&
                             ptx::mbar_try_wait(&kv_full[st_qk], ph_qk) &&
                             (t_qk == 0 || ptx::mbar_try_wait(s_free, (t_qk - 1) & 1));
          if (ready) {
            if (need_q) ++u;
            need_q = false;
            ptx::tc_fence_after();
            const uint32_t stg = kv_s + st_qk * kStageBytes;
#pragma unroll
            for (int kb = 0; kb < kLatSubs; ++kb) {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint64_t b = ptx::umma_desc_sw128(stg + kb * kLatSubBytes + ks * 32, 16, 1024);
                ptx::umma_f16_ts(tmem + kColS, tmem + kColQ + kb * 32 + ks * 8, b, kIdQK,
                                 (kb | ks) != 0);
              }
            }
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
              const uint64_t b = ptx::umma_desc_sw64(stg + kLatSubs * kLatSubBytes + ks * 32, 16, 512);
              ptx::umma_f16_ts(tmem + kColS, tmem + kColQ + 128 + ks * 8, b, kIdQK, true);
            }
            ptx::umma_commit(s_full);
            first_bits = (first_bits & ~(1u << (t_qk & 31))) | (uint32_t(i == 0) << (t_qk & 31));
            ++t_qk;
            ++i;
            if (++st_qk == kStages) {
              st_qk = 0;
              ph_qk ^= 1;
            }
            progress = true;
          }
        }
        if (t_pv < t_qk && ptx::mbar_try_wait(p_full, t_pv & 1)) {
          ptx::tc_fence_after();
          const bool first = (first_bits >> (t_pv & 31)) & 1u;
          const uint32_t stg = kv_s + st_pv * kStageBytes;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            // V_r: 16 tokens x 256 dims, dims contiguous in four 64-dim sub-tiles
            const uint64_t b = ptx::umma_desc_sw128(stg + ks * 2048, kLatSubBytes, 1024);
            ptx::umma_f16_ts(tmem + kColO, tmem + kColP + ks * 8, b, kIdPV, !(first && ks == 0));
          }
          ptx::umma_commit(&kv_empty[st_pv]);
          ptx::umma_commit(pv_done);
          ++t_pv;
          if (++st_pv == kStages) st_pv = 0;
          progress = true;
        }
        if (qk_done && t_pv == t_qk) break;
        if (progress) {
          last_progress = ptx::globaltimer();
        } else if (flags[0] || ptx::globaltimer() - last_progress > ptx::kWaitLimitNs) {
          flags[0] = 1;
          atomicOr(p.err, 2);
          break;
        }
      }
      // Wait (bounded) for the last MMAs before tensor memory is released.
      if (t_pv > 0) {
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(pv_done, (t_pv - 1) & 1) &&
               ptx::globaltimer() - t0 < ptx::kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // ============================== softmax / epilogue warps ==============================
    const int sp = warp & 3;                 // TMEM sub-partition of this warp
    const int h = 32 * sp + lane;            // head of the group = TMEM lane
    const int ctid = threadIdx.x - 64;       // 0 .. 127
    const uint32_t t_lane = tmem + (uint32_t(32 * sp) << 16);
    const uint32_t sw = uint32_t(h & 7);     // 16-byte chunk swizzle of the score rows
    const uint32_t row_off = uint32_t(h) * (kPage * 4);
    const uint32_t x_own = ptx::smem_addr(xbuf) + row_off;
    const uint32_t s_own = ptx::smem_addr(stg_out) + row_off;
    const uint32_t blk = uint32_t(32 * sp) * (kPage * 4);   // this warp's 32 rows
    const uint32_t x_peer_blk = ptx::mapa_shared(ptx::smem_addr(xbuf) + blk, rank ^ 1);
    const uint32_t xfull_peer = ptx::mapa_shared(ptx::smem_addr(x_full), rank ^ 1);
    const uint32_t xfree_peer = ptx::mapa_shared(ptx::smem_addr(x_free), rank ^ 1);
    const T* qg = static_cast<const T*>(p.q);
    T* outg = static_cast<T*>(p.out);
    bool aborted = false;
    float sown[kPage];   // this CTA's partial scores of the page being exchanged

    // q_r of this head for the piece into tensor memory: latent dims [256r, 256r+256)
    // in columns [0, 128), rope dims [512+32r, 512+32r+32) in [128, 144).
    auto load_q = [&](const Portion& pq) {
      const T* qrow = qg + (int64_t(pq.b) * p.num_q_heads + int64_t(pq.seg) * kHeads + h) * kDqk;
#pragma unroll
      for (int c0 = 0; c0 < 9; c0 += 3) {
        uint4 v[12];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int c = c0 + k;
          const T* src = c < 8 ? qrow + int(rank) * kHalfDv + 32 * c : qrow + kDv + int(rank) * kRopeHalf;
#pragma unroll
          for (int e = 0; e < 4; ++e) v[4 * k + e] = __ldg(reinterpret_cast<const uint4*>(src) + e);
        }
        if (!aborted) {
#pragma unroll
          for (int k = 0; k < 3; ++k)
            ptx::tmem_st16(t_lane + kColQ + 16 * (c0 + k), *reinterpret_cast<float(*)[16]>(v + 4 * k));
        }
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(q_full);
    };

    // Own partial scores of page tt from TMEM into the staging rows, then one bulk
    // copy per warp into the peer's buffer once the peer has read the previous page's.
    auto fetch_send = [&](int tt) {
      if (!aborted && !bounded_wait(s_full, tt & 1, flags, p.err)) aborted = true;
      aborted = __any_sync(kFullMask, aborted);
      ptx::tc_fence_after();
      if (!aborted) {
#pragma unroll
        for (int c = 0; c < kPage; c += 16)
          ptx::tmem_ld16(t_lane + kColS + c, *reinterpret_cast<float(*)[16]>(sown + c));
        ptx::tmem_ld_wait();
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(s_free);
      if (!aborted && !bounded_wait_cluster(x_free, (tt & 1) ^ 1, flags, p.err)) aborted = true;
      if (lane == 0) ptx::bulk_wait_read_all();   // the staging rows are free again
      __syncwarp();
#pragma unroll
      for (int j = 0; j < kPage / 4; ++j)
        ptx::st_shared_v4(s_own + ((uint32_t(j) ^ sw) << 4), sown[4 * j], sown[4 * j + 1],
                          sown[4 * j + 2], sown[4 * j + 3]);
      ptx::fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0 && !aborted) {
        ptx::bulk_copy_to_peer(x_peer_blk, ptx::smem_addr(stg_out) + blk, 32 * kPage * 4, xfull_peer);
        ptx::bulk_commit();
      }
    };

    int t = 0;           // page index within this CTA's range
    // running maximum (log2 units), the sum of the fp32 weights (for the LSE) and the sum
    // of the 16-bit weights the PV MMA multiplies V by (O is normalised by this one, so
    // the output is a convex combination of V rows whatever the rounding of P)
    float m = 0.f, l = 0.f, lq = 0.f;
    Portion cur = walker_next(walk, spec, g_hi);
    load_q(cur);
    fetch_send(0);
    while (true) {
      const bool have_next = walk.g < g_hi;
      Portion nxt = cur;
      if (have_next) nxt = walker_next(walk, spec, g_hi);
      const int npg = cur.p1 - cur.p0;
      const int ctx = __ldg(p.context_lens + cur.b);

      for (int i = 0; i < npg; ++i, ++t) {
        // ---- the peer's partial scores of page t: S = S_own + S_peer
        float s[kPage];
        if (!aborted && !bounded_wait_cluster(x_full, t & 1, flags, p.err)) aborted = true;
        if (ctid == 0 && !aborted) ptx::mbar_arrive_expect_tx(x_full, kXBytes);  // next page
#pragma unroll
        for (int j = 0; j < kPage / 4; ++j) {
          const float4 v = aborted ? make_float4(0.f, 0.f, 0.f, 0.f)
                                   : ptx::ld_shared_v4(x_own + ((uint32_t(j) ^ sw) << 4));
          s[4 * j] = sown[4 * j] + v.x;
          s[4 * j + 1] = sown[4 * j + 1] + v.y;
          s[4 * j + 2] = sown[4 * j + 2] + v.z;
          s[4 * j + 3] = sown[4 * j + 3] + v.w;
        }
        __syncwarp();
        if (lane == 0 && !aborted) ptx::mbar_arrive_remote(xfree_peer);

        // ---- send the next page's partial scores before this page's softmax when its
        // scores are ready (same piece), so the exchange overlaps the exponentials
        const bool last = (i + 1 == npg);
        const bool more = !last || have_next;
        bool sent = false;
        if (!last) {
          int rdy = (lane == 0) ? int(ptx::mbar_try_wait(s_full, (t + 1) & 1)) : 0;
          if (__shfl_sync(kFullMask, rdy, 0)) {
            fetch_send(t + 1);
            sent = true;
          }
        }

        // ---- online softmax of page t (one head per thread)
        const int nvalid = min(kPage, ctx - (cur.p0 + i) * kPage);
        if (nvalid < kPage) {
#pragma unroll
          for (int j = 0; j < kPage; ++j)
            if (j >= nvalid) s[j] = -INFINITY;
        }
        float smax = s[0];
#pragma unroll
        for (int j = 1; j < kPage; ++j) smax = fmaxf(smax, s[j]);
        const float mx = smax * p.scale_log2;
        float alpha = 1.f;
        bool rescale = false;
        if (i == 0) {
          m = mx;
          l = 0.f;
          lq = 0.f;
        } else {
          // lazy maximum: raised only when a score exceeds the one in use by 2^8
          const bool need = mx > m + kRescaleLog2;
          rescale = __any_sync(kFullMask, need);
          if (need) {
            alpha = ptx::exp2_approx(m - mx);
            l *= alpha;
            lq *= alpha;
            m = mx;
          }
        }
        float pk[kPage / 2];   // P as 16-bit pairs (bit patterns)
        float lsum = 0.f, lqsum = 0.f;
#pragma unroll
        for (int j = 0; j < kPage / 2; ++j) {
          const float p0 = ptx::exp2_approx(fmaf(s[2 * j], p.scale_log2, -m));
          const float p1 = ptx::exp2_approx(fmaf(s[2 * j + 1], p.scale_log2, -m));
          const uint32_t w = pack2<T>(p0, p1);
          lsum += p0 + p1;
          lqsum += sum2<T>(w);
          pk[j] = __uint_as_float(w);
        }
        l += lsum;
        lq += lqsum;
        // P and O were last used by the PV of page t-1
        if (t >= 1 && !aborted && !bounded_wait(pv_done, (t - 1) & 1, flags, p.err)) aborted = true;
        aborted = __any_sync(kFullMask, aborted);
        ptx::tc_fence_after();
        if (!aborted) {
          if (rescale) {
            // O holds the piece's pages up to t-1: rescale this head's row
#pragma unroll 4
            for (int c = 0; c < kHalfDv; c += 16) {
              float v[16];
              ptx::tmem_ld16(t_lane + kColO + c, v);
              ptx::tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] *= alpha;
              ptx::tmem_st16(t_lane + kColO + c, v);
            }
          }
          ptx::tmem_st16(t_lane + kColP, *reinterpret_cast<float(*)[16]>(pk));
          ptx::tmem_st16(t_lane + kColP + 16, *reinterpret_cast<float(*)[16]>(pk + 16));
          ptx::tmem_st_wait();
        }
        // Slots past ctx: P is 0 there, but 0 * (whatever the slot holds, NaN included)
        // must not reach O, so their V rows are cleared before the PV MMA (the score MMA
        // has consumed the page). Thread ctid clears token ctid % 64 in two sub-tiles.
        if (nvalid < kPage) {
          const int r = ctid & (kPage - 1);
          if (r >= nvalid) {
            uint8_t* stg = kv + (t % kStages) * kStageBytes;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              uint4* dst =
                  reinterpret_cast<uint4*>(stg + ((ctid >> 6) * 2 + k) * kLatSubBytes + r * 128);
#pragma unroll
              for (int c = 0; c < 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          ptx::fence_proxy_async_shared();
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(p_full);

        if (more && !sent) {
          if (last) load_q(nxt);   // the score MMA of page t (the piece's last) is done
          fetch_send(t + 1);
        }
      }

      // ---- end of the piece: O_r / lq for this head
      const int tl = t - 1;
      if (!aborted && !bounded_wait(pv_done, tl & 1, flags, p.err)) aborted = true;
      aborted = __any_sync(kFullMask, aborted);
      ptx::tc_fence_after();

      const bool whole = (cur.p0 == 0 && cur.p1 == cur.np);
      const int slot = piece_slot(cur.seg_start, g_lo);
      const int64_t head_row = int64_t(cur.b) * p.num_q_heads + int64_t(cur.seg) * kHeads + h;
      const int64_t slot_row = (pair * 2 + slot) * kHeads + h;
      const float inv = 1.f / lq;
#pragma unroll 4
      for (int c = 0; c < kHalfDv; c += 16) {
        float v[16];
        if (!aborted) {
          ptx::tmem_ld16(t_lane + kColO + c, v);
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0.f;
        }
        const int d = int(rank) * kHalfDv + c;
        if (whole) {
          uint4 w0, w1;
          w0.x = pack2<T>(v[0] * inv, v[1] * inv);
          w0.y = pack2<T>(v[2] * inv, v[3] * inv);
          w0.z = pack2<T>(v[4] * inv, v[5] * inv);
          w0.w = pack2<T>(v[6] * inv, v[7] * inv);
          w1.x = pack2<T>(v[8] * inv, v[9] * inv);
          w1.y = pack2<T>(v[10] * inv, v[11] * inv);
          w1.z = pack2<T>(v[12] * inv, v[13] * inv);
          w1.w = pack2<T>(v[14] * inv, v[15] * inv);
          uint4* o = reinterpret_cast<uint4*>(outg + head_row * kDv + d);
          o[0] = w0;
          o[1] = w1;
        } else {
          float4* o = reinterpret_cast<float4*>(p.part_out + slot_row * kDv + d);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            __stcg(o + e, make_float4(v[4 * e] * inv, v[4 * e + 1] * inv, v[4 * e + 2] * inv,
                                      v[4 * e + 3] * inv));
        }
      }
      const float lse_nat = (m + log2f(l)) * kLn2;
      if (whole) {
        if (rank == 0 && p.lse != nullptr) p.lse[head_row] = lse_nat;
      } else {
        // both CTAs of the pair store this same value, so each half's merge finds it
        // once its own counter says every piece has arrived
        __stcg(p.part_lse + slot_row, lse_nat);
      }
      ptx::tc_fence_before();

      if (!whole) {
        // few pieces: the last to arrive merges its output half here; many: the
        // split-merge kernel that follows
        const int64_t c0 = cur.seg_start / p.tiles_per_cta;
        const int64_t c1 = (cur.seg_start + cur.np - 1) / p.tiles_per_cta;
        const int pieces = int(c1 - c0 + 1);
        if (pieces <= p.heavy_min) {
          __threadfence();
          ptx::named_barrier_sync(1, 32 * kSoftmaxWarps);
          int32_t* counter = p.counters + (int64_t(cur.b) * p.groups + cur.seg) * 2 + rank;
          if (ctid == 0) {
            const int prev = aborted ? -1 : atomicAdd(counter, 1);
            flags[1] = (prev == pieces - 1) ? 1 : 0;
          }
          ptx::named_barrier_sync(1, 32 * kSoftmaxWarps);
          if (flags[1]) {
            __threadfence();
            const int64_t head0 = int64_t(cur.b) * p.num_q_heads + int64_t(cur.seg) * kHeads;
            for (int idx = ctid; idx < kHeads * (kHalfDv / 4); idx += 32 * kSoftmaxWarps) {
              const int j = idx / (kHalfDv / 4);
              const int dq = idx - j * (kHalfDv / 4);
              float mxl = -INFINITY;
              for (int64_t c = c0; c <= c1; ++c) {
                const int sl = (c == c0 && cur.seg_start > c * p.tiles_per_cta) ? 1 : 0;
                mxl = fmaxf(mxl, __ldcg(p.part_lse + (c * 2 + sl) * kHeads + j));
              }
              float den = 0.f;
              float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int64_t c = c0; c <= c1; ++c) {
                const int sl = (c == c0 && cur.seg_start > c * p.tiles_per_cta) ? 1 : 0;
                const int64_t rowi = (c * 2 + sl) * kHeads + j;
                const float wgt = ptx::exp2_approx((__ldcg(p.part_lse + rowi) - mxl) * kLog2e);
                const float4 o = __ldcg(reinterpret_cast<const float4*>(
                                            p.part_out + rowi * kDv + int(rank) * kHalfDv) + dq);
                den += wgt;
                acc.x += wgt * o.x;
                acc.y += wgt * o.y;
                acc.z += wgt * o.z;
                acc.w += wgt * o.w;
              }
              const float dinv = 1.f / den;
              uint2 w;
              w.x = pack2<T>(acc.x * dinv, acc.y * dinv);
              w.y = pack2<T>(acc.z * dinv, acc.w * dinv);
              *reinterpret_cast<uint2*>(outg + (head0 + j) * kDv + int(rank) * kHalfDv + dq * 4) = w;
              if (rank == 0 && dq == 0 && p.lse != nullptr) p.lse[head0 + j] = mxl + logf(den);
            }
            if (ctid == 0) atomicExch(counter, 0);
          }
        }
      }
      ptx::named_barrier_sync(1, 32 * kSoftmaxWarps);
      if (!have_next) break;
      cur = nxt;
    }
    if (lane == 0) ptx::bulk_wait_all();   // the last copy into the peer has landed
  }

  // ---- teardown: no access to this CTA's shared memory from the peer after the
  // cluster barrier, and everyone is done with tensor memory before it is released
  ptx::tc_fence_before();
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn pair_encode_fn() {
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

// kv [blocks, 64, 576]:
//   latent: dims (d mod 64, slot, d / 64, block), box (64, 64, 4, 1) -> four [64][64] sub-tiles
//   rope:   dims (d, slot, block), box (32, 64, 1)                   -> one [64][32] tile
bool encode_pair_maps(CUtensorMap* kv_lat, CUtensorMap* kv_rope, const void* kv,
                      int64_t num_blocks, bool bf16) {
  EncodeTiledFn fn = pair_encode_fn();
  if (fn == nullptr) return false;
  const CUtensorMapDataType dt =
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const auto sw128 = CU_TENSOR_MAP_SWIZZLE_128B;
  const auto sw64 = CU_TENSOR_MAP_SWIZZLE_64B;
  const auto l2 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  const auto none = CU_TENSOR_MAP_INTERLEAVE_NONE;
  const auto fill = CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE;
  const cuuint32_t e4[4] = {1, 1, 1, 1};
  void* kp = const_cast<void*>(kv);
  {
    const cuuint64_t dims[4] = {64, kPage, kDqk / 64, cuuint64_t(num_blocks)};
    const cuuint64_t str[3] = {kDqk * 2, 128, cuuint64_t(kPage) * kDqk * 2};
    const cuuint32_t box[4] = {64, kPage, kLatSubs, 1};
    if (fn(kv_lat, dt, 4, kp, dims, str, box, e4, none, sw128, l2, fill) != CUDA_SUCCESS)
      return false;
  }
  {
    const cuuint64_t dims[3] = {kDqk, kPage, cuuint64_t(num_blocks)};
    const cuuint64_t str[2] = {kDqk * 2, cuuint64_t(kPage) * kDqk * 2};
    const cuuint32_t box[3] = {kRopeHalf, kPage, 1};
    if (fn(kv_rope, dt, 3, kp, dims, str, box, e4, none, sw64, l2, fill) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

template <typename T>
cudaError_t pair_kernel_attributes() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(mla_pair_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Layout::kSmem);
  });
  return err;
}

}  // namespace

bool mla_uses_pairs(const pda_problem& p) { return p.num_q_heads % kHeads == 0; }

int mla_pair_units(int num_sms) {
  int clusters = 0;
  if (pair_kernel_attributes<__nv_bfloat16>() == cudaSuccess) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * (num_sms / 2));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Layout::kSmem;
    if (cudaOccupancyMaxActiveClusters(&clusters, mla_pair_kernel<__nv_bfloat16>, &cfg) !=
        cudaSuccess)
      clusters = 0;
  }
  cudaGetLastError();
  const int by_sms = num_sms / 2;
  if (clusters <= 0) return by_sms > 0 ? by_sms : 1;
  return clusters < by_sms ? clusters : (by_sms > 0 ? by_sms : 1);
}

int launch_mla_pair(const Plan& plan, const MlaArgs& a, const Workspace& ws, void* stream) {
  const pda_problem& pr = plan.prob;
  const bool bf16 = pr.dtype == PDA_BF16;
  CUtensorMap tkl, tkr;
  if (!encode_pair_maps(&tkl, &tkr, a.kv_cache, pr.num_blocks, bf16)) return -1;
  PairParams prm{};
  prm.q = a.q;
  prm.out = a.out;
  prm.lse = a.lse;
  prm.block_tables = a.block_tables;
  prm.context_lens = a.context_lens;
  prm.batch = pr.batch;
  prm.num_q_heads = pr.num_q_heads;
  prm.groups = plan.segs_per_seq;
  prm.max_blocks = pr.max_blocks_per_seq;
  prm.num_blocks = pr.num_blocks;
  prm.scale_log2 = a.scale * kLog2e;
  prm.total_tiles = plan.total_tiles;
  prm.tiles_per_cta = plan.tiles_per_cta;
  prm.heavy_min = plan.heavy_min_pieces;
  prm.err = ws.err;
  prm.counters = ws.counters;
  prm.part_lse = ws.part_lse;
  prm.part_out = ws.part_out;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t attr =
      bf16 ? pair_kernel_attributes<__nv_bfloat16>() : pair_kernel_attributes<__half>();
  if (attr != cudaSuccess) return attr;
  const dim3 grid(2 * plan.num_ctas);
  if (bf16)
    mla_pair_kernel<__nv_bfloat16><<<grid, kThreads, Layout::kSmem, s>>>(tkl, tkr, prm);
  else
    mla_pair_kernel<__half><<<grid, kThreads, Layout::kSmem, s>>>(tkl, tkr, prm);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_split_merge(plan, ws, a.out, a.lse, stream);
}

}  // namespace pda
