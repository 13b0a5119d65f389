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
//  * CTA r owns the softmax of heads [64r, 64r+64), kept on tensor-memory lanes 64..127
//    (the peer's heads on lanes 0..63). Four "owner" warps (two per sub-partition,
//    splitting each page's tokens) add the peer's partial scores for their heads, run the
//    online softmax and send their P rows (8 KB, 16-bit) and rescale factors back; two
//    "relay" warps send the partial scores of the peer's heads (16 KB fp32 per page) as
//    soon as they exist and take in the peer's P rows and factors. The transfers between
//    the two SMs (bulk copies and st.async counted on the receiver's mbarriers) run about
//    40 GB/s each way with ~0.4 us latency, so they are double-buffered, and the owners
//    read their scores one page ahead so that the exchange overlaps a page of work.
//  * P[128 x 64] in shared memory is the A operand of the PV MMA:
//    O_r[128 x 256] += P * V_r[64 x 256] (M=128, N=256, 4 MMAs), V_r read in place
//    from the page's latent sub-tiles. CTA r owns output dims [256r, 256r+256); the
//    owners rescale their heads' rows of O_r, the relays the peer's heads' rows.
//  * At the end of a piece the owners send (m, l, lq) of their heads to the peer, and
//    both CTAs normalise and write their output half. Split pieces and their merge
//    follow the other decode kernels; each CTA merges its half of the output dims.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "pda_internal.h"
#include "ptx.cuh"
#include "ptx_ext.cuh"
#include "ptx_cluster.cuh"
#include "tile_walk.cuh"

namespace pda {

namespace {

constexpr int kPage = 64;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kHeads = 128;                 // query heads per pair
constexpr int kOwnHeads = kHeads / 2;       // heads whose softmax a CTA runs
constexpr int kHalfDv = kDv / 2;            // output / latent dims per CTA
constexpr int kLatSubs = kHalfDv / 64;      // 128-byte-swizzled 64-dim sub-tiles per CTA
constexpr int kRopeHalf = 32;               // rope dims per CTA (64-byte swizzle)
constexpr int kStages = 4;
constexpr int kLatSubBytes = kPage * 128;                          // [64 tokens][64 dims]
constexpr int kRopeBytes = kPage * kRopeHalf * 2;                  // [64 tokens][32 dims]
constexpr int kStageBytes = kLatSubs * kLatSubBytes + kRopeBytes;  // 36 KB
// 64 heads' fp32 scores of one page, laid out [token half][64 heads][32 tokens] so that
// each owner warp's half and each sender's half-block are contiguous
constexpr int kXsBytes = kOwnHeads * kPage * 4;
constexpr int kXsHalfBytes = kXsBytes / 2;
constexpr int kPBytes = kHeads * kPage * 2;                        // P tile, 16-bit
constexpr int kPRowsBytes = kOwnHeads * kPage * 2;                 // 64 heads' P rows
constexpr int kPMsgBytes = kPRowsBytes + kOwnHeads * 4;            // P rows + factors
constexpr int kFinBytes = kOwnHeads * 16;                          // (m, l, lq, -) per head
// Softmax group: two owner warps on each of the two sub-partitions that hold this CTA's
// heads (they split each page's tokens) and one relay warp on each of the other two.
constexpr int kGroupWarps = 6;
constexpr int kHalfTok = kPage / 2;
constexpr int kQWarps = kGroupWarps;     // warps that load q rows
constexpr int kPWarps = kGroupWarps;     // warps that arrive on p_full
constexpr int kSWarps = kGroupWarps;     // warps that read S
constexpr int kMergeThreads = 32 * kGroupWarps;   // the end-of-piece work
constexpr int kThreads = 64 + 32 * kGroupWarps;
constexpr int kTmemCols = 512;
// tensor-memory columns (32-bit): q_r as 16-bit pairs, S, O_r
constexpr int kColQ = 0;     // 144 columns: latent dims in [0, 128), rope dims in [128, 144)
constexpr int kColS = 192;   // 64 columns
constexpr int kColO = 256;   // 256 columns
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;   // lazy-max slack (log2 units)

struct Layout {
  static constexpr int kKV = 0;
  static constexpr int kXs = kKV + kStages * kStageBytes;   // [2] the peer's partials, own heads
  static constexpr int kSstg = kXs + 2 * kXsBytes;          // [2 relays] 32 heads x 64 tokens
  static constexpr int kP = kSstg + kXsBytes;                // [2] P tiles (both CTAs' rows)
  static constexpr int kAlpha = kP + 2 * kPBytes;            // [2][64] the peer's factors
  static constexpr int kFin = kAlpha + 2 * kOwnHeads * 4;    // [64] the peer's (m, l, lq)
  static constexpr int kRed = kFin + kFinBytes;              // owner halves: maxima, sums
  static constexpr int kBar = kRed + 1024;
  static constexpr int kBarCount = 32;
  // The dynamic shared memory must start on a 1024-byte boundary (checked at run time):
  // the layout leaves no room to align it by hand.
  static constexpr int kSmem = kBar + kBarCount * 8;
  static_assert(kStageBytes % 1024 == 0 && kXs % 1024 == 0 && kP % 1024 == 0,
                "swizzled tiles stay 1024-byte aligned");
  static_assert(kSmem <= 227 * 1024, "fits one SM's shared memory");
};

struct PairParams {
  const void* q;
  void* out;
  float* lse;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t batch, num_q_heads, groups, max_blocks;
  // S query tokens per sequence: rows R = i*Hq + h (query token i, head h) are contiguous in
  // q and out; head group seg holds rows [128 seg, 128 seg + 128), all of one query token
  int32_t rows_per_seq, seq_len_q;
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
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // Swizzled tiles need 1024-byte alignment and the layout has no slack to align by hand.
  // Both CTAs of a pair see the same address, so both leave here together if it is not.
  if ((ptx::smem_addr(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, 4);
    return;
  }
  uint8_t* base = smem_raw;
  uint8_t* kv = base + Layout::kKV;
  uint8_t* xs = base + Layout::kXs;
  uint8_t* sstg = base + Layout::kSstg;
  uint8_t* pbuf = base + Layout::kP;
  float* alpha_in = reinterpret_cast<float*>(base + Layout::kAlpha);
  float4* fin_in = reinterpret_cast<float4*>(base + Layout::kFin);
  float* red = reinterpret_cast<float*>(base + Layout::kRed);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + Layout::kBar);
  uint64_t* kv_full = bars + 0;    // [3] (4 slots kept)
  uint64_t* kv_empty = bars + 4;   // [3]
  uint64_t* q_full = bars + 8;     // q of the current piece is in tensor memory
  uint64_t* s_full = bars + 9;     // S written by the score MMA
  uint64_t* s_free = bars + 10;    // S read by the four softmax-group warps
  uint64_t* p_full = bars + 11;    // [2] P tile complete, O rows rescaled
  uint64_t* pv_done = bars + 13;   // [2] PV of a page completed
  uint64_t* xs_full = bars + 15;   // [2] the peer's partial scores of this CTA's heads
  uint64_t* xs_free = bars + 17;   // [2] the peer's owners have read what this CTA sent
  uint64_t* pr_full = bars + 19;   // [2] the peer's P rows and factors have landed
  uint64_t* pr_free = bars + 21;   // [2] the peer's PV of the page two back completed
  uint64_t* fin_full = bars + 23;  // the peer's (m, l, lq) of a piece have landed
  uint64_t* fin_free = bars + 24;  // the peer's relays have read this CTA's (m, l, lq)
  // [0] abort, [1] last piece to arrive
  volatile int* flags = reinterpret_cast<volatile int*>(bars + 26);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 30);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const uint32_t peer = rank ^ 1;
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
    ptx::mbar_init(q_full, kQWarps);
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(s_free, kSWarps);
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&p_full[b], kPWarps);
      ptx::mbar_init(&pv_done[b], 1);
      ptx::mbar_init(&xs_full[b], 1);
      ptx::mbar_init(&xs_free[b], 4);   // the peer's four owner warps
      ptx::mbar_init(&pr_full[b], 1);
      ptx::mbar_init(&pr_free[b], 1);   // the peer's MMA commit
    }
    ptx::mbar_init(fin_full, 1);
    ptx::mbar_init(fin_free, 2);        // the peer's two relay warps
    for (int i = 0; i < 8; ++i) flags[i] = 0;
    ptx::fence_mbarrier_init();
    // what the peer sends for the first two pages and the first piece (it may land first)
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_arrive_expect_tx(&xs_full[b], kXsBytes);
      ptx::mbar_arrive_expect_tx(&pr_full[b], kPMsgBytes);
    }
    ptx::mbar_arrive_expect_tx(fin_full, kFinBytes);
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
    // tile is complete.
    constexpr uint32_t kIdQK = ptx::umma_idesc_f16(128, 64, 0, 0, kBf16);
    constexpr uint32_t kIdPV = ptx::umma_idesc_f16(128, 256, 0, 1, kBf16);
    const uint32_t kv_s = ptx::smem_addr(kv);
    const uint32_t p_s = ptx::smem_addr(pbuf);
    if (lane == 0) {
      int u = 0, i = 0, npg = 0;
      int t_qk = 0, t_pv = 0, st_qk = 0, st_pv = 0;
      uint32_t ph_qk = 0;
      bool have = false, need_q = false, qk_done = false;
      uint32_t first_bits = 0;   // bit (t & 31): page t is the first of its piece
      ptx::Watchdog watchdog;
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
          const bool ready = (!need_q || ptx::mbar_test_wait(q_full, u & 1)) &&
                             ptx::mbar_test_wait(&kv_full[st_qk], ph_qk) &&
                             (t_qk == 0 || ptx::mbar_test_wait(s_free, (t_qk - 1) & 1));
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
        if (t_pv < t_qk && ptx::mbar_test_wait(&p_full[t_pv & 1], (t_pv >> 1) & 1)) {
          ptx::tc_fence_after();
          const bool first = (first_bits >> (t_pv & 31)) & 1u;
          const uint32_t stg = kv_s + st_pv * kStageBytes;
          const uint32_t pt = p_s + (t_pv & 1) * kPBytes;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            // P: 128 heads x 16 tokens (K-major, 128-byte swizzle); V_r: 16 tokens x 256
            // dims (dims contiguous in four 64-dim sub-tiles)
            const uint64_t a = ptx::umma_desc_sw128(pt + ks * 32, 16, 1024);
            const uint64_t b = ptx::umma_desc_sw128(stg + ks * 2048, kLatSubBytes, 1024);
            ptx::umma_f16(tmem + kColO, a, b, kIdPV, !(first && ks == 0));
          }
          ptx::umma_commit(&kv_empty[st_pv]);
          ptx::umma_commit(&pv_done[t_pv & 1]);
          // the peer may now write its P rows of the page two ahead into this CTA's tile
          ptx::umma_commit_multicast(&pr_free[t_pv & 1], uint16_t(1u << peer));
          ++t_pv;
          if (++st_pv == kStages) st_pv = 0;
          progress = true;
        }
        if (qk_done && t_pv == t_qk) break;
        if (progress) {
          watchdog.progress();
        } else if (flags[0] || watchdog.expired()) {
          flags[0] = 1;
          atomicOr(p.err, 2);
          break;
        }
      }
      // Wait (bounded) for the last MMAs before tensor memory is released.
      if (t_pv > 0) {
        const int tl = t_pv - 1;
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(&pv_done[tl & 1], (tl >> 1) & 1) &&
               ptx::globaltimer() - t0 < ptx::kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // ============================== softmax group: owners and relays ==============================
    // Tensor-memory lane L of CTA r holds head (L + 64 (1 - r)) mod 128: each CTA's own
    // heads sit on lanes 64..127 (sub-partitions 2 and 3, which have two warps each: the
    // owners), the peer's on lanes 0..63 (one relay warp on each of sub-partitions 0, 1).
    const int sp = warp & 3;                   // TMEM sub-partition of this warp
    const int pos = (warp - 2) >> 2;           // owners: which of the sub-partition's two warps
    const bool owner = sp >= 2;
    const int lrow = 32 * sp + lane;           // TMEM lane = row of S, P and O_r
    const int h = (lrow + kOwnHeads * (1 - int(rank))) & (kHeads - 1);   // head of this lane
    const int r = lrow & (kOwnHeads - 1);      // row of the head among its owner's 64
    const int gw = sp & 1;                     // sub-partition within its role
    const uint32_t t_lane = tmem + (uint32_t(32 * sp) << 16);
    const uint32_t swz = uint32_t(lrow & 7);
    const uint32_t row_off = uint32_t(r) * (kHalfTok * 4);       // half score rows: 128 B
    const uint32_t wblk_off = uint32_t(32 * gw) * (kHalfTok * 4);  // a sub-partition's 32 rows
    const uint32_t xs_s = ptx::smem_addr(xs);
    const uint32_t p_s = ptx::smem_addr(pbuf);
    const uint32_t pair_bar = 2 + sp;          // named barrier of a sub-partition's two warps
    const bool owner_lead = owner && gw == 0 && pos == 0 && lane == 0;
    const bool relay_lead = !owner && gw == 0 && lane == 0;
    const T* qg = static_cast<const T*>(p.q);
    T* outg = static_cast<T*>(p.out);
    bool aborted = false;

    auto remote = [&](const void* local) __attribute__((always_inline)) -> uint32_t {
      return ptx::mapa_shared(ptx::smem_addr(local), peer);
    };
    // q_r rows of this warp's heads into tensor memory (latent dims in columns [0, 128),
    // rope dims in [128, 144)); the two owner warps of a sub-partition split the chunks
    auto load_q = [&](const Portion& pq) __attribute__((always_inline)) {
      const T* qrow = qg + (int64_t(pq.b) * p.rows_per_seq + int64_t(pq.seg) * kHeads + h) * kDqk;
      const int c_lo = owner ? (pos == 0 ? 0 : 5) : 0;
      const int c_hi = owner ? (pos == 0 ? 5 : 9) : 9;
#pragma unroll
      for (int c0 = 0; c0 < 9; c0 += 3) {
        uint4 v[12];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int c = c0 + k;
          const T* src = c < 8 ? qrow + int(rank) * kHalfDv + 32 * c : qrow + kDv + int(rank) * kRopeHalf;
          if (c >= c_lo && c < c_hi) {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[4 * k + e] = __ldg(reinterpret_cast<const uint4*>(src) + e);
          }
        }
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int c = c0 + k;
          if (!aborted && c >= c_lo && c < c_hi)
            ptx::tmem_st16(t_lane + kColQ + 16 * c, *reinterpret_cast<float(*)[16]>(v + 4 * k));
        }
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(q_full);
    };
    // NC partial scores of page tt from column col0 of S; releases the S columns
    auto read_s = [&](int tt, int col0, auto& v) __attribute__((always_inline)) {
      constexpr int NC = sizeof(v) / sizeof(float);
      if (!aborted && !bounded_wait(s_full, tt & 1, flags, p.err)) aborted = true;
      aborted = __any_sync(kFullMask, aborted);
      ptx::tc_fence_after();
      if (!aborted) {
#pragma unroll
        for (int c = 0; c < NC; c += 16)
          ptx::tmem_ld16(t_lane + kColS + col0 + c, *reinterpret_cast<float(*)[16]>(&v[c]));
        ptx::tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < NC; ++j) v[j] = 0.f;
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(s_free);
    };
    // rescale columns [c0, c0 + n) of this head's row of O_r once the PV of page tt-1 is done
    auto rescale_row = [&](int tt, float alpha, int c0, int n) __attribute__((always_inline)) {
      if (!aborted && !bounded_wait(&pv_done[(tt - 1) & 1], ((tt - 1) >> 1) & 1, flags, p.err))
        aborted = true;
      aborted = __any_sync(kFullMask, aborted);
      ptx::tc_fence_after();
      if (!aborted) {
#pragma unroll 1
        for (int c = c0; c < c0 + n; c += 16) {
          float v[16];
          ptx::tmem_ld16(t_lane + kColO + c, v);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] *= alpha;
          ptx::tmem_st16(t_lane + kColO + c, v);
        }
        ptx::tmem_st_wait();
      }
    };
    // lse is [B][Hq][S]: row R = i*Hq + hh of the sequence goes to (b*Hq + hh)*S + i
    auto lse_at = [&](const Portion& pc, int row) __attribute__((always_inline)) -> int64_t {
      const int R = pc.seg * kHeads + row;
      const int qi = R / p.num_q_heads;
      return (int64_t(pc.b) * p.num_q_heads + (R - qi * p.num_q_heads)) * p.seq_len_q + qi;
    };
    // normalise columns [c0, c0 + n) of this head's row of O_r by 1/lq and write them out
    // (lq = 0: a causal head group that saw no token of a split piece; its O is 0)
    auto write_out = [&](const Portion& pc, float lq_tot, float lse_nat, int c0, int n,
                         bool write_lse) __attribute__((always_inline)) {
      const bool whole = (pc.p0 == 0 && pc.p1 == pc.np);
      const int slot = piece_slot(pc.seg_start, g_lo);
      const int64_t head_row = int64_t(pc.b) * p.rows_per_seq + int64_t(pc.seg) * kHeads + h;
      const int64_t slot_row = (pair * 2 + slot) * kHeads + h;
      const float inv = lq_tot > 0.f ? 1.f / lq_tot : 0.f;
#pragma unroll 2
      for (int c = c0; c < c0 + n; c += 16) {
        float o16[16];
        if (!aborted) {
          ptx::tmem_ld16(t_lane + kColO + c, o16);
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) o16[e] = 0.f;
        }
        const int d = int(rank) * kHalfDv + c;
        if (whole) {
          uint4 w0, w1;
          w0.x = pack2<T>(o16[0] * inv, o16[1] * inv);
          w0.y = pack2<T>(o16[2] * inv, o16[3] * inv);
          w0.z = pack2<T>(o16[4] * inv, o16[5] * inv);
          w0.w = pack2<T>(o16[6] * inv, o16[7] * inv);
          w1.x = pack2<T>(o16[8] * inv, o16[9] * inv);
          w1.y = pack2<T>(o16[10] * inv, o16[11] * inv);
          w1.z = pack2<T>(o16[12] * inv, o16[13] * inv);
          w1.w = pack2<T>(o16[14] * inv, o16[15] * inv);
          uint4* o = reinterpret_cast<uint4*>(outg + head_row * kDv + d);
          o[0] = w0;
          o[1] = w1;
        } else {
          float4* o = reinterpret_cast<float4*>(p.part_out + slot_row * kDv + d);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            __stcg(o + e, make_float4(o16[4 * e] * inv, o16[4 * e + 1] * inv, o16[4 * e + 2] * inv,
                                      o16[4 * e + 3] * inv));
        }
      }
      if (write_lse) {
        if (whole) {
          if (owner && p.lse != nullptr) p.lse[lse_at(pc, h)] = lse_nat;
        } else {
          // each CTA stores the LSE of all 128 heads (its owners' values and the peer's,
          // received at the end of the piece), so each half's merge finds them once its own
          // counter says every piece has arrived
          __stcg(p.part_lse + slot_row, lse_nat);
        }
      }
    };
    // the merge of a split segment's pieces by the last to arrive (this CTA's output half),
    // or nothing when the segment is whole or heavily split (the merge kernel's work);
    // run by all softmax-group warps (kMergeThreads, dense index mtid)
    auto merge_tail = [&](const Portion& pc) __attribute__((always_inline)) {
      const bool whole = (pc.p0 == 0 && pc.p1 == pc.np);
      const int mtid = (owner ? gw * 2 + pos : 4 + gw) * 32 + lane;
      if (!whole) {
        const int64_t c0 = pc.seg_start / p.tiles_per_cta;
        const int64_t c1 = (pc.seg_start + pc.np - 1) / p.tiles_per_cta;
        const int pieces = int(c1 - c0 + 1);
        if (pieces <= p.heavy_min) {
          __threadfence();
          ptx::named_barrier_sync(1, kMergeThreads);
          int32_t* counter = p.counters + (int64_t(pc.b) * p.groups + pc.seg) * 2 + rank;
          if (mtid == 0) {
            const int prev = aborted ? -1 : atomicAdd(counter, 1);
            flags[1] = (prev == pieces - 1) ? 1 : 0;
          }
          ptx::named_barrier_sync(1, kMergeThreads);
          if (flags[1]) {
            __threadfence();
            const int64_t head0 = int64_t(pc.b) * p.rows_per_seq + int64_t(pc.seg) * kHeads;
            for (int idx = mtid; idx < kHeads * (kHalfDv / 4); idx += kMergeThreads) {
              const int j = idx / (kHalfDv / 4);
              const int dq = idx - j * (kHalfDv / 4);
              float mxl = -INFINITY;
              for (int64_t c = c0; c <= c1; ++c) {
                const int sl = (c == c0 && pc.seg_start > c * p.tiles_per_cta) ? 1 : 0;
                mxl = fmaxf(mxl, __ldcg(p.part_lse + (c * 2 + sl) * kHeads + j));
              }
              float den = 0.f;
              float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int64_t c = c0; c <= c1; ++c) {
                const int sl = (c == c0 && pc.seg_start > c * p.tiles_per_cta) ? 1 : 0;
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
              if (rank == 0 && dq == 0 && p.lse != nullptr) p.lse[lse_at(pc, j)] = mxl + logf(den);
            }
            if (mtid == 0) atomicExch(counter, 0);
          }
        }
      }
      ptx::named_barrier_sync(1, kMergeThreads);
    };

    int t = 0;           // page index within this CTA's range
    int u = 0;           // piece index within this CTA's range
    Portion cur = walker_next(walk, spec, g_hi);
    load_q(cur);

    if (!owner) {
      // ---- relay: this CTA's partial scores of the peer's heads go out as soon as they
      // exist, and the peer's P rows and factors for those heads come in; one warp polls
      // both. After an abort every step counts as ready, so the relay still reaches each
      // piece's end (and its named barrier with the owners) exactly once.
      const int total = int(g_hi - g_lo);
      int ts = 0;                        // next page to send
      int s_rem = cur.p1 - cur.p0;       // pages of the send cursor's piece still to send
      Walker swalk = walk;               // send cursor, positioned after `cur`
      int i = 0;                         // receive cursor: page within `cur`
      // this warp's 8 KB staging block: [token half][32 rows][32 fp32]
      const uint32_t sblk = ptx::smem_addr(sstg) + uint32_t(gw) * (32 * kPage * 4);
      const uint32_t srow = sblk + uint32_t(lane) * (kHalfTok * 4);
      ptx::Watchdog watchdog;
      while (t < total) {
        if (flags[0]) aborted = true;
        aborted = __any_sync(kFullMask, aborted);
        bool progress = false;
        if (ts < total) {
          if (s_rem == 0) {
            // the previous piece's scores were all sent, so its last score MMA is done
            const Portion np = walker_next(swalk, spec, g_hi);
            s_rem = np.p1 - np.p0;
            load_q(np);
          }
          // ready: the page's scores exist, and the peer's owners have read page ts-2 from
          // the buffer this page goes to. Both are polled, never waited for here: this warp
          // must keep taking in the peer's P rows meanwhile (the peer's owners wait for this
          // CTA's PV of a page two back, which waits for those rows).
          const int b2 = ts & 1;
          const uint32_t par2 = uint32_t(ts >> 1) & 1;
          const int rdy = (lane == 0) ? int(aborted ||
                                            (ptx::mbar_try_wait(s_full, ts & 1) &&
                                             ptx::mbar_try_wait_cluster(&xs_free[b2], par2 ^ 1)))
                                      : 0;
          if (__shfl_sync(kFullMask, rdy, 0)) {
            float v[kPage];
            read_s(ts, 0, v);
            // both half-rows through this warp's staging block (its previous page's copies
            // have long been read), then one copy per half
            if (lane == 0) ptx::bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
              for (int j = 0; j < kHalfTok / 4; ++j)
                ptx::st_shared_v4(srow + hf * (32 * kHalfTok * 4) + ((uint32_t(j) ^ swz) << 4),
                                  v[32 * hf + 4 * j], v[32 * hf + 4 * j + 1],
                                  v[32 * hf + 4 * j + 2], v[32 * hf + 4 * j + 3]);
            ptx::fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0 && !aborted) {
#pragma unroll
              for (int hf = 0; hf < 2; ++hf)
                ptx::bulk_copy_to_peer(remote(xs + b2 * kXsBytes + hf * kXsHalfBytes + wblk_off),
                                       sblk + hf * (32 * kHalfTok * 4), 32 * kHalfTok * 4,
                                       remote(&xs_full[b2]));
              ptx::bulk_commit();
            }
            ++ts;
            --s_rem;
            progress = true;
          }
        }
        if (t < ts) {
          const int b2 = t & 1;
          const uint32_t par2 = uint32_t(t >> 1) & 1;
          const int rdy =
              (lane == 0) ? int(aborted || ptx::mbar_try_wait_cluster(&pr_full[b2], par2)) : 0;
          if (__shfl_sync(kFullMask, rdy, 0)) {
            // the peer's P rows of page t are in this CTA's tile: rescale those heads' O rows
            const float alpha = aborted ? 1.f : alpha_in[b2 * kOwnHeads + r];
            __syncwarp();
            if (relay_lead && !aborted) ptx::mbar_arrive_expect_tx(&pr_full[b2], kPMsgBytes);  // page t+2
            if (__any_sync(kFullMask, alpha != 1.f)) rescale_row(t, alpha, 0, kHalfDv);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&p_full[b2]);
            if (++i == cur.p1 - cur.p0) {
              // end of the piece: the owner's (m, l, lq) of this head, then the output
              if (!aborted && !bounded_wait_cluster(fin_full, u & 1, flags, p.err)) aborted = true;
              // acquire load: the relaxed arrive on fin_free below comes after it
              const float4 f = aborted ? make_float4(0.f, 1.f, 1.f, 0.f)
                                       : ptx::ld_shared_v4_acquire(ptx::smem_addr(fin_in + r));
              __syncwarp();
              if (lane == 0 && !aborted) ptx::mbar_arrive_remote_relaxed(remote(fin_free));
              if (relay_lead && !aborted) ptx::mbar_arrive_expect_tx(fin_full, kFinBytes);  // next piece
              if (!aborted && !bounded_wait(&pv_done[b2], par2, flags, p.err)) aborted = true;
              aborted = __any_sync(kFullMask, aborted);
              ptx::tc_fence_after();
              write_out(cur, f.z, (f.x + log2f(f.y)) * kLn2, 0, kHalfDv, true);
              ptx::tc_fence_before();
              merge_tail(cur);
              ++u;
              i = 0;
              if (walk.g < g_hi) cur = walker_next(walk, spec, g_hi);
            }
            ++t;
            progress = true;
          }
        }
        if (progress) {
          watchdog.progress();
        } else if (watchdog.expired()) {
          if (lane == 0) {
            flags[0] = 1;
            atomicOr(p.err, 2);
          }
          aborted = true;
        }
      }
      if (lane == 0) ptx::bulk_wait_all();   // the last copies into the peer have landed
    } else {
      // ---- owner (token half `pos`): S = S_own + S_peer, online softmax, P row half out
      // [2 halves][64 rows] half maxima of the page in hand; at the end of a piece the same
      // words hold [2 halves][2 sums][64 rows] (the pair barriers order the reuse)
      float* hmx = red;
      float* hsm = red;
      const int o = (gw * 2 + pos) * 32 + lane;   // 0 .. 127 over the owner warps
      // running maximum (log2 units), this half's sums of the fp32 weights (for the LSE)
      // and of the 16-bit weights the PV MMA multiplies V by (O is normalised by the
      // latter, so the output is a convex combination of V rows whatever the rounding of P)
      float m = 0.f, l = 0.f, lq = 0.f;
      // Scores are read one page ahead: reading S(t+1) at the top of page t frees the S
      // columns, so the score MMA runs two pages ahead of this loop and the peer's partial
      // scores of page t have a whole page of work to arrive in.
      const int total = int(g_hi - g_lo);
      float vn[kHalfTok];      // own partial scores of the page read ahead
      int tr = 0;              // next page to read
      int r_rem = cur.p1 - cur.p0;   // pages of the read cursor's piece still to read
      Walker rwalk = walk;     // positioned after `cur`
      Portion q_next = cur;    // a piece whose q is to be loaded at the end of this page
      bool q_pending = false;
      auto read_next = [&]() __attribute__((always_inline)) {
        read_s(tr, kHalfTok * pos, vn);
        ++tr;
        if (--r_rem == 0 && rwalk.g < g_hi) {
          // the piece's last score MMA is done: q of the next piece, loaded once this
          // page's registers are free (and before the next read needs it)
          q_next = walker_next(rwalk, spec, g_hi);
          r_rem = q_next.p1 - q_next.p0;
          q_pending = true;
        }
      };
      read_next();
      if (q_pending) {
        load_q(q_next);
        q_pending = false;
      }
      while (true) {
        const int npg = cur.p1 - cur.p0;
        // this head group's query token qi sees tokens [0, ctx - S + 1 + qi) (all of them
        // with S = 1); a page past that limit (the last page, for an earlier token) adds
        // nothing, and a piece made only of such pages ends with l = 0, LSE = -inf
        const int qi = cur.seg * kHeads / p.num_q_heads;
        const int ctx = __ldg(p.context_lens + cur.b) - p.seq_len_q + 1 + qi;
        for (int i = 0; i < npg; ++i, ++t) {
          const int b2 = t & 1;
          const uint32_t par2 = uint32_t(t >> 1) & 1;
          const int nvalid = min(kPage, ctx - (cur.p0 + i) * kPage);
          float v[kHalfTok];
#pragma unroll
          for (int j = 0; j < kHalfTok; ++j) v[j] = vn[j];
          if (tr < total) read_next();
          if (!aborted && !bounded_wait_cluster(&xs_full[b2], par2, flags, p.err)) aborted = true;
          if (owner_lead && !aborted) ptx::mbar_arrive_expect_tx(&xs_full[b2], kXsBytes);  // page t+2
          const uint32_t xr = xs_s + b2 * kXsBytes + pos * kXsHalfBytes + row_off;
          // The peer overwrites this buffer once it sees the relaxed arrive on xs_free below.
          // The loads are plain shared-memory loads, not acquire loads: every loaded value is
          // added into v before the warp barrier, and lane 0 issues the arrive after that
          // barrier, so each lane's loads have returned their data before the arrive is
          // issued and no later write by the peer can reach them. (The PTX memory model
          // alone would ask for acquire loads or a release arrive here: acquire loads cost
          // 410.5 against 399.8 us per step at B=16, ctx 64K, and a release arrive, which
          // also waits for this thread's outstanding stores to the peer, ~70 us.)
#pragma unroll
          for (int j = 0; j < kHalfTok / 4; ++j) {
            const float4 x = aborted ? make_float4(0.f, 0.f, 0.f, 0.f)
                                     : ptx::ld_shared_v4(xr + ((uint32_t(j) ^ swz) << 4));
            v[4 * j] += x.x;
            v[4 * j + 1] += x.y;
            v[4 * j + 2] += x.z;
            v[4 * j + 3] += x.w;
          }
          __syncwarp();
          if (lane == 0 && !aborted) ptx::mbar_arrive_remote_relaxed(remote(&xs_free[b2]));
          const int nv = nvalid - kHalfTok * pos;   // valid tokens of this half
          // The largest scaled score is the scale times the largest raw score (scale >= 0)
          // or the smallest (scale < 0); masked tokens take no part in it.
          const float sc = p.scale_log2;
          const bool neg = sc < 0.f;
          if (nv < kHalfTok) {
#pragma unroll
            for (int j = 0; j < kHalfTok; ++j)
              if (j >= nv) v[j] = neg ? INFINITY : -INFINITY;
          }
          float smax = v[0];
          if (neg) {
#pragma unroll
            for (int j = 1; j < kHalfTok; ++j) smax = fminf(smax, v[j]);
          } else {
#pragma unroll
            for (int j = 1; j < kHalfTok; ++j) smax = fmaxf(smax, v[j]);
          }
          // the head's extreme over both halves (the two warps agree on every decision)
          hmx[pos * kOwnHeads + r] = smax;
          ptx::named_barrier_sync(pair_bar, 64);
          const float ext = neg ? fminf(hmx[r], hmx[kOwnHeads + r])
                                : fmaxf(hmx[r], hmx[kOwnHeads + r]);
          const float mx = ext * sc;
          float alpha = 1.f;
          bool need = false;
          if (i == 0) {
            m = mx;
            l = 0.f;
            lq = 0.f;
          } else if (mx > m + kRescaleLog2) {
            // lazy maximum: raised only when a score exceeds the one in use by 2^8
            need = true;
            alpha = ptx::exp2_approx(m - mx);
            l *= alpha;
            lq *= alpha;
            m = mx;
          }
          uint32_t pk[kHalfTok / 2];   // P as 16-bit pairs
          float lsum = 0.f, lqsum = 0.f;
#pragma unroll
          for (int j = 0; j < kHalfTok / 2; ++j) {
            float p0 = ptx::exp2_approx(fmaf(v[2 * j], sc, -m));
            float p1 = ptx::exp2_approx(fmaf(v[2 * j + 1], sc, -m));
            if (nv < kHalfTok) {   // masked tokens weigh 0 (whatever the scale's sign)
              if (2 * j >= nv) p0 = 0.f;
              if (2 * j + 1 >= nv) p1 = 0.f;
            }
            pk[j] = pack2<T>(p0, p1);
            lsum += p0 + p1;
            lqsum += sum2<T>(pk[j]);
          }
          l += lsum;
          lq += lqsum;
          if (__any_sync(kFullMask, need)) rescale_row(t, alpha, (kHalfDv / 2) * pos, kHalfDv / 2);
          // this CTA's P tile of page t was last read by the PV of page t-2, and its owner
          // rows by the copy to the peer (issued by warp pos 0 of each sub-partition)
          if (t >= 2 && !aborted &&
              !bounded_wait(&pv_done[b2], ((t >> 1) - 1) & 1, flags, p.err))
            aborted = true;
          if (pos == 0 && lane == 0) ptx::bulk_wait_read_all();
          ptx::named_barrier_sync(pair_bar, 64);
          const uint32_t prow = p_s + b2 * kPBytes + uint32_t(lrow) * 128;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             prow + ((uint32_t(4 * pos + j) ^ swz) << 4)),
                         "r"(pk[4 * j]), "r"(pk[4 * j + 1]), "r"(pk[4 * j + 2]), "r"(pk[4 * j + 3])
                         : "memory");
          }
          // Slots past ctx: P is 0 there, but 0 * (whatever the slot holds, NaN included)
          // must not reach O, so their V rows are cleared before the PV MMA (the score MMA
          // has consumed the page). Owner thread o clears token o % 64 in two sub-tiles.
          if (nvalid < kPage && (o & (kPage - 1)) >= nvalid) {
            uint8_t* stg = kv + (t % kStages) * kStageBytes + (o & (kPage - 1)) * 128;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              uint4* dst = reinterpret_cast<uint4*>(stg + ((o >> 6) * 2 + k) * kLatSubBytes);
#pragma unroll
              for (int c = 0; c < 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          ptx::fence_proxy_async_shared();
          ptx::named_barrier_sync(pair_bar, 64);
          // to the peer, once its PV of page t-2 is done: the factors and this sub-partition's
          // P rows (32 heads x 128 B)
          if (pos == 0) {
            int ok = 1;
            if (lane == 0 && !aborted &&
                !bounded_wait_cluster(&pr_free[b2], par2 ^ 1, flags, p.err))
              ok = 0;
            if (!__shfl_sync(kFullMask, ok, 0)) aborted = true;
            const uint32_t pr_peer = remote(&pr_full[b2]);
            if (!aborted)
              ptx::st_async_b32(remote(alpha_in + b2 * kOwnHeads + r), __float_as_uint(alpha), pr_peer);
            __syncwarp();
            if (lane == 0 && !aborted) {
              // this CTA's lanes 64..127 are the peer's lanes 0..63 (the same heads)
              const uint32_t src = b2 * kPBytes + uint32_t(32 * sp) * 128;
              const uint32_t dst = b2 * kPBytes + uint32_t(32 * gw) * 128;
              ptx::bulk_copy_to_peer(remote(pbuf + dst), p_s + src, 32 * 128, pr_peer);
              ptx::bulk_commit();
            }
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&p_full[b2]);
          if (q_pending) {
            load_q(q_next);
            q_pending = false;
          }
        }
        // ---- the next piece (its q was loaded by the read-ahead)
        const bool have_next = walk.g < g_hi;
        Portion nxt = cur;
        if (have_next) nxt = walker_next(walk, spec, g_hi);
        // ---- end of the piece: both halves' sums, (m, l, lq) to the peer, then O_r / lq
        hsm[(pos * 2) * kOwnHeads + r] = l;
        hsm[(pos * 2 + 1) * kOwnHeads + r] = lq;
        ptx::named_barrier_sync(pair_bar, 64);
        const float l_tot = hsm[r] + hsm[2 * kOwnHeads + r];
        const float lq_tot = hsm[kOwnHeads + r] + hsm[3 * kOwnHeads + r];
        ptx::named_barrier_sync(pair_bar, 64);
        if (pos == 0) {
          int ok = 1;
          if (lane == 0 && !aborted && !bounded_wait_cluster(fin_free, (u & 1) ^ 1, flags, p.err))
            ok = 0;
          if (!__shfl_sync(kFullMask, ok, 0)) aborted = true;
          if (!aborted)
            ptx::st_async_v4(remote(fin_in + r), __float_as_uint(m), __float_as_uint(l_tot),
                             __float_as_uint(lq_tot), 0u, remote(fin_full));
        }
        const int tl = t - 1;
        if (!aborted && !bounded_wait(&pv_done[tl & 1], (tl >> 1) & 1, flags, p.err)) aborted = true;
        aborted = __any_sync(kFullMask, aborted);
        ptx::tc_fence_after();
        write_out(cur, lq_tot, (m + log2f(l_tot)) * kLn2, (kHalfDv / 2) * pos, kHalfDv / 2, pos == 0);
        ptx::tc_fence_before();
        merge_tail(cur);
        ++u;
        if (!have_next) break;
        cur = nxt;
      }
      if (lane == 0) ptx::bulk_wait_all();   // the last copies into the peer have landed
    }
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

bool mla_uses_pairs(const pda_problem& p) {
  return p.head_dim_qk == kDqk && p.num_q_heads % kHeads == 0 &&
         p.kv_format == PDA_KV_SAME_AS_Q;
}

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
  CUtensorMap m[2];
  if (!plan.map_cache.get(a.kv_cache, nullptr, m, nullptr, [&](CUtensorMap* t, int32_t*) {
        return encode_pair_maps(&t[0], &t[1], a.kv_cache, pr.num_blocks, bf16);
      }))
    return -1;
  const CUtensorMap& tkl = m[0];
  const CUtensorMap& tkr = m[1];
  PairParams prm{};
  prm.q = a.q;
  prm.out = a.out;
  prm.lse = a.lse;
  prm.block_tables = a.block_tables;
  prm.context_lens = a.context_lens;
  prm.batch = pr.batch;
  prm.num_q_heads = pr.num_q_heads;
  prm.seq_len_q = pr.seq_len_q > 1 ? pr.seq_len_q : 1;
  prm.rows_per_seq = prm.seq_len_q * pr.num_q_heads;
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
