// Absorbed-MLA paged decode for sm_103a on the 5th-generation tensor cores.
//
// What it computes ("From MHA to MLA", section 6; FlashMLA-ETAP README, "Usage"
// and "Supported configurations"): every query head attends to one shared record
// per cached token of Dqk values, Dv latent then 64 rope: (576, 512) for kv_lora_rank
// 512, (320, 256) for kv_lora_rank 256. The score of head h and token j is
// scale * (<q_h[:Dv], c_j> + <q_h[Dv:], k_j^R>) = scale * <q_h, rec_j>; the value is
// the latent c_j = rec_j[:Dv]. Output [B, Hq, Dv] and fp32 LSE.
//
// How (GB300 design; the FlashMLA-ETAP page describes a Hopper WGMMA kernel with
// the transposed pipeline, whose idea of putting keys on the MMA's M axis is kept):
//  * One CTA per range of (sequence, head group, page) tiles, the same equal-work
//    split as the GQA kernel; a head group is N = min(Hq, 64) heads, so TMEM holds
//    the N score columns plus Dv / 128 x N columns of the transposed output.
//  * Warp 0 streams pages with one TMA copy each (a 64-token x Dqk page lands as
//    Dqk / 64 128-byte-swizzled [64][64] sub-tiles) into a two-stage ring, and
//    loads the head group's q once per piece.
//  * Warp 1 issues tcgen05.mma from one thread:
//      S^T[64 tokens x N]  = K[64 x Dqk] * q^T        (M=64, K-major A and B)
//      O^T[Dv x N]        += V^T[Dv x 64] * P^T        (Dv / 128 x M=128, MN-major A and B)
//    V^T is read in place from the same page sub-tiles (MN-major descriptor), so
//    each latent byte is read from HBM once.
//  * Warps 2-5 read S^T from TMEM (tcgen05.ld), run the online softmax down each
//    head column and write P^T (bf16/fp16) over the page's rope sub-tile, which
//    the score MMA no longer needs. The running maximum is kept lazily: an exact
//    column maximum is taken on a piece's first page and whenever some score
//    exceeds the maximum in use by more than 2^8; only then is O^T rescaled in
//    TMEM. The result is the same softmax (the common factor cancels in O/l).
//  * At the end of a piece the same warps normalise O^T and write the output, or
//    write a split piece that is merged like the GQA splits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "mla_maps.h"
#include "pda_internal.h"
#include "ptx.cuh"
#include "ptx_ext.cuh"
#include "tile_walk.cuh"

namespace pda {

namespace {

constexpr int kPage = 64;
constexpr int kSubBytes = kPage * 128;        // [64 tokens][64 dims] x 16 bit
// A cached record of DQK 16-bit values: DQK - 64 latent dims (the value) then 64 rope
// dims. FlashMLA-ETAP "Supported configurations": (576, 512) for kv_lora_rank 512 and
// (320, 256) for kv_lora_rank 256.
template <int DQK>
struct Rec {
  static constexpr int kDv = DQK - 64;
  static constexpr int kSubTiles = DQK / 64;          // 64-dim sub-tiles per record
  static constexpr int kPageBytes = kSubTiles * kSubBytes;
  static constexpr int kRopeSub = kSubTiles - 1;      // sub-tile reused for P^T
  static constexpr int kMTiles = kDv / 128;           // 128-dim O^T tiles of the PV MMA
  // Page ring stages: two 72 KB pages of the 576 record (with q for 64 heads, most of
  // shared memory), four 40 KB pages of the 320 record.
  static constexpr int kStages = DQK == 576 ? 2 : 4;
  static_assert(DQK % 64 == 0 && (DQK - 64) % 128 == 0, "latent width a multiple of 128");
};
// Warp 0 TMA, warp 1 MMA, then the softmax warps: 4 (one per TMEM sub-partition) for
// N = 16 heads, 8 for N >= 32 (two per sub-partition, each owning half the head columns).
template <int N>
struct SoftmaxWarps {
  static constexpr int kWarps = N >= 32 ? 8 : 4;
  static constexpr int kThreads = 64 + 32 * kWarps;
  static constexpr int kCols = N / (kWarps / 4);   // head columns per softmax thread
};
// E4M3 caches add converter warps after the softmax warps (groups of 16 or 32 rows): one
// per sub-partition beside 16 heads' four softmax warps, two beside 32 heads' eight (more
// would cap the registers of every warp below what the softmax warps use).
template <int N, bool F8>
struct Roles {
  static constexpr int kConvWarps = F8 ? (N == 16 ? 4 : 2) : 0;
  static constexpr int kThreads = SoftmaxWarps<N>::kThreads + 32 * kConvWarps;
};
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;           // lazy-max slack (log2 units)

struct MlaParams {
  const void* q;
  void* out;
  float* lse;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t batch, num_q_heads, groups, max_blocks;
  // S query tokens per sequence: the S*Hq rows of a sequence (row R = i*Hq + h, query
  // token i, head h) are contiguous in q and out; with S > 1 they form one head group
  int32_t rows_per_seq, seq_len_q;
  int64_t num_blocks;
  float scale_log2;   // softmax scale (times the record scale for E4M3 caches) times log2(e)
  float v_scale;      // E4M3 caches: the record's dequantization scale (1 for 16-bit caches)
  int64_t total_tiles, tiles_per_cta;
  int32_t heavy_min;
  int32_t* err;
  int32_t* counters;
  float* part_lse;
  float* part_out;
};

template <int N, int DQK, bool F8 = false>
struct MlaLayout {
  using R = Rec<DQK>;
  // E4M3 caches with the two-stage ring (576 record): one page of codes beside the ring,
  // so the next page's copy lands while the ring's stages are busy
  static constexpr bool kSepCodes = F8 && R::kStages == 2;
  static constexpr int kQBytes = R::kSubTiles * N * 128;  // q as K-major [N][64] sub-tiles
  static constexpr int kKV = 0;
  static constexpr int kQ = kKV + R::kStages * R::kPageBytes;
  static constexpr int kRed = kQ + kQBytes;            // [64 heads][4 warps] floats
  static constexpr int kMused = kRed + 64 * 4 * 4;     // running maximum per head (log2 units)
  static constexpr int kAlpha = kMused + 64 * 4;       // rescale factor per head
  static constexpr int kLtot = kAlpha + 64 * 4;        // softmax denominator per head
  static constexpr int kLqtot = kLtot + 64 * 4;        // sum of the rounded weights per head
  static constexpr int kCodes = (kLqtot + 64 * 4 + 1023) / 1024 * 1024;   // [page of codes]
  static constexpr int kBar = kCodes + (kSepCodes ? DQK * 64 : 0);
  static constexpr int kBarCount = 2 * R::kStages + 24;
  static constexpr int kSmem = 1024 + kBar + kBarCount * 8 + 64;
  static_assert(kSmem <= 232448, "fits the 227 KB of dynamic shared memory per block");
  // TMEM columns: S^T double-buffered at [0, 2N), O^T d-tile mt at 2N + mt*N
  static constexpr int kCols = (2 + R::kMTiles) * N;
  static constexpr int kTmemCols = kCols <= 128 ? 128 : (kCols <= 256 ? 256 : 512);
  static constexpr int kColS = 0;
  static constexpr int kColO = 2 * N;
  static_assert(kQBytes % 1024 == 0, "q sub-tiles stay 1024-byte aligned");
};

__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                             int32_t* err) {
  if (wait_phase(bar, parity, abort)) return true;
  *abort = 1;
  atomicOr(err, 2);
  return false;
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

template <int N, int DQK, typename T, bool F8>
__global__ void __launch_bounds__(Roles<N, F8>::kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_kv, const MlaParams p) {
  using L = MlaLayout<N, DQK, F8>;
  using R = Rec<DQK>;
  constexpr int kDv = R::kDv;
  constexpr int kSubTiles = R::kSubTiles;
  constexpr int kPageBytes = R::kPageBytes;
  constexpr int kRopeSub = R::kRopeSub;
  constexpr int KS = R::kStages;
  // The MMAs' operand type: q's type for 16-bit caches. For E4M3 caches the codes become
  // fp16 (exact, one conversion per two codes), and q (converted in shared memory once per
  // piece, exact for |q| in [2^-14, 65504]) and P follow, since both operands of one MMA
  // share a type; the output keeps q's type.
  using TM = typename std::conditional<F8, __half, T>::type;
  constexpr bool kBf16 = std::is_same<TM, __nv_bfloat16>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* kv = base + L::kKV;
  uint8_t* qs = base + L::kQ;
  float* red = reinterpret_cast<float*>(base + L::kRed);
  float* mused = reinterpret_cast<float*>(base + L::kMused);
  float* alpha_s = reinterpret_cast<float*>(base + L::kAlpha);
  float* ltot = reinterpret_cast<float*>(base + L::kLtot);
  float* lqtot = reinterpret_cast<float*>(base + L::kLqtot);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::kBar);
  // Page t sits in ring stage t % KS (its P^T in that stage's rope sub-tile).
  uint64_t* kv_full = bars + 0;        // [KS]
  uint64_t* kv_empty = bars + KS;      // [KS]
  uint64_t* q_full = bars + 2 * KS;
  uint64_t* q_empty = bars + 2 * KS + 1;
  // Barriers that complete once per page come in pairs indexed by page parity, so a
  // waiter is never two phases behind (the S^T buffer alternates too).
  uint64_t* s_full = bars + 2 * KS + 2;    // [2] S^T buffer written
  uint64_t* s_free = bars + 2 * KS + 4;    // [2] S^T buffer read, P^T written
  uint64_t* p_full = bars + 2 * KS + 6;    // [2]
  uint64_t* pv_done = bars + 2 * KS + 8;   // [2] PV of a page completed
  // [0] abort, [1] last piece, [2..9] softmax-warp votes (5 slots)
  volatile int* flags = reinterpret_cast<volatile int*>(bars + 2 * KS + 10);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * KS + 16);
  // E4M3 caches: a page's codes have landed in the upper half of its stage (the converters
  // then arrive on kv_full once the stage holds the 16-bit record)
  uint64_t* kv_f8 = bars + 2 * KS + 17;   // [KS]
  // separate code page (L::kSepCodes): kv_f8[0] = the page of codes has landed, kv_f8[1] =
  // the converters have read it
  constexpr bool kSep = L::kSepCodes;
  uint8_t* codes_buf = base + L::kCodes;
  uint64_t* q_cvt = bars + 2 * KS + 17 + KS;   // E4M3 caches: q is in the MMAs' type
  constexpr int kConvWarps = Roles<N, F8>::kConvWarps;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t g_lo = int64_t(blockIdx.x) * p.tiles_per_cta;
  const int64_t g_hi = min(p.total_tiles, g_lo + p.tiles_per_cta);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (g_lo >= g_hi) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < KS; ++s) {
      ptx::mbar_init(&kv_full[s], F8 ? kConvWarps : 1);
      ptx::mbar_init(&kv_empty[s], 1);
      ptx::mbar_init(&kv_f8[s], (kSep && s == 1) ? kConvWarps : 1);
    }
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_empty, 1);
    ptx::mbar_init(q_cvt, kConvWarps > 0 ? kConvWarps : 1);
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&s_full[b], 1);
      ptx::mbar_init(&s_free[b], SoftmaxWarps<N>::kWarps);
      ptx::mbar_init(&p_full[b], SoftmaxWarps<N>::kWarps);
      ptx::mbar_init(&pv_done[b], 1);
    }
    for (int i = 0; i < 10; ++i) flags[i] = 0;
    ptx::fence_mbarrier_init();
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, L::kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const WalkSpec spec{p.context_lens, p.batch, p.groups, kPage};
  Walker walk;
  walker_init(walk, spec, g_lo, lane);

  if (warp == 0) {
    // ============================== TMA producer ==============================
    if (lane == 0) {
      ptx::prefetch_tensormap(&tm_q);
      ptx::prefetch_tensormap(&tm_kv);
    }
    const uint64_t pol_stream = ptx::policy_evict_first();
    int t = 0, u = 0;
    bool ok = true;
    while (ok && walk.g < g_hi) {
      const Portion pt = walker_next(walk, spec, g_hi);
      if (lane == 0) {
        if (u > 0) ok = bounded_wait(q_empty, (u - 1) & 1, flags, p.err);
        if (ok) {
          ptx::mbar_arrive_expect_tx(q_full, L::kQBytes);
          ptx::tma_load_3d(qs, &tm_q, q_full, 0, pt.b * p.rows_per_seq + pt.seg * N, 0,
                           pol_stream);
        }
      }
      ok = __shfl_sync(kFullMask, ok ? 1 : 0, 0) != 0;
      const int32_t* row = p.block_tables + int64_t(pt.b) * p.max_blocks;
      for (int base_pg = pt.p0; ok && base_pg < pt.p1; base_pg += 32) {
        const int32_t ids = (base_pg + lane < pt.p1) ? __ldg(row + base_pg + lane) : 0;
        const int n = min(32, pt.p1 - base_pg);
        for (int j = 0; j < n; ++j, ++t) {
          const int32_t phys = __shfl_sync(kFullMask, ids, j);
          int good = 1;
          if (lane == 0) {
            const int s = t % KS;
            // the separate code page waits for the converters to have read the previous
            // page (they wait for the ring stage); otherwise the stage itself must be free
            if (kSep ? (t > 0 && !bounded_wait(&kv_f8[1], (t - 1) & 1, flags, p.err))
                     : !bounded_wait(&kv_empty[s], ((t / KS) & 1) ^ 1, flags, p.err)) {
              good = 0;
            } else {
              if (phys < 0 || int64_t(phys) >= p.num_blocks) atomicOr(p.err, 1);
              if constexpr (kSep) {
                ptx::mbar_arrive_expect_tx(&kv_f8[0], kPageBytes / 2);
                ptx::tma_load_4d(codes_buf, &tm_kv, &kv_f8[0], 0, 0, 0, phys, pol_stream);
              } else if constexpr (F8) {
                // the page's E4M3 codes, [sub-tile][64 tokens][64 B], into the stage's upper half
                ptx::mbar_arrive_expect_tx(&kv_f8[s], kPageBytes / 2);
                ptx::tma_load_4d(kv + s * kPageBytes + kPageBytes / 2, &tm_kv, &kv_f8[s], 0, 0,
                                 0, phys, pol_stream);
              } else {
                ptx::mbar_arrive_expect_tx(&kv_full[s], kPageBytes);
                ptx::tma_load_4d(kv + s * kPageBytes, &tm_kv, &kv_full[s], 0, 0, 0, phys,
                                 pol_stream);
              }
              // Two-stage ring (576 record): the page that reuses this stage next goes to
              // L2 now; its load is issued only when this page's PV has freed the stage, and
              // then reads L2, not HBM (B=16, ctx 64K, Hq=16: 281.5 -> 274.1 us). The
              // four-stage ring of the 320 record hides the latency already.
              if constexpr (KS == 2) {
                const int pf = base_pg + j + KS;
                if (pf < pt.p1) ptx::tma_prefetch_l2_4d(&tm_kv, 0, 0, 0, __ldg(row + pf));
              }
            }
          }
          ok = __shfl_sync(kFullMask, good, 0) != 0;
          if (!ok) break;
        }
      }
      ++u;
    }
    // Leave no copy in flight: the last fill of each stage and of q (bounded).
    if (lane == 0) {
      uint64_t* tma_bar = F8 ? kv_f8 : kv_full;   // completed by the copies themselves
      if (kSep) {
        if (t > 0) {
          const uint64_t t0 = ptx::globaltimer();
          while (!ptx::mbar_try_wait(&kv_f8[0], (t - 1) & 1) &&
                 ptx::globaltimer() - t0 < ptx::kWaitLimitNs) {
          }
        }
      } else {
        for (int k = 1; k <= KS && t - k >= 0; ++k) {
          const int tt = t - k;
          const uint64_t t0 = ptx::globaltimer();
          while (!ptx::mbar_try_wait(&tma_bar[tt % KS], (tt / KS) & 1) &&
                 ptx::globaltimer() - t0 < ptx::kWaitLimitNs) {
          }
        }
      }
      if (u > 0) {
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(q_full, (u - 1) & 1) &&
               ptx::globaltimer() - t0 < ptx::kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ============================== MMA issuer ==============================
    // One thread polls for whichever MMA group is ready and issues it: the scores of
    // the next page (its data, q and an S^T buffer are ready) or the PV of the oldest
    // page whose P^T is written. PV never waits behind the next page's load, so the
    // stage it frees is refilled as early as possible. The polls are non-blocking tests
    // (a try_wait may suspend the thread while another group is ready).
    constexpr uint32_t kIdQK = ptx::umma_idesc_f16(64, N, 0, 0, kBf16);
    constexpr uint32_t kIdPV = ptx::umma_idesc_f16(128, N, 1, 1, kBf16);
    const uint32_t kv_s = ptx::smem_addr(kv);
    const uint32_t q_s = ptx::smem_addr(qs);
    int t_qk = 0, t_pv = 0;   // next page to score / to apply
    if (lane == 0) {
      int u = 0, i = 0, npg = 0;
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
          const int s = t_qk & 1;          // S^T buffer
          const int kst = t_qk % KS;       // ring stage
          const bool ready = (!need_q || ptx::mbar_test_wait(F8 ? q_cvt : q_full, u & 1)) &&
                             ptx::mbar_test_wait(&kv_full[kst], (t_qk / KS) & 1) &&
                             (t_qk < 2 || ptx::mbar_test_wait(&s_free[s], ((t_qk >> 1) - 1) & 1));
          if (ready) {
            need_q = false;
            ptx::tc_fence_after();
            const uint32_t st = kv_s + kst * kPageBytes;
#pragma unroll
            for (int kb = 0; kb < kSubTiles; ++kb) {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint64_t a = ptx::umma_desc_sw128(st + kb * kSubBytes + ks * 32, 16, 1024);
                const uint64_t b = ptx::umma_desc_sw128(q_s + kb * (N * 128) + ks * 32, 16, 1024);
                ptx::umma_f16(tmem + L::kColS + s * N, a, b, kIdQK, (kb | ks) != 0);
              }
            }
            if (i == npg - 1) {
              ptx::umma_commit(q_empty);
              ++u;
            }
            ptx::umma_commit(&s_full[s]);
            first_bits = (first_bits & ~(1u << (t_qk & 31))) | (uint32_t(i == 0) << (t_qk & 31));
            ++t_qk;
            ++i;
            progress = true;
          }
        }
        if (t_pv < t_qk && ptx::mbar_test_wait(&p_full[t_pv & 1], (t_pv >> 1) & 1)) {
          ptx::tc_fence_after();
          const bool first = (first_bits >> (t_pv & 31)) & 1u;
          const uint32_t st = kv_s + (t_pv % KS) * kPageBytes;
#pragma unroll
          for (int mt = 0; mt < R::kMTiles; ++mt) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t a =
                  ptx::umma_desc_sw128(st + 2 * mt * kSubBytes + ks * 2048, kSubBytes, 1024);
              const uint64_t b =
                  ptx::umma_desc_sw128(st + kRopeSub * kSubBytes + ks * 2048, kSubBytes, 1024);
              ptx::umma_f16(tmem + L::kColO + mt * N, a, b, kIdPV, !(first && ks == 0));
            }
          }
          ptx::umma_commit(&kv_empty[t_pv % KS]);
          ptx::umma_commit(&pv_done[t_pv & 1]);
          ++t_pv;
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
      // Wait (bounded) for the last MMAs before TMEM is released.
      if (t_pv > 0) {
        const int tl = t_pv - 1;
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(&pv_done[tl & 1], (tl >> 1) & 1) &&
               ptx::globaltimer() - t0 < ptx::kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else if (F8 && warp >= 2 + SoftmaxWarps<N>::kWarps) {
    // ============================== E4M3 converters ==============================
    // A page's E4M3 codes land in the upper half of its stage as kSubTiles blocks of
    // [64 tokens][64 bytes]; the converter warps rewrite the stage in place as the 16-bit
    // record the MMAs read: kSubTiles 128-byte-swizzled [64 tokens][64 dims] sub-tiles,
    // the layout the 16-bit cache's TMA map gives. Codes convert exactly to fp16
    // (cvt.rn.f16x2.e4m3x2); the record scale is applied to the scores and the output instead.
    // With the codes in the stage's upper half (the four-stage ring of the 320 record),
    // sub-tile k is written over bytes [8K k, 8K k + 8K), which reach the codes from
    // k = kFirstOverlap on, and there only blocks j <= k: each sub-tile is read into
    // registers first, and from kFirstOverlap on the converters meet at a named barrier
    // between reading and writing, so every block is read before anything overwrites it.
    // The barrier count never depends on an abort, so the warps always meet. (The 576
    // record's two-stage ring keeps the codes in a page of their own instead.)
    constexpr int kCT = 32 * (kConvWarps > 0 ? kConvWarps : 1);
    constexpr int kPer = (kPage * 4) / kCT;      // 16-byte code chunks per thread per sub-tile
    // the first sub-tile whose 16-bit bytes reach the codes in the stage's upper half
    constexpr int kFirstOverlap = (kPageBytes / 2) / kSubBytes;
    const int ct = threadIdx.x - SoftmaxWarps<N>::kThreads;
    bool aborted = false;
    int t = 0, u = 0;
    while (walk.g < g_hi) {
      const Portion pt = walker_next(walk, spec, g_hi);
      // this piece's q in the MMAs' type: bf16 -> fp16 in place (16 bytes at a time)
      if (!aborted && !bounded_wait(q_full, u & 1, flags, p.err)) aborted = true;
      if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        if (!aborted) {
          for (int i = ct; i < L::kQBytes / 16; i += kCT) {
            uint4* w = reinterpret_cast<uint4*>(qs) + i;
            uint4 v = *w;
            uint32_t* e = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float lo = __uint_as_float(e[k] << 16), hi = __uint_as_float(e[k] & 0xffff0000u);
              e[k] = ptx::Mma<__half>::pack(lo, hi);
            }
            *w = v;
          }
        }
      }
      ptx::fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(q_cvt);
      ++u;
      for (int i = pt.p0; i < pt.p1; ++i, ++t) {
        const int s = t % KS;
        if (kSep) {
          // the page's codes have landed, and the ring stage is free (PV of page t - KS)
          if (!aborted && !bounded_wait(&kv_f8[0], t & 1, flags, p.err)) aborted = true;
          if (!aborted && !bounded_wait(&kv_empty[s], ((t / KS) & 1) ^ 1, flags, p.err))
            aborted = true;
        } else if (!aborted && !bounded_wait(&kv_f8[s], (t / KS) & 1, flags, p.err)) {
          aborted = true;
        }
        uint8_t* stg = kv + s * kPageBytes;
        const uint8_t* codes = kSep ? codes_buf : stg + kPageBytes / 2;
#pragma unroll 1
        for (int k = 0; k < kSubTiles; ++k) {
          uint4 x[kPer];
#pragma unroll
          for (int c = 0; c < kPer; ++c) {
            const int idx = ct + c * kCT;          // row idx / 4, 16-byte piece idx % 4
            x[c] = aborted ? make_uint4(0u, 0u, 0u, 0u)
                           : *reinterpret_cast<const uint4*>(codes + k * (kPage * 64) +
                                                             (idx >> 2) * 64 + (idx & 3) * 16);
          }
          if (!kSep && k >= kFirstOverlap) ptx::named_barrier_sync(2, kCT);
#pragma unroll
          for (int c = 0; c < kPer; ++c) {
            const int idx = ct + c * kCT;
            const int r = idx >> 2, m = idx & 3;
            uint4 w0, w1;
            ptx::e4m3x4_to_f16x2(x[c].x, w0.x, w0.y);
            ptx::e4m3x4_to_f16x2(x[c].y, w0.z, w0.w);
            ptx::e4m3x4_to_f16x2(x[c].z, w1.x, w1.y);
            ptx::e4m3x4_to_f16x2(x[c].w, w1.z, w1.w);
            uint8_t* row = stg + k * kSubBytes + r * 128;
            *reinterpret_cast<uint4*>(row + (((2 * m) ^ (r & 7)) << 4)) = w0;
            *reinterpret_cast<uint4*>(row + (((2 * m + 1) ^ (r & 7)) << 4)) = w1;
          }
        }
        ptx::fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
          if (kSep) ptx::mbar_arrive(&kv_f8[1]);   // the code page may be refilled
          ptx::mbar_arrive(&kv_full[s]);
        }
      }
    }
  } else {
    // ============================== softmax / epilogue warps ==============================
    constexpr int kSW = SoftmaxWarps<N>::kWarps;
    constexpr int NC = SoftmaxWarps<N>::kCols;   // head columns this thread owns
    constexpr int kST = 32 * kSW;                // softmax threads
    const int sw = warp - 2;               // 0 .. kSW-1
    const int sp = warp & 3;               // TMEM sub-partition of this warp
    const int cb = (sw / 4) * NC;          // first head column of this warp
    const bool active = lane < 16;         // M=64 scores: rows in lanes 0..15 of each sub-partition
    const int row = 16 * sp + lane;        // token within the page (active lanes)
    const int ctid = threadIdx.x - 64;     // 0 .. kST-1
    const uint32_t t_lane = tmem + (uint32_t(32 * sp) << 16);
    T* outg = static_cast<T*>(p.out);
    // per head: the sum of the weights (for the LSE) and the sum of the weights as
    // rounded for the PV product (O is divided by the latter, so the output is a convex
    // combination of value rows whatever the rounding of P)
    float l_reg[NC], lq_reg[NC];
    bool aborted = false;
    int t = 0;

    // this thread's NC scaled scores (or -inf): NC/16 TMEM loads behind one wait
    auto load_scores = [&](bool valid, float (&x)[NC]) {
      if (!aborted) {
#pragma unroll
        for (int c = 0; c < NC; c += 16)
          ptx::tmem_ld16(t_lane + L::kColS + (t & 1) * N + cb + c,
                         *reinterpret_cast<float(*)[16]>(x + c));
        ptx::tmem_ld_wait();
      }
#pragma unroll
      for (int h = 0; h < NC; ++h) x[h] = valid ? x[h] * p.scale_log2 : -INFINITY;
    };
    // exact per-head maximum over the page's 64 tokens -> red[h*4 + sub-partition]
    auto column_max = [&](const float (&x)[NC]) {
#pragma unroll
      for (int h = 0; h < NC; ++h) {
        float v = x[h];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, o));
        if (lane == (h & 31)) red[(cb + h) * 4 + sp] = v;
      }
      ptx::named_barrier_sync(1, kST);
    };

    while (walk.g < g_hi) {
      const Portion pt = walker_next(walk, spec, g_hi);
      const int npg = pt.p1 - pt.p0;
      const int ctx = __ldg(p.context_lens + pt.b);
#pragma unroll
      for (int h = 0; h < NC; ++h) l_reg[h] = lq_reg[h] = 0.f;

      for (int i = 0; i < npg; ++i, ++t) {
        if (!aborted && !bounded_wait(&s_full[t & 1], (t >> 1) & 1, flags, p.err)) aborted = true;
        aborted = __any_sync(kFullMask, aborted);  // keep .sync.aligned TMEM accesses warp-uniform
        ptx::tc_fence_after();
        const int token = (pt.p0 + i) * kPage + row;
        const bool valid = active && token < ctx && !aborted;
        float x[NC];
        load_scores(valid, x);
        // causal rows (S > 1): row R = i*Hq + h of the sequence (R = seg*N + column),
        // query token i, sees tokens [0, ctx - S + 1 + i). Token ctx - S + 1 + k is hidden
        // from the rows of query tokens 0..k, i.e. rows R < (k + 1) * Hq.
        if (valid && token >= ctx - p.seq_len_q + 1) {
          const int cut = (token - (ctx - p.seq_len_q)) * p.num_q_heads - pt.seg * N - cb;
#pragma unroll
          for (int h = 0; h < NC; ++h)
            if (h < cut) x[h] = -INFINITY;
        }
        if (i == 0) {
          // first page of the piece: the running maximum starts at the exact column maximum
          column_max(x);
          if (ctid < N) {
            const float4 r = *reinterpret_cast<const float4*>(red + ctid * 4);
            mused[ctid] = fmaxf(fmaxf(r.x, r.y), fmaxf(r.z, r.w));
          }
          ptx::named_barrier_sync(1, kST);
        } else {
          // lazy maximum: only if a score exceeds the maximum in use by 2^8 is it raised
          bool need = false;
#pragma unroll
          for (int c = 0; c < NC; c += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(mused + cb + c);
            need |= (x[c] > m4.x + kRescaleLog2) | (x[c + 1] > m4.y + kRescaleLog2) |
                    (x[c + 2] > m4.z + kRescaleLog2) | (x[c + 3] > m4.w + kRescaleLog2);
          }
          const bool wneed = __any_sync(kFullMask, need);
          if (lane == 0) flags[2 + sw] = wneed ? 1 : 0;
          ptx::named_barrier_sync(1, kST);
          int any = 0;
#pragma unroll
          for (int k = 0; k < kSW; ++k) any |= flags[2 + k];
          ptx::named_barrier_sync(1, kST);
          if (any) {
            column_max(x);
            if (ctid < N) {
              const float4 r = *reinterpret_cast<const float4*>(red + ctid * 4);
              const float mo = mused[ctid];
              const float mn = fmaxf(mo, fmaxf(fmaxf(r.x, r.y), fmaxf(r.z, r.w)));
              // a causal row that has seen no token yet has nothing to rescale
              alpha_s[ctid] = mn == -INFINITY ? 1.f : ptx::exp2_approx(mo - mn);
              mused[ctid] = mn;
            }
            ptx::named_barrier_sync(1, kST);
#pragma unroll
            for (int h = 0; h < NC; ++h) {
              l_reg[h] *= alpha_s[cb + h];
              lq_reg[h] *= alpha_s[cb + h];
            }
            // O^T holds the pages up to t-1: wait for their PV, then rescale it in TMEM
            if (!aborted && !bounded_wait(&pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, flags, p.err))
              aborted = true;
            aborted = __any_sync(kFullMask, aborted);
            ptx::tc_fence_after();
            if (!aborted) {
#pragma unroll
              for (int mt = 0; mt < R::kMTiles; ++mt) {
#pragma unroll
                for (int c = 0; c < NC; c += 16) {
                  float v[16];
                  const uint32_t a = t_lane + L::kColO + mt * N + cb + c;
                  ptx::tmem_ld16(a, v);
                  ptx::tmem_ld_wait();
#pragma unroll
                  for (int e = 0; e < 16; ++e) v[e] *= alpha_s[cb + c + e];
                  ptx::tmem_st16(a, v);
                }
              }
              ptx::tmem_st_wait();
            }
          }
        }
        // P^T row `row` (heads contiguous) over the page's rope sub-tile
        uint8_t* pbuf = kv + (t % KS) * kPageBytes + kRopeSub * kSubBytes;
#pragma unroll
        for (int c = 0; c < NC; c += 8) {
          const float4 ma = *reinterpret_cast<const float4*>(mused + cb + c);
          const float4 mb = *reinterpret_cast<const float4*>(mused + cb + c + 4);
          const float mm[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
          float pv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            // m = -inf: a causal row with no token seen yet, whose scores are all -inf
            pv[e] = ptx::exp2_approx(x[c + e] - (mm[e] == -INFINITY ? 0.f : mm[e]));
            l_reg[c + e] += pv[e];
          }
          uint4 w;
          w.x = ptx::Mma<TM>::pack(pv[0], pv[1]);
          w.y = ptx::Mma<TM>::pack(pv[2], pv[3]);
          w.z = ptx::Mma<TM>::pack(pv[4], pv[5]);
          w.w = ptx::Mma<TM>::pack(pv[6], pv[7]);
          {
            float r[8];
            ptx::Mma<TM>::unpack(w.x, r[0], r[1]);
            ptx::Mma<TM>::unpack(w.y, r[2], r[3]);
            ptx::Mma<TM>::unpack(w.z, r[4], r[5]);
            ptx::Mma<TM>::unpack(w.w, r[6], r[7]);
#pragma unroll
            for (int e = 0; e < 8; ++e) lq_reg[c + e] += r[e];
          }
          if (active) {
            const int chunk = (cb + c) / 8;
            *reinterpret_cast<uint4*>(pbuf + row * 128 + ((chunk ^ (row & 7)) << 4)) = w;
          }
        }
        // Slots past ctx in the last page: their P is 0, but 0 * (whatever the slot holds,
        // NaN included) must not reach O, so their V rows are cleared before the PV MMA
        // (the score MMA has already consumed the page). The warps of a sub-partition
        // split the latent sub-tiles.
        if (active && token >= ctx) {
          uint8_t* stg = kv + (t % KS) * kPageBytes;
          constexpr int kSubPerWarp = (kDv / 64) / (kSW / 4);
#pragma unroll
          for (int k = 0; k < kSubPerWarp; ++k) {
            const int sub = (sw / 4) * kSubPerWarp + k;
            uint4* r = reinterpret_cast<uint4*>(stg + sub * kSubBytes + row * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) r[c] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        ptx::tc_fence_before();
        ptx::fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(&s_free[t & 1]);   // S^T buffer has been read
          ptx::mbar_arrive(&p_full[t & 1]);   // P^T is in shared memory
        }
      }

      // ---- end of the piece: softmax denominators, then O = O^T / l
#pragma unroll
      for (int h = 0; h < NC; ++h) {
        float v = l_reg[h];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) v += __shfl_xor_sync(kFullMask, v, o);
        if (lane == (h & 31)) red[(cb + h) * 4 + sp] = v;
      }
      ptx::named_barrier_sync(1, kST);
      if (ctid < N) {
        const float4 r = *reinterpret_cast<const float4*>(red + ctid * 4);
        ltot[ctid] = (r.x + r.y) + (r.z + r.w);
      }
      ptx::named_barrier_sync(1, kST);
#pragma unroll
      for (int h = 0; h < NC; ++h) {
        float v = lq_reg[h];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) v += __shfl_xor_sync(kFullMask, v, o);
        if (lane == (h & 31)) red[(cb + h) * 4 + sp] = v;
      }
      ptx::named_barrier_sync(1, kST);
      if (ctid < N) {
        const float4 r = *reinterpret_cast<const float4*>(red + ctid * 4);
        lqtot[ctid] = (r.x + r.y) + (r.z + r.w);
      }
      ptx::named_barrier_sync(1, kST);
      if (!aborted && !bounded_wait(&pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, flags, p.err))
        aborted = true;
      aborted = __any_sync(kFullMask, aborted);
      ptx::tc_fence_after();

      const bool whole = (pt.p0 == 0 && pt.p1 == pt.np);
      const int slot = piece_slot(pt.seg_start, g_lo);
      const int64_t head0 = int64_t(pt.b) * p.rows_per_seq + int64_t(pt.seg) * N;
      // lse is [B][Hq][S]: row R = i*Hq + h of the sequence goes to (b*Hq + h)*S + i
      auto lse_at = [&](int r) {
        const int R = pt.seg * N + r;
        const int qi = R / p.num_q_heads;
        return (int64_t(pt.b) * p.num_q_heads + (R - qi * p.num_q_heads)) * p.seq_len_q + qi;
      };
      const int64_t slot_row = (int64_t(blockIdx.x) * 2 + slot) * N;
#pragma unroll
      for (int mt = 0; mt < R::kMTiles; ++mt) {
        const int d = mt * 128 + 32 * sp + lane;
#pragma unroll
        for (int c = 0; c < NC; c += 16) {
          float v[16];
          if (!aborted) {
            ptx::tmem_ld16(t_lane + L::kColO + mt * N + cb + c, v);
            ptx::tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = 0.f;
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int h = cb + c + e;
            // ltot = 0 only for a causal row that saw no token of a split piece: O = 0
            const float o = ltot[h] > 0.f ? v[e] * p.v_scale / lqtot[h] : 0.f;
            if (whole)
              outg[(head0 + h) * kDv + d] = from_f32<T>(o);
            else
              __stcg(p.part_out + (slot_row + h) * kDv + d, o);
          }
        }
      }
      if (ctid < N) {
        const float lse_nat =
            ltot[ctid] > 0.f ? (mused[ctid] + log2f(ltot[ctid])) * kLn2 : -INFINITY;
        if (whole) {
          if (p.lse != nullptr) p.lse[lse_at(ctid)] = lse_nat;
        } else {
          __stcg(p.part_lse + slot_row + ctid, lse_nat);
        }
      }
      ptx::tc_fence_before();

      if (!whole) {
        // few pieces: the last to arrive merges them here; many: the split-merge kernel
        const int64_t c0 = pt.seg_start / p.tiles_per_cta;
        const int64_t c1 = (pt.seg_start + pt.np - 1) / p.tiles_per_cta;
        const int pieces = int(c1 - c0 + 1);
        if (pieces <= p.heavy_min) {
          __threadfence();
          ptx::named_barrier_sync(1, kST);
          int32_t* counter = p.counters + int64_t(pt.b) * p.groups + pt.seg;
          if (ctid == 0) {
            const int prev = aborted ? -1 : atomicAdd(counter, 1);
            flags[1] = (prev == pieces - 1) ? 1 : 0;
          }
          ptx::named_barrier_sync(1, kST);
          if (flags[1]) {
            __threadfence();
            for (int idx = ctid; idx < N * (kDv / 4); idx += kST) {
              const int j = idx / (kDv / 4);
              const int dq = idx - j * (kDv / 4);
              float mx = -INFINITY;
              for (int64_t c = c0; c <= c1; ++c) {
                const int sl = (c == c0 && pt.seg_start > c * p.tiles_per_cta) ? 1 : 0;
                mx = fmaxf(mx, __ldcg(p.part_lse + (c * 2 + sl) * N + j));
              }
              float den = 0.f;
              float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int64_t c = c0; c <= c1; ++c) {
                const int sl = (c == c0 && pt.seg_start > c * p.tiles_per_cta) ? 1 : 0;
                const int64_t rowi = (c * 2 + sl) * N + j;
                const float wgt = ptx::exp2_approx((__ldcg(p.part_lse + rowi) - mx) * kLog2e);
                const float4 o = __ldcg(reinterpret_cast<const float4*>(p.part_out + rowi * kDv) + dq);
                den += wgt;
                acc.x += wgt * o.x; acc.y += wgt * o.y; acc.z += wgt * o.z; acc.w += wgt * o.w;
              }
              const float inv = 1.f / den;
              T* o = outg + (head0 + j) * kDv + dq * 4;
              o[0] = from_f32<T>(acc.x * inv);
              o[1] = from_f32<T>(acc.y * inv);
              o[2] = from_f32<T>(acc.z * inv);
              o[3] = from_f32<T>(acc.w * inv);
              if (dq == 0 && p.lse != nullptr) p.lse[lse_at(j)] = mx + logf(den);
            }
            if (ctid == 0) atomicExch(counter, 0);
          }
        }
      }
      ptx::named_barrier_sync(1, kST);
    }
  }

  // ---- teardown: everyone done with TMEM before it is released
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::kTmemCols);
  }
}

}  // namespace

// ------------------------------------------------------------------ host side
namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn mla_encode_fn() {
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

}  // namespace

bool encode_mla_maps(CUtensorMap* tq, CUtensorMap* tkv, const void* q, int64_t rows, int n,
                     const void* kv, int64_t num_blocks, bool bf16, int dqk) {
  EncodeTiledFn fn = mla_encode_fn();
  if (fn == nullptr) return false;
  const CUtensorMapDataType dt =
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint32_t kSubTiles = cuuint32_t(dqk / 64);
  const cuuint64_t kDqk = cuuint64_t(dqk);
  const cuuint64_t qdims[3] = {64, cuuint64_t(rows), kSubTiles};
  const cuuint64_t qstr[2] = {kDqk * 2, 128};
  const cuuint32_t qbox[3] = {64, cuuint32_t(n), kSubTiles};
  const cuuint32_t e3[3] = {1, 1, 1};
  if (fn(tq, dt, 3, const_cast<void*>(q), qdims, qstr, qbox, e3, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  const cuuint64_t kdims[4] = {64, kPage, kSubTiles, cuuint64_t(num_blocks)};
  const cuuint64_t kstr[3] = {kDqk * 2, 128, cuuint64_t(kPage) * kDqk * 2};
  const cuuint32_t kbox[4] = {64, kPage, kSubTiles, 1};
  const cuuint32_t e4[4] = {1, 1, 1, 1};
  return fn(tkv, dt, 4, const_cast<void*>(kv), kdims, kstr, kbox, e4,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 record cache [blocks, 64, dqk] bytes: dims (d mod 64, slot, d / 64, block), box
// (64, 64, S, 1), no swizzle: S blocks of [64 tokens][64 bytes] per page.
bool encode_mla_cache_f8(CUtensorMap* tkv, const void* kv, int64_t num_blocks, int dqk) {
  EncodeTiledFn fn = mla_encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t kDqk = cuuint64_t(dqk);
  const cuuint64_t kdims[4] = {64, kPage, cuuint64_t(dqk / 64), cuuint64_t(num_blocks)};
  const cuuint64_t kstr[3] = {kDqk, 64, cuuint64_t(kPage) * kDqk};
  const cuuint32_t kbox[4] = {64, kPage, cuuint32_t(dqk / 64), 1};
  const cuuint32_t e4[4] = {1, 1, 1, 1};
  return fn(tkv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(kv), kdims, kstr, kbox, e4,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <int N, int DQK, typename T, bool F8>
int launch_mla_n(const CUtensorMap& tq, const CUtensorMap& tkv, const MlaParams& prm, int grid,
                 cudaStream_t stream) {
  auto kern = mla_decode_kernel<N, DQK, T, F8>;
  using L = MlaLayout<N, DQK, F8>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  kern<<<grid, Roles<N, F8>::kThreads, L::kSmem, stream>>>(tq, tkv, prm);
  return cudaGetLastError();
}

template <int DQK, typename T>
int launch_mla_t(int n, bool f8, const CUtensorMap& tq, const CUtensorMap& tkv,
                 const MlaParams& prm, int grid, cudaStream_t s) {
  if (f8)   // E4M3 caches: groups of 16 or 32 rows (mla_supported)
    return n == 16 ? launch_mla_n<16, DQK, T, true>(tq, tkv, prm, grid, s)
                   : launch_mla_n<32, DQK, T, true>(tq, tkv, prm, grid, s);
  switch (n) {
    case 16: return launch_mla_n<16, DQK, T, false>(tq, tkv, prm, grid, s);
    case 32: return launch_mla_n<32, DQK, T, false>(tq, tkv, prm, grid, s);
    default: return launch_mla_n<64, DQK, T, false>(tq, tkv, prm, grid, s);
  }
}

template <typename T>
int launch_mla_dt(int dqk, int n, bool f8, const CUtensorMap& tq, const CUtensorMap& tkv,
                  const MlaParams& prm, int grid, cudaStream_t s) {
  return dqk == 320 ? launch_mla_t<320, T>(n, f8, tq, tkv, prm, grid, s)
                    : launch_mla_t<576, T>(n, f8, tq, tkv, prm, grid, s);
}

}  // namespace

int mla_heads_per_cta(const pda_problem& p) {
  if (p.seq_len_q > 1) {
    const int64_t rows = int64_t(p.seq_len_q) * p.num_q_heads;
    if (rows <= 64) return int(rows);          // all rows of a sequence in one group
    // groups of one query token's heads: 128 on the heads-on-M and two-CTA kernels
    return (mla_uses_rows(p) || mla_uses_pairs(p)) ? 128 : 64;
  }
  if (mla_uses_pairs(p)) return 128;   // one 128-head group per CTA pair
  if (mla_uses_rows(p)) return 128;    // one 128-head group per CTA, heads on M
  return p.num_q_heads <= 64 ? p.num_q_heads : 64;
}
int mla_ctas_per_sm(const pda_problem&) { return 1; }

bool mla_supported(const pda_problem& p, std::string* why) {
  if (p.kv_format == PDA_KV_FP8_E4M3) {
    const int64_t rows = int64_t(p.seq_len_q > 1 ? p.seq_len_q : 1) * p.num_q_heads;
    if (rows != 16 && rows != 32) {
      *why = "MLA decode over E4M3 caches supports seq_len_q * num_q_heads in {16, 32}";
      return false;
    }
  } else if (p.kv_format != PDA_KV_SAME_AS_Q) {
    *why = "MLA decode supports 16-bit or E4M3 caches";
    return false;
  }
  if (p.seq_len_q > 1) {
    const int64_t rows = int64_t(p.seq_len_q) * p.num_q_heads;
    if (!(rows == 16 || rows == 32 || rows == 64 || (rows > 64 && p.num_q_heads % 64 == 0))) {
      *why = "MLA decode of several query tokens needs seq_len_q * num_q_heads in {16, 32, 64} "
             "or num_q_heads a multiple of 64";
      return false;
    }
  }
  if (!((p.head_dim_qk == 576 && p.head_dim_v == 512) ||
        (p.head_dim_qk == 320 && p.head_dim_v == 256))) {
    *why = "MLA decode supports (head_dim_qk, head_dim_v) = (576, 512) or (320, 256)";
    return false;
  }
  if (p.page_size != kPage) {
    *why = "MLA decode supports page_size 64";
    return false;
  }
  if (p.num_kv_heads != 1) {
    *why = "MLA decode has one shared latent head (num_kv_heads must be 1)";
    return false;
  }
  const int n = mla_heads_per_cta(p);
  if (!(n == 16 || n == 32 || n == 64 || n == 128) ||
      (p.seq_len_q <= 1 && p.num_q_heads % n != 0)) {
    *why = "MLA decode supports num_q_heads 16, 32 or a multiple of 64";
    return false;
  }
  if (p.num_blocks > INT32_MAX) {
    *why = "num_blocks must fit in int32 (block-table entries are int32)";
    return false;
  }
  return true;
}

int launch_mla_decode(const Plan& plan, const MlaArgs& a, const Workspace& ws, void* stream) {
  if (plan.cluster == 2) return launch_mla_pair(plan, a, ws, stream);
  if (mla_uses_rows(plan.prob)) return launch_mla_rows(plan, a, ws, stream);
  const pda_problem& pr = plan.prob;
  const bool bf16 = pr.dtype == PDA_BF16;
  const bool f8 = pr.kv_format == PDA_KV_FP8_E4M3;
  const int n = plan.group;
  CUtensorMap m[2];
  const int sq = pr.seq_len_q > 1 ? pr.seq_len_q : 1;
  if (!plan.map_cache.get(a.q, a.kv_cache, m, nullptr, [&](CUtensorMap* t, int32_t*) {
        return encode_mla_maps(&t[0], &t[1], a.q, int64_t(pr.batch) * sq * pr.num_q_heads, n,
                               a.kv_cache, pr.num_blocks, bf16, pr.head_dim_qk) &&
               (!f8 || encode_mla_cache_f8(&t[1], a.kv_cache, pr.num_blocks, pr.head_dim_qk));
      }))
    return -1;
  const CUtensorMap& tq = m[0];
  const CUtensorMap& tkv = m[1];
  MlaParams prm{};
  prm.q = a.q;
  prm.out = a.out;
  prm.lse = a.lse;
  prm.block_tables = a.block_tables;
  prm.context_lens = a.context_lens;
  prm.batch = pr.batch;
  prm.num_q_heads = pr.num_q_heads;
  prm.rows_per_seq = sq * pr.num_q_heads;
  prm.seq_len_q = sq;
  prm.groups = plan.segs_per_seq;
  prm.max_blocks = pr.max_blocks_per_seq;
  prm.num_blocks = pr.num_blocks;
  prm.scale_log2 = a.scale * a.kv_scale * kLog2e;
  prm.v_scale = a.kv_scale;
  prm.total_tiles = plan.total_tiles;
  prm.tiles_per_cta = plan.tiles_per_cta;
  prm.heavy_min = plan.heavy_min_pieces;
  prm.err = ws.err;
  prm.counters = ws.counters;
  prm.part_lse = ws.part_lse;
  prm.part_out = ws.part_out;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int dqk = pr.head_dim_qk;
  const int e = bf16 ? launch_mla_dt<__nv_bfloat16>(dqk, n, f8, tq, tkv, prm, plan.num_ctas, s)
                     : launch_mla_dt<__half>(dqk, n, f8, tq, tkv, prm, plan.num_ctas, s);
  if (e != 0) return e;
  return launch_split_merge(plan, ws, a.out, a.lse, stream);
}

}  // namespace pda
