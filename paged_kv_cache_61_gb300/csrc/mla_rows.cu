// Absorbed-MLA decode of the 320-wide record (kv_lora_rank 256: 256 latent + 64 rope,
// V = the first 256) for head groups of 128, with the heads on the MMA's M axis.
//
// What it computes: as the 64-head kernel ("From MHA to MLA", section 6; FlashMLA-ETAP
// "Supported configurations", (320, 256)): score(h, j) = scale * <q_h, rec_j>, value
// rec_j[:256], output [B, Hq, 256] and fp32 LSE. With S query tokens (FlashMLA-ETAP
// "Usage": seq_len_q, causal) a group holds the 128 heads of one token i, which sees
// tokens [0, ctx - S + 1 + i); q and out are [B, S, Hq, .], lse [B, Hq, S].
//
// How: the 320-wide record lets one SM hold a whole 128-head group, so every page is
// read once (the 64-head kernel splits 128 heads into two groups that each read it):
//  * Warp 0 streams 64-token pages (five 128-byte-swizzled [64][64] sub-tiles, 40 KB)
//    into a 5-stage ring.
//  * Warp 1 issues from one thread S[128 heads x 64 tokens] = q * K^T (20 MMAs M=128,
//    N=64, K=16) and O[128 x 256] += P * V (4 MMAs M=128, N=256, V read in place from the
//    page's first four sub-tiles, MN-major). q and P, the A operands, sit in tensor
//    memory, which leaves shared memory (80 KB of q, 16 KB of P) to the page ring; the
//    MMAs take as long with A in shared memory.
//  * Warps 2-5 own one head each per thread (TMEM lane = head). At the start of a piece
//    each thread puts its head's q row into tensor memory. Per page the row's 64 scores
//    come out of TMEM, the online softmax runs in the thread without any reduction (lazy
//    maximum: raised, and O rescaled in TMEM, only when a score exceeds the maximum in
//    use by 2^8) and the P row goes back to TMEM. At the end of a piece the thread
//    normalises its O row and writes it out, or writes a split piece merged like the
//    other kernels' pieces.
// TMEM (32-bit columns, 16-bit operands packed in pairs): q [0, 160), S [160, 224),
// P [224, 256), O [256, 512).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "mla_maps.h"
#include "pda_internal.h"
#include "ptx.cuh"
#include "ptx_ext.cuh"
#include "ptx_cluster.cuh"
#include "tile_walk.cuh"

namespace pda {
namespace {

constexpr int kRows = 128;                 // heads of a group = TMEM lanes = MMA M
constexpr int kPage = 64;
constexpr int kDqk = 320;
constexpr int kDv = 256;
constexpr int kSub = kDqk / 64;            // five 64-dim sub-tiles per record
constexpr int kSubBytes = kPage * 128;     // [64 tokens][64 dims] x 16 bit
constexpr int kPageBytes = kSub * kSubBytes;
constexpr int kStages = 5;
constexpr int kSoftWarps = 4;
constexpr int kThreads = (2 + kSoftWarps) * 32;
constexpr int kST = kSoftWarps * 32;
constexpr int kColQ = 0;                   // q row: 320 dims in 160 columns
constexpr int kColS = kColQ + kDqk / 2;    // S row: 64 fp32 scores
constexpr int kColP = kColS + kPage;       // P row: 64 tokens in 32 columns
constexpr int kColO = kColP + kPage / 2;   // O row: 256 fp32
constexpr int kTmemCols = 512;
static_assert(kColO + kDv == kTmemCols, "q, S, P and O fill the 512 columns");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;

// shared memory (offsets from a 1024-byte aligned base)
constexpr int kOffKV = 0;
constexpr int kOffBar = kOffKV + kStages * kPageBytes;
constexpr int kBarCount = 2 * kStages + 11;
constexpr int kSmem = 1024 + kOffBar + kBarCount * 8 + 64;
static_assert(kSmem <= 232448, "fits the 227 KB of dynamic shared memory per block");

struct RowsParams {
  const void* q;
  void* out;
  float* lse;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t batch, num_q_heads, groups, max_blocks;
  // S query tokens per sequence: its S*Hq rows (row R = i*Hq + h) are contiguous in q and
  // out, in groups of 128 rows (128 heads of one token; S*Hq / 128 groups per sequence)
  int32_t rows_per_seq, seq_len_q;
  int64_t num_blocks;
  float scale_log2;
  int64_t total_tiles, tiles_per_cta;
  int32_t heavy_min;
  int32_t* err;
  int32_t* counters;
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

template <typename T>
__device__ __forceinline__ T cvt_out(float x);
template <>
__device__ __forceinline__ __half cvt_out<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 cvt_out<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    mla_rows_kernel(const __grid_constant__ CUtensorMap tm_kv, const RowsParams p) {
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* kv = base + kOffKV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kOffBar);
  // Page t sits in ring stage t % kStages.
  uint64_t* kv_full = bars + 0;                // [kStages]
  uint64_t* kv_empty = bars + kStages;         // [kStages]
  uint64_t* q_full = bars + 2 * kStages;   // the piece's q rows are in TMEM
  // Barriers completing once per page come in pairs indexed by page parity, so a waiter is
  // never two phases behind.
  uint64_t* s_full = q_full + 1;    // [2] S written by the score MMAs
  uint64_t* s_free = q_full + 3;    // [2] S read by the four softmax warps
  uint64_t* p_full = q_full + 5;    // [2] P written, O rows rescaled
  uint64_t* pv_done = q_full + 7;   // [2] PV of a page completed
  volatile int* flags = reinterpret_cast<volatile int*>(q_full + 9);  // [0] abort, [1] last piece
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_full + 10);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t g_lo = int64_t(blockIdx.x) * p.tiles_per_cta;
  const int64_t g_hi = min(p.total_tiles, g_lo + p.tiles_per_cta);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (g_lo >= g_hi) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&kv_full[s], 1);
      ptx::mbar_init(&kv_empty[s], 1);
    }
    ptx::mbar_init(q_full, kSoftWarps);
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&s_full[b], 1);
      ptx::mbar_init(&s_free[b], kSoftWarps);
      ptx::mbar_init(&p_full[b], kSoftWarps);
      ptx::mbar_init(&pv_done[b], 1);
    }
    flags[0] = 0;
    flags[1] = 0;
    ptx::fence_mbarrier_init();
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const WalkSpec spec{p.context_lens, p.batch, p.groups, kPage};
  Walker walk;
  walker_init(walk, spec, g_lo, lane);

  if (warp == 0) {
    // ============================== TMA producer ==============================
    if (lane == 0) ptx::prefetch_tensormap(&tm_kv);
    const uint64_t pol_stream = ptx::policy_evict_first();
    int t = 0;
    bool ok = true;
    while (ok && walk.g < g_hi) {
      const Portion pt = walker_next(walk, spec, g_hi);
      const int32_t* row = p.block_tables + int64_t(pt.b) * p.max_blocks;
      for (int base_pg = pt.p0; ok && base_pg < pt.p1; base_pg += 32) {
        const int32_t ids = (base_pg + lane < pt.p1) ? __ldg(row + base_pg + lane) : 0;
        const int n = min(32, pt.p1 - base_pg);
        for (int j = 0; j < n; ++j, ++t) {
          const int32_t phys = __shfl_sync(kFullMask, ids, j);
          int good = 1;
          if (lane == 0) {
            const int s = t % kStages;
            if (!bounded_wait(&kv_empty[s], ((t / kStages) & 1) ^ 1, flags, p.err)) {
              good = 0;
            } else {
              // an entry outside the pool is flagged; the copy of an out-of-range block
              // reads the map's zero fill
              if (phys < 0 || int64_t(phys) >= p.num_blocks) atomicOr(p.err, 1);
              ptx::mbar_arrive_expect_tx(&kv_full[s], kPageBytes);
              ptx::tma_load_4d(kv + s * kPageBytes, &tm_kv, &kv_full[s], 0, 0, 0, phys,
                               pol_stream);
            }
          }
          ok = __shfl_sync(kFullMask, good, 0) != 0;
          if (!ok) break;
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
    // One thread issues whichever MMA group is ready, PV first: the PV of the oldest page
    // whose P is written, the scores of the next page (its data and q ready, the previous
    // page's S read). The MMAs of a group go out back to back: any other work between
    // them (a barrier test costs about as much as an MMA) leaves the tensor pipe idle.
    constexpr uint32_t kIdQK = ptx::umma_idesc_f16(kRows, kPage, 0, 0, kBf16);
    constexpr uint32_t kIdPV = ptx::umma_idesc_f16(kRows, kDv, 0, 1, kBf16);
    const uint32_t kv_s = ptx::smem_addr(kv);
    int t_qk = 0, t_pv = 0;   // next page to score / to apply
    if (lane == 0) {
      int u = 0, i = 0, npg = 0;
      bool have = false, need_q = false, qk_done = false;
      uint32_t first_bits = 0;   // bit (t & 31): page t is the first of its piece
      ptx::Watchdog watchdog;
      while (true) {
        bool progress = false;
        // PV first: the softmax of the next page waits for it before writing P
        if (t_pv < t_qk && ptx::mbar_test_wait(&p_full[t_pv & 1], (t_pv >> 1) & 1)) {
          ptx::tc_fence_after();
          const bool first = (first_bits >> (t_pv & 31)) & 1u;
          const uint32_t st = kv_s + (t_pv % kStages) * kPageBytes;
          // O[128 x 256] += P[128 x 64 tokens] * V[64 tokens x 256]; V is the page's
          // first four sub-tiles read MN-major (dims contiguous), 16 tokens per MMA
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t b = ptx::umma_desc_sw128(st + ks * 2048, kSubBytes, 1024);
            ptx::umma_f16_ts(tmem + kColO, tmem + kColP + ks * 8, b, kIdPV, !(first && ks == 0));
          }
          ptx::umma_commit(&kv_empty[t_pv % kStages]);
          ptx::umma_commit(&pv_done[t_pv & 1]);
          ++t_pv;
          progress = true;
        }
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
          const int kst = t_qk % kStages;      // ring stage
          const int tp = t_qk - 1;             // its S must have been read
          const bool ready = (!need_q || ptx::mbar_test_wait(q_full, u & 1)) &&
                             ptx::mbar_test_wait(&kv_full[kst], (t_qk / kStages) & 1) &&
                             (t_qk == 0 || ptx::mbar_test_wait(&s_free[tp & 1], (tp >> 1) & 1));
          if (ready) {
            need_q = false;
            ptx::tc_fence_after();
            const uint32_t st = kv_s + kst * kPageBytes;
            // S[128 heads x 64 tokens] = q[128 x 320] * K[64 x 320]^T, K = 16 per MMA
            // (8 TMEM columns of q, 32 bytes of each K row)
#pragma unroll
            for (int kb = 0; kb < kSub; ++kb) {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint64_t b = ptx::umma_desc_sw128(st + kb * kSubBytes + ks * 32, 16, 1024);
                ptx::umma_f16_ts(tmem + kColS, tmem + kColQ + kb * 32 + ks * 8, b, kIdQK,
                                 (kb | ks) != 0);
              }
            }
            if (i == npg - 1) ++u;
            ptx::umma_commit(&s_full[t_qk & 1]);
            first_bits = (first_bits & ~(1u << (t_qk & 31))) | (uint32_t(i == 0) << (t_qk & 31));
            ++t_qk;
            ++i;
            progress = true;
          }
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
  } else {
    // ============================== softmax / epilogue warps ==============================
    // Thread = one head of the group, on TMEM lane 32 * (warp % 4) + lane.
    const int sp = warp & 3;
    const int h = 32 * sp + lane;
    const int ctid = threadIdx.x - 64;          // 0 .. kST-1
    const uint32_t t_lane = tmem + (uint32_t(32 * sp) << 16);
    T* outg = static_cast<T*>(p.out);
    bool aborted = false;
    int t = 0;

    while (walk.g < g_hi) {
      const Portion pt = walker_next(walk, spec, g_hi);
      const int npg = pt.p1 - pt.p0;
      const int ctx = __ldg(p.context_lens + pt.b);
      // this group's query token qi sees tokens [0, ctx - S + 1 + qi) (all of them, S = 1)
      const int qi = pt.seg * kRows / p.num_q_heads;
      const int lim = ctx - p.seq_len_q + 1 + qi;
      float m = -INFINITY;   // maximum in use (log2 units)
      float l = 0.f;         // softmax denominator relative to m
      // the same sum over the weights as rounded for the PV product: O is divided by it,
      // so the output is a convex combination of value rows whatever the rounding of P
      float lq = 0.f;

      // This head's q row into TMEM (dims 2c, 2c+1 in column c). The MMAs that read the
      // previous piece's q have completed: the previous piece ended waiting for its last PV.
      {
        const uint4* qrow = reinterpret_cast<const uint4*>(
            static_cast<const T*>(p.q) +
            (int64_t(pt.b) * p.rows_per_seq + int64_t(pt.seg) * kRows + h) * kDqk);
#pragma unroll
        for (int c0 = 0; c0 < kDqk / 32; c0 += 5) {
          uint4 v[20];
#pragma unroll
          for (int k = 0; k < 20; ++k) v[k] = __ldg(qrow + 4 * c0 + k);
          if (!aborted) {
#pragma unroll
            for (int k = 0; k < 5; ++k)
              ptx::tmem_st16(t_lane + kColQ + 16 * (c0 + k),
                             *reinterpret_cast<float(*)[16]>(v + 4 * k));
          }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(q_full);
      }

      for (int i = 0; i < npg; ++i, ++t) {
        if (!aborted && !bounded_wait(&s_full[t & 1], (t >> 1) & 1, flags, p.err)) aborted = true;
        aborted = __any_sync(kFullMask, aborted);  // keep .sync.aligned TMEM accesses warp-uniform
        ptx::tc_fence_after();
        float x[kPage];
        if (!aborted) {
#pragma unroll
          for (int c = 0; c < kPage; c += 16)
            ptx::tmem_ld16(t_lane + kColS + c, *reinterpret_cast<float(*)[16]>(x + c));
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < kPage; ++j) x[j] = 0.f;
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&s_free[t & 1]);   // S may be rewritten

        // The row's arithmetic is written for few FMA-pipe instructions (three-input
        // max, paired f32 FMA and add): the MMA-issuing thread shares an SM sub-partition
        // with one of these warps, and FMA-pipe work there slows the MMA issue (a page's
        // MMAs took ~2600 cycles beside the scalar version, 1300 alone).
        // Tokens from lim on get no weight. A page past lim (S > 1: the last page for an
        // earlier query token) leaves the row unchanged with P = 0; once one is, so are the
        // piece's later pages.
        const int nvalid = min(kPage, lim - (pt.p0 + i) * kPage);
        uint32_t pk[kPage / 2];
        float alpha = 1.f;
        if (nvalid <= 0) {
#pragma unroll
          for (int c = 0; c < kPage / 2; ++c) pk[c] = 0u;
        } else {
          const float sc = p.scale_log2;
          // the page's maximum scaled score: scale times the largest raw score (scale >= 0)
          // or the smallest (scale < 0)
          float mr;
          if (nvalid == kPage) {
            if (sc >= 0.f) {
              float a = ptx::max3(x[0], x[1], x[2]), b = ptx::max3(x[3], x[4], x[5]);
#pragma unroll
              for (int j = 6; j < kPage - 2; j += 4) {
                a = ptx::max3(a, x[j], x[j + 1]);
                b = ptx::max3(b, x[j + 2], x[j + 3]);
              }
              mr = ptx::max3(a, b, fmaxf(x[kPage - 2], x[kPage - 1]));
            } else {
              float a = ptx::min3(x[0], x[1], x[2]), b = ptx::min3(x[3], x[4], x[5]);
#pragma unroll
              for (int j = 6; j < kPage - 2; j += 4) {
                a = ptx::min3(a, x[j], x[j + 1]);
                b = ptx::min3(b, x[j + 2], x[j + 3]);
              }
              mr = ptx::min3(a, b, fminf(x[kPage - 2], x[kPage - 1]));
            }
          } else {
            mr = x[0];
#pragma unroll
            for (int j = 1; j < kPage; ++j)
              if (j < nvalid) mr = sc >= 0.f ? fmaxf(mr, x[j]) : fminf(mr, x[j]);
          }
          const float mx = mr * sc;
          // lazy maximum: set on a piece's first page, raised only when a score exceeds the
          // maximum in use by 2^8 (the common factor cancels in O / l)
          const float mn = (i == 0 || mx > m + kRescaleLog2) ? mx : m;
          alpha = i == 0 ? 1.f : ptx::exp2_approx(m - mn);
          m = mn;
          // exponent arguments x * scale - m, two per instruction
          const uint64_t sc2 = ptx::f2_pack(sc, sc);
          const uint64_t nm2 = ptx::f2_pack(-mn, -mn);
#pragma unroll
          for (int j = 0; j < kPage; j += 2)
            ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(x[j], x[j + 1]), sc2, nm2), x[j], x[j + 1]);
          if (nvalid < kPage) {
#pragma unroll
            for (int j = 1; j < kPage; ++j)
              if (j >= nvalid) x[j] = -INFINITY;
          }
          uint64_t sum_a = ptx::f2_pack(0.f, 0.f), sum_b = sum_a, sq_a = sum_a, sq_b = sum_a;
#pragma unroll
          for (int j = 0; j < kPage; j += 4) {
            const float p0 = ptx::exp2_approx(x[j]);
            const float p1 = ptx::exp2_approx(x[j + 1]);
            const float p2 = ptx::exp2_approx(x[j + 2]);
            const float p3 = ptx::exp2_approx(x[j + 3]);
            sum_a = ptx::f2_add(sum_a, ptx::f2_pack(p0, p1));
            sum_b = ptx::f2_add(sum_b, ptx::f2_pack(p2, p3));
            pk[j / 2] = ptx::Mma<T>::pack(p0, p1);
            pk[j / 2 + 1] = ptx::Mma<T>::pack(p2, p3);
            float r0, r1, r2, r3;
            ptx::Mma<T>::unpack(pk[j / 2], r0, r1);
            ptx::Mma<T>::unpack(pk[j / 2 + 1], r2, r3);
            sq_a = ptx::f2_add(sq_a, ptx::f2_pack(r0, r1));
            sq_b = ptx::f2_add(sq_b, ptx::f2_pack(r2, r3));
          }
          float s0, s1, s2, s3;
          ptx::f2_unpack(sum_a, s0, s1);
          ptx::f2_unpack(sum_b, s2, s3);
          l = l * alpha + ((s0 + s1) + (s2 + s3));
          ptx::f2_unpack(sq_a, s0, s1);
          ptx::f2_unpack(sq_b, s2, s3);
          lq = lq * alpha + ((s0 + s1) + (s2 + s3));
        }

        // P and O hold page t-1 until its PV completes (the previous piece's end already
        // waited for it when i == 0).
        if (i > 0) {
          if (!aborted && !bounded_wait(&pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, flags, p.err))
            aborted = true;
          aborted = __any_sync(kFullMask, aborted);
          ptx::tc_fence_after();
          if (!aborted && __any_sync(kFullMask, alpha != 1.f)) {
#pragma unroll 4
            for (int c = 0; c < kDv; c += 16) {
              float v[16];
              ptx::tmem_ld16(t_lane + kColO + c, v);
              ptx::tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] *= alpha;
              ptx::tmem_st16(t_lane + kColO + c, v);
            }
            ptx::tmem_st_wait();
          }
        }
        // this head's P row: tokens 2c, 2c+1 in column c
        if (!aborted) {
          ptx::tmem_st16(t_lane + kColP, *reinterpret_cast<float(*)[16]>(pk));
          ptx::tmem_st16(t_lane + kColP + 16, *reinterpret_cast<float(*)[16]>(pk + 16));
          ptx::tmem_st_wait();
        }
        // Slots from lim on: P is 0 there, but 0 * (whatever a slot past ctx holds, NaN
        // included) must not reach O, so their V rows (the first four sub-tiles) are
        // cleared; the score MMAs have consumed the page.
        if (nvalid < kPage) {
          const int nz = max(nvalid, 0);
          uint8_t* stg = kv + (t % kStages) * kPageBytes;
          const int n16 = (kPage - nz) * (kDv / 8);   // 16-byte pieces to clear
          for (int idx = ctid; idx < n16; idx += kST) {
            const int r = nz + idx / (kDv / 8);
            const int rem = idx % (kDv / 8);
            *reinterpret_cast<uint4*>(stg + (rem >> 3) * kSubBytes + r * 128 + (rem & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
        }
        ptx::tc_fence_before();
        ptx::fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&p_full[t & 1]);
      }

      // ---- end of the piece: O = O / l, written whole or as a split piece
      if (!aborted && !bounded_wait(&pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, flags, p.err))
        aborted = true;
      aborted = __any_sync(kFullMask, aborted);
      ptx::tc_fence_after();

      const bool whole = (pt.p0 == 0 && pt.p1 == pt.np);
      const int slot = piece_slot(pt.seg_start, g_lo);
      const int64_t head0 = int64_t(pt.b) * p.rows_per_seq + int64_t(pt.seg) * kRows;
      // lse is [B][Hq][S]: row R = i*Hq + h of the sequence goes to (b*Hq + h)*S + i
      auto lse_at = [&](int r) {
        const int R = pt.seg * kRows + r;
        const int i = R / p.num_q_heads;
        return (int64_t(pt.b) * p.num_q_heads + (R - i * p.num_q_heads)) * p.seq_len_q + i;
      };
      const int64_t slot_row = (int64_t(blockIdx.x) * 2 + slot) * kRows;
      const float inv = l > 0.f ? 1.f / lq : 0.f;
#pragma unroll 2
      for (int c = 0; c < kDv; c += 16) {
        float v[16];
        if (!aborted) {
          ptx::tmem_ld16(t_lane + kColO + c, v);
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] *= inv;
        if (whole) {
          uint4 w0, w1;
          w0.x = ptx::Mma<T>::pack(v[0], v[1]);
          w0.y = ptx::Mma<T>::pack(v[2], v[3]);
          w0.z = ptx::Mma<T>::pack(v[4], v[5]);
          w0.w = ptx::Mma<T>::pack(v[6], v[7]);
          w1.x = ptx::Mma<T>::pack(v[8], v[9]);
          w1.y = ptx::Mma<T>::pack(v[10], v[11]);
          w1.z = ptx::Mma<T>::pack(v[12], v[13]);
          w1.w = ptx::Mma<T>::pack(v[14], v[15]);
          uint4* o = reinterpret_cast<uint4*>(outg + (head0 + h) * kDv + c);
          o[0] = w0;
          o[1] = w1;
        } else {
          float4* o = reinterpret_cast<float4*>(p.part_out + (slot_row + h) * kDv + c);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            __stcg(o + e, make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]));
        }
      }
      const float lse_nat = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
      if (whole) {
        if (p.lse != nullptr) p.lse[lse_at(h)] = lse_nat;
      } else {
        __stcg(p.part_lse + slot_row + h, lse_nat);
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
            for (int idx = ctid; idx < kRows * (kDv / 4); idx += kST) {
              const int j = idx / (kDv / 4);
              const int dq = idx - j * (kDv / 4);
              float mxp = -INFINITY;
              for (int64_t c = c0; c <= c1; ++c) {
                const int sl = (c == c0 && pt.seg_start > c * p.tiles_per_cta) ? 1 : 0;
                mxp = fmaxf(mxp, __ldcg(p.part_lse + (c * 2 + sl) * kRows + j));
              }
              float den = 0.f;
              float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int64_t c = c0; c <= c1; ++c) {
                const int sl = (c == c0 && pt.seg_start > c * p.tiles_per_cta) ? 1 : 0;
                const int64_t rowi = (c * 2 + sl) * kRows + j;
                const float wgt = ptx::exp2_approx((__ldcg(p.part_lse + rowi) - mxp) * kLog2e);
                const float4 o =
                    __ldcg(reinterpret_cast<const float4*>(p.part_out + rowi * kDv) + dq);
                den += wgt;
                acc.x += wgt * o.x;
                acc.y += wgt * o.y;
                acc.z += wgt * o.z;
                acc.w += wgt * o.w;
              }
              const float iv = den > 0.f ? 1.f / den : 0.f;
              T* o = outg + (head0 + j) * kDv + dq * 4;
              o[0] = cvt_out<T>(acc.x * iv);
              o[1] = cvt_out<T>(acc.y * iv);
              o[2] = cvt_out<T>(acc.z * iv);
              o[3] = cvt_out<T>(acc.w * iv);
              if (dq == 0 && p.lse != nullptr) p.lse[lse_at(j)] = mxp + logf(den);
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
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename T>
int launch_rows_t(const CUtensorMap& tkv, const RowsParams& prm, int grid, cudaStream_t stream) {
  auto kern = mla_rows_kernel<T>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  kern<<<grid, kThreads, kSmem, stream>>>(tkv, prm);
  return cudaGetLastError();
}

}  // namespace

bool mla_uses_rows(const pda_problem& p) {
  return p.head_dim_qk == kDqk && p.head_dim_v == kDv && p.num_q_heads % kRows == 0 &&
         p.kv_format == PDA_KV_SAME_AS_Q;
}

int launch_mla_rows(const Plan& plan, const MlaArgs& a, const Workspace& ws, void* stream) {
  const pda_problem& pr = plan.prob;
  const bool bf16 = pr.dtype == PDA_BF16;
  CUtensorMap m[2];   // q is read row by row; only the cache map is passed
  const int sq = pr.seq_len_q > 1 ? pr.seq_len_q : 1;
  if (!plan.map_cache.get(a.q, a.kv_cache, m, nullptr, [&](CUtensorMap* t, int32_t*) {
        return encode_mla_maps(&t[0], &t[1], a.q, int64_t(pr.batch) * sq * pr.num_q_heads,
                               kRows, a.kv_cache, pr.num_blocks, bf16, kDqk);
      }))
    return -1;
  const CUtensorMap& tkv = m[1];
  RowsParams prm{};
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
  prm.scale_log2 = a.scale * kLog2e;
  prm.total_tiles = plan.total_tiles;
  prm.tiles_per_cta = plan.tiles_per_cta;
  prm.heavy_min = plan.heavy_min_pieces;
  prm.err = ws.err;
  prm.counters = ws.counters;
  prm.part_lse = ws.part_lse;
  prm.part_out = ws.part_out;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int e = bf16 ? launch_rows_t<__nv_bfloat16>(tkv, prm, plan.num_ctas, s)
                     : launch_rows_t<__half>(tkv, prm, plan.num_ctas, s);
  if (e != 0) return e;
  return launch_split_merge(plan, ws, a.out, a.lse, stream);
}

}  // namespace pda
