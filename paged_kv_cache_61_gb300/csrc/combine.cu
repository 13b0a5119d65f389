// Flash-Decoding combine as a stand-alone kernel ("From MHA to MLA", section 4):
// each row merges its S locally normalized split outputs O_s by weights
// exp(L_s - L), L = max_s L_s + ln sum_s exp(L_s - max_s L_s). The fused split
// path in the decode kernels applies the same formula to its per-CTA slots.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "pda_internal.h"
#include "tile_walk.cuh"

namespace pda {

namespace {

constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

template <typename T>
__device__ __forceinline__ T to_out(float x);
template <>
__device__ __forceinline__ __half to_out<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
    combine_kernel(const float* __restrict__ part_out, const float* __restrict__ part_lse,
                   int num_splits, int dv, T* __restrict__ out, float* __restrict__ lse) {
  const int64_t row = blockIdx.x;
  const float* pl = part_lse + row * num_splits;
  float mx = -INFINITY;
  for (int s = 0; s < num_splits; ++s) mx = fmaxf(mx, __ldg(pl + s));
  const bool empty_row = (mx == -INFINITY);
  for (int d4 = threadIdx.x; d4 < dv / 4; d4 += kThreads) {
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < num_splits; ++s) {
      const float ls = __ldg(pl + s);
      if (ls == -INFINITY) continue;  // an empty split carries no weight
      const float w = exp2f((ls - mx) * kLog2e);
      const float4 o =
          __ldg(reinterpret_cast<const float4*>(part_out + (row * num_splits + s) * dv) + d4);
      den += w;
      acc.x += w * o.x;
      acc.y += w * o.y;
      acc.z += w * o.z;
      acc.w += w * o.w;
    }
    const float inv = empty_row ? 0.f : 1.f / den;
    T* o = out + row * dv + d4 * 4;
    o[0] = to_out<T>(acc.x * inv);
    o[1] = to_out<T>(acc.y * inv);
    o[2] = to_out<T>(acc.z * inv);
    o[3] = to_out<T>(acc.w * inv);
    if (d4 == 0 && lse != nullptr) lse[row] = empty_row ? -INFINITY : mx + logf(den);
  }
}

// ---------------------------------------------------------------- heavy-segment merge
// One CTA per (heavy segment, head, COLS float4 output columns) with 256 / COLS
// piece lanes. Each thread merges its pieces online (running max, rescaled sum and
// accumulator) with four pieces' loads in flight; the piece lanes of a column are
// then merged through shared memory. The launcher picks COLS from the piece count:
// wide CTAs for a few pieces of long rows (MLA), narrow ones with many piece lanes
// when a segment was cut into hundreds of pieces (one long MQA sequence).
constexpr int kMergeThreads = 256;

struct MergeParams {
  const float* part_out;
  const float* part_lse;
  void* out;
  float* lse;
  int64_t tiles_per_cta;
  int32_t group, dv, num_q_heads, count;
  int32_t heads_per_seg, seq_len_q;  // G and S of a KV head's rows (row r = i*G + g)
  // GQA: segment seg is KV head seg / row_chunks, rows (seg % row_chunks) * group + j
  int32_t row_chunks;
  // MLA: segment seg holds rows R = seg*group + r of the sequence's S*Hq rows (R = i*Hq + h)
  int32_t mla_rows;
  HeavySegment seg[kMaxHeavySegments];
};

template <typename T, int COLS>
__global__ void __launch_bounds__(kMergeThreads)
    merge_heavy_kernel(const __grid_constant__ MergeParams p) {
  constexpr int kLanes = kMergeThreads / COLS;
  // Let the next decode grid on the stream be scheduled early (its consumers wait for
  // this grid to complete before they touch q, out, lse or the workspace), then wait
  // until the decode grid that wrote the pieces has completed (programmatic dependent
  // launch lets this grid be scheduled while that one drains).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float sm_m[kLanes][COLS];
  __shared__ float sm_l[kLanes][COLS];
  __shared__ float4 sm_o[kLanes][COLS];

  const int chunks = p.dv / (4 * COLS);
  int w = blockIdx.x;
  const int dchunk = w % chunks;
  w /= chunks;
  const int j = w % p.group;
  const HeavySegment hs = p.seg[w / p.group];
  // GQA: the last row chunk of a KV head may hold fewer than `group` rows
  const int kvh = hs.seg / p.row_chunks;
  const int r = (hs.seg - kvh * p.row_chunks) * p.group + j;
  if (!p.mla_rows && r >= p.heads_per_seg * p.seq_len_q) return;
  const int64_t q = p.tiles_per_cta;
  const int64_t c0 = hs.seg_start / q;
  const int n = int((hs.seg_start + hs.np - 1) / q - c0 + 1);
  const int col = threadIdx.x % COLS;
  const int pl = threadIdx.x / COLS;
  const int64_t dofs = (int64_t(dchunk) * COLS + col) * 4;

  float m = -INFINITY, l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = pl; i0 < n; i0 += 4 * kLanes) {
    float ls[4];
    float4 o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * kLanes;
      ls[u] = -INFINITY;
      o[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < n) {
        const int slot = (i == 0 && hs.seg_start > c0 * q) ? 1 : 0;
        const int64_t row = ((c0 + i) * 2 + slot) * p.group + j;
        ls[u] = __ldcg(p.part_lse + row);
        o[u] = __ldcg(reinterpret_cast<const float4*>(p.part_out + row * p.dv + dofs));
      }
    }
    const float nm = fmaxf(fmaxf(m, fmaxf(ls[0], ls[1])), fmaxf(ls[2], ls[3]));
    if (nm == -INFINITY) continue;
    const float f = exp2f((m - nm) * kLog2e);
    l *= f;
    acc.x *= f; acc.y *= f; acc.z *= f; acc.w *= f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float wgt = exp2f((ls[u] - nm) * kLog2e);
      l += wgt;
      acc.x += wgt * o[u].x; acc.y += wgt * o[u].y; acc.z += wgt * o[u].z; acc.w += wgt * o[u].w;
    }
    m = nm;
  }
  sm_m[pl][col] = m;
  sm_l[pl][col] = l;
  sm_o[pl][col] = acc;
  __syncthreads();
  if (pl == 0) {
    float mx = -INFINITY;
    for (int r = 0; r < kLanes; ++r) mx = fmaxf(mx, sm_m[r][col]);
    float den = 0.f;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0; r < kLanes; ++r) {
      if (sm_m[r][col] == -INFINITY) continue;
      const float f = exp2f((sm_m[r][col] - mx) * kLog2e);
      den += f * sm_l[r][col];
      s.x += f * sm_o[r][col].x; s.y += f * sm_o[r][col].y;
      s.z += f * sm_o[r][col].z; s.w += f * sm_o[r][col].w;
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    RowIndex ri;
    if (p.mla_rows) {
      const int R = hs.seg * p.group + j;
      const int qi = R / p.num_q_heads;
      const int h = R - qi * p.num_q_heads;
      ri = {(int64_t(hs.b) * p.seq_len_q + qi) * p.num_q_heads + h,
            (int64_t(hs.b) * p.num_q_heads + h) * p.seq_len_q + qi};
    } else {
      ri = seg_row(hs.b, kvh, r, p.heads_per_seg, p.seq_len_q, p.num_q_heads);
    }
    T* out = static_cast<T*>(p.out) + ri.out_row * p.dv + dofs;
    out[0] = to_out<T>(s.x * inv);
    out[1] = to_out<T>(s.y * inv);
    out[2] = to_out<T>(s.z * inv);
    out[3] = to_out<T>(s.w * inv);
    if (dchunk == 0 && col == 0 && p.lse != nullptr) p.lse[ri.lse] = mx + logf(den);
  }
}

template <typename T>
cudaError_t launch_merge_t(int cols, const cudaLaunchConfig_t& base, const MergeParams& prm) {
  cudaLaunchConfig_t cfg = base;
  cfg.gridDim = dim3(unsigned(prm.count * prm.group * (prm.dv / (4 * cols))));
  switch (cols) {
    case 8: return cudaLaunchKernelEx(&cfg, merge_heavy_kernel<T, 8>, prm);
    case 16: return cudaLaunchKernelEx(&cfg, merge_heavy_kernel<T, 16>, prm);
    case 32: return cudaLaunchKernelEx(&cfg, merge_heavy_kernel<T, 32>, prm);
    case 64: return cudaLaunchKernelEx(&cfg, merge_heavy_kernel<T, 64>, prm);
    default: return cudaLaunchKernelEx(&cfg, merge_heavy_kernel<T, 128>, prm);
  }
}

}  // namespace

int launch_split_merge(const Plan& plan, const Workspace& ws, void* out, float* lse,
                       void* stream) {
  if (plan.heavy.empty()) return 0;
  MergeParams prm{};
  prm.part_out = ws.part_out;
  prm.part_lse = ws.part_lse;
  prm.out = out;
  prm.lse = lse;
  prm.tiles_per_cta = plan.tiles_per_cta;
  prm.group = plan.group;
  prm.dv = plan.prob.head_dim_v;
  prm.num_q_heads = plan.prob.num_q_heads;
  prm.heads_per_seg = plan.heads_per_seg;
  prm.seq_len_q = plan.seq_len_q;
  prm.row_chunks = plan.row_chunks;
  prm.mla_rows = plan.prob.kind == PDA_KIND_MLA ? 1 : 0;
  prm.count = int32_t(plan.heavy.size());
  int max_pieces = 0;
  for (size_t i = 0; i < plan.heavy.size(); ++i) {
    prm.seg[i] = plan.heavy[i];
    const HeavySegment& h = plan.heavy[i];
    const int64_t pieces =
        (h.seg_start + h.np - 1) / plan.tiles_per_cta - h.seg_start / plan.tiles_per_cta + 1;
    max_pieces = std::max(max_pieces, int(pieces));
  }
  // float4 columns per CTA: the widest rows for which the CTA's piece lanes
  // (kMergeThreads / cols of them, 4 loads each in flight) cover every piece in one round
  // of loads; rows narrower than that with more pieces than 4 * kMergeThreads / 8
  int cols = 128;
  while (cols > 8 && 4 * (kMergeThreads / cols) < max_pieces) cols /= 2;
  while (cols > prm.dv / 4) cols /= 2;
  if (cols < 8 || (prm.dv / 4) % cols != 0) cols = 8;
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return plan.prob.dtype == PDA_BF16 ? launch_merge_t<__nv_bfloat16>(cols, cfg, prm)
                                     : launch_merge_t<__half>(cols, cfg, prm);
}

int launch_combine(const float* partial_out, const float* partial_lse, int rows, int num_splits,
                   int head_dim_v, void* out, int out_dtype, float* lse, void* stream) {
  if (rows == 0) return 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (out_dtype == PDA_BF16)
    combine_kernel<__nv_bfloat16><<<rows, kThreads, 0, s>>>(
        partial_out, partial_lse, num_splits, head_dim_v, static_cast<__nv_bfloat16*>(out), lse);
  else
    combine_kernel<__half><<<rows, kThreads, 0, s>>>(partial_out, partial_lse, num_splits,
                                                     head_dim_v, static_cast<__half*>(out), lse);
  return cudaGetLastError();
}

}  // namespace pda
