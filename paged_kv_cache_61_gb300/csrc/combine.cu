// Flash-Decoding combine as a stand-alone kernel ("From MHA to MLA", section 4):
// each row merges its S locally normalized split outputs O_s by weights
// exp(L_s - L), L = max_s L_s + ln sum_s exp(L_s - max_s L_s). The fused split
// path in the decode kernels applies the same formula to its per-CTA slots.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "pda_internal.h"

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
// One CTA per (heavy segment, head, 32 output dims). The pieces' LSEs are reduced
// across the CTA, then 16 piece lanes x 8 float4 columns accumulate the weighted
// partial outputs with independent loads, so a segment cut into hundreds of
// pieces is merged by many SMs at once instead of by one.
constexpr int kMergeThreads = 128;
constexpr int kPieceLanes = 16;

struct MergeParams {
  const float* part_out;
  const float* part_lse;
  void* out;
  float* lse;
  int64_t tiles_per_cta;
  int32_t group, dv, num_q_heads, count;
  HeavySegment seg[kMaxHeavySegments];
};

__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
  for (int o = 16; o > 0; o >>= 1) {
    const float u = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, u) : v + u;
  }
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
  for (int w = 1; w < kMergeThreads / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
  __syncthreads();
  return r;
}

template <typename T>
__global__ void __launch_bounds__(kMergeThreads)
    merge_heavy_kernel(const __grid_constant__ MergeParams p) {
  // Wait until the decode grid that wrote the pieces has completed (programmatic
  // dependent launch lets this grid be scheduled while that one drains).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float wts[kMaxCtas];
  __shared__ float red[kMergeThreads / 32];
  __shared__ float4 part[kPieceLanes][8];

  const int chunks = p.dv / 32;
  int w = blockIdx.x;
  const int dchunk = w % chunks;
  w /= chunks;
  const int j = w % p.group;
  const HeavySegment hs = p.seg[w / p.group];
  const int64_t q = p.tiles_per_cta;
  const int64_t c0 = hs.seg_start / q;
  const int n = int((hs.seg_start + hs.np - 1) / q - c0 + 1);
  auto row_of = [&](int i) -> int64_t {
    const int slot = (i == 0 && hs.seg_start > c0 * q) ? 1 : 0;
    return ((c0 + i) * 2 + slot) * p.group + j;
  };

  float mx = -INFINITY;
  for (int i = threadIdx.x; i < n; i += kMergeThreads) {
    const float ls = __ldcg(p.part_lse + row_of(i));
    wts[i] = ls;
    mx = fmaxf(mx, ls);
  }
  mx = block_reduce(mx, red, true);
  float sum = 0.f;
  for (int i = threadIdx.x; i < n; i += kMergeThreads) {
    const float ls = wts[i];
    const float wgt = (ls == -INFINITY) ? 0.f : exp2f((ls - mx) * kLog2e);
    wts[i] = wgt;
    sum += wgt;
  }
  const float den = block_reduce(sum, red, false);  // also orders the wts[] writes

  const int col = threadIdx.x & 7;
  const int pl = threadIdx.x >> 3;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int64_t dofs = int64_t(dchunk) * 32 + col * 4;
#pragma unroll 4
  for (int i = pl; i < n; i += kPieceLanes) {
    const float wgt = wts[i];
    const float4 o = __ldcg(reinterpret_cast<const float4*>(p.part_out + row_of(i) * p.dv + dofs));
    acc.x += wgt * o.x;
    acc.y += wgt * o.y;
    acc.z += wgt * o.z;
    acc.w += wgt * o.w;
  }
  part[pl][col] = acc;
  __syncthreads();
  if (pl == 0) {
    float4 r = part[0][col];
    for (int l = 1; l < kPieceLanes; ++l) {
      r.x += part[l][col].x;
      r.y += part[l][col].y;
      r.z += part[l][col].z;
      r.w += part[l][col].w;
    }
    const float inv = 1.f / den;
    const int64_t orow = int64_t(hs.b) * p.num_q_heads + int64_t(hs.seg) * p.group + j;
    T* o = static_cast<T*>(p.out) + orow * p.dv + dofs;
    o[0] = to_out<T>(r.x * inv);
    o[1] = to_out<T>(r.y * inv);
    o[2] = to_out<T>(r.z * inv);
    o[3] = to_out<T>(r.w * inv);
    if (dchunk == 0 && col == 0 && p.lse != nullptr) p.lse[orow] = mx + logf(den);
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
  prm.count = int32_t(plan.heavy.size());
  for (size_t i = 0; i < plan.heavy.size(); ++i) prm.seg[i] = plan.heavy[i];
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(prm.count * prm.group * (prm.dv / 32)));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (plan.prob.dtype == PDA_BF16)
    e = cudaLaunchKernelEx(&cfg, merge_heavy_kernel<__nv_bfloat16>, prm);
  else
    e = cudaLaunchKernelEx(&cfg, merge_heavy_kernel<__half>, prm);
  return e;
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
