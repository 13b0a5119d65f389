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

}  // namespace

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
