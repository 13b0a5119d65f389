// Appending the new tokens' keys and values (or MLA records) to the paged caches.
//
// What it computes ("From MHA to MLA", section 2: at each decode step the new key and
// value are appended to the cache, and every later step rereads them; section 5: logical
// token n of sequence b lives in block block_tables[b][n / P], slot n % P): the S new
// tokens of sequence b are its logical tokens ctx_b - S + i (ctx_b counts them), and
// token i's rows [rows][width] are copied from new[b][i] into cache[phys][slot].
//
// fp8 (E4M3) caches store code = e4m3(x / scale): the division in fp32 (IEEE, round to
// nearest), one rounding to E4M3 with ties to even and saturation to +-448.
//
// One thread moves 8 values (16 bytes of the 16-bit source). A block-table entry outside
// [0, num_blocks), a position outside the table or a context shorter than S sets bit 0
// of the error word and that token is not written.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pda_internal.h"

namespace pda {
namespace {

struct AppendParams {
  const void* src0;          // [B][S][rows][width] 16-bit (K, or the MLA record)
  const void* src1;          // V (GQA), selected by blockIdx.y == 1
  void* dst0;                // [num_blocks][P][rows][width], 16-bit or E4M3 bytes
  void* dst1;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t batch, seq_len_q, rows, width, page, max_blocks;
  int64_t num_blocks;
  float scale0, scale1;      // E4M3 only
  int32_t* err;
};

__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// two fp32 values -> two E4M3 codes (lo in the low byte), nearest-even, saturating
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// blockIdx.y selects one of up to two (src, dst) pairs (K and V)
template <typename T, bool F8>
__global__ void __launch_bounds__(128) append_kernel(const AppendParams p) {
  const bool second = blockIdx.y != 0;
  const T* src = static_cast<const T*>(second ? p.src1 : p.src0);
  void* dst = second ? p.dst1 : p.dst0;
  const float scale = second ? p.scale1 : p.scale0;
  const int per_token = p.rows * p.width / 8;           // 8-value chunks per token
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= int64_t(p.batch) * p.seq_len_q * per_token) return;
  const int64_t tk = idx / per_token;
  const int within = int(idx - tk * per_token) * 8;    // value offset inside the token
  const int b = int(tk / p.seq_len_q);
  const int i = int(tk - int64_t(b) * p.seq_len_q);
  const int64_t n = int64_t(__ldg(p.context_lens + b)) - p.seq_len_q + i;
  const int64_t lp = n / p.page;
  if (n < 0 || lp >= p.max_blocks) {
    if (within == 0) atomicOr(p.err, 1);
    return;
  }
  const int32_t phys = __ldg(p.block_tables + int64_t(b) * p.max_blocks + lp);
  if (phys < 0 || int64_t(phys) >= p.num_blocks) {
    if (within == 0) atomicOr(p.err, 1);
    return;
  }
  const int64_t slot = n - lp * p.page;
  const int64_t dst_elem = ((int64_t(phys) * p.page + slot) * p.rows) * p.width + within;
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + tk * p.rows * p.width + within));
  if constexpr (!F8) {
    *reinterpret_cast<uint4*>(static_cast<T*>(dst) + dst_elem) = v;
  } else {
    const T* x = reinterpret_cast<const T*>(&v);
    uint16_t c[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      c[e] = e4m3x2(__fdiv_rn(to_f32(x[2 * e]), scale), __fdiv_rn(to_f32(x[2 * e + 1]), scale));
    uint2 w;
    w.x = uint32_t(c[0]) | (uint32_t(c[1]) << 16);
    w.y = uint32_t(c[2]) | (uint32_t(c[3]) << 16);
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(dst) + dst_elem) = w;
  }
}

template <typename T, bool F8>
int launch_t(const AppendParams& p, int tensors, cudaStream_t s) {
  const int64_t threads = int64_t(p.batch) * p.seq_len_q * (p.rows * p.width / 8);
  const dim3 grid(unsigned((threads + 127) / 128), unsigned(tensors));
  append_kernel<T, F8><<<grid, 128, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

int launch_append(const Plan& plan, const AppendArgs& a, const Workspace& ws, void* stream) {
  const pda_problem& pr = plan.prob;
  if (pr.batch == 0) return 0;
  AppendParams p{};
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.batch = pr.batch;
  p.seq_len_q = plan.seq_len_q;
  p.page = pr.page_size;
  p.max_blocks = pr.max_blocks_per_seq;
  p.num_blocks = pr.num_blocks;
  p.err = ws.err;
  const bool mla = pr.kind == PDA_KIND_MLA;
  p.rows = mla ? 1 : pr.num_kv_heads;
  p.width = pr.head_dim_qk;
  p.src0 = a.k_new;
  p.dst0 = a.k_cache;
  p.scale0 = a.k_scale;
  p.src1 = a.v_new;
  p.dst1 = a.v_cache;
  p.scale1 = a.v_scale;
  const int tensors = mla ? 1 : 2;
  const bool f8 = pr.kv_format == PDA_KV_FP8_E4M3;
  const bool bf16 = pr.dtype == PDA_BF16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (f8)
    return bf16 ? launch_t<__nv_bfloat16, true>(p, tensors, s)
                : launch_t<__half, true>(p, tensors, s);
  return bf16 ? launch_t<__nv_bfloat16, false>(p, tensors, s)
              : launch_t<__half, false>(p, tensors, s);
}

}  // namespace pda
