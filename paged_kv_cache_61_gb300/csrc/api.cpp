// C-ABI entry points: argument validation on the host, then kernel launch.
// Nothing here computes attention; every step of the path runs in the kernels.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <string>

#include "pda_internal.h"

using pda::fail;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

pda_status cuda_fail(int err, const char* what) {
  cudaGetLastError();
  return fail(PDA_ERR_CUDA, std::string(what) + ": " +
                                cudaGetErrorString(static_cast<cudaError_t>(err)));
}

pda_status check_common(const pda_plan* plan, int kind, const void* q,
                        const int32_t* block_tables, const int32_t* context_lens, float scale,
                        const void* out, const void* workspace) {
  if (plan == nullptr) return fail(PDA_ERR_INVALID_ARG, "plan is NULL");
  if (plan->prob.kind != kind)
    return fail(PDA_ERR_INVALID_ARG, "plan was created for the other kernel kind");
  if (!std::isfinite(scale)) return fail(PDA_ERR_INVALID_ARG, "scale must be finite");
  if (plan->prob.batch == 0) return PDA_OK;
  if (q == nullptr || block_tables == nullptr || context_lens == nullptr || out == nullptr)
    return fail(PDA_ERR_INVALID_ARG, "a required tensor pointer is NULL");
  if (!aligned(q, 16) || !aligned(out, 16))
    return fail(PDA_ERR_INVALID_ARG, "q and out must start on a 16-byte boundary");
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4))
    return fail(PDA_ERR_INVALID_ARG, "block_tables and context_lens must be 4-byte aligned");
  if (workspace == nullptr) return fail(PDA_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 256))
    return fail(PDA_ERR_WORKSPACE, "workspace must start on a 256-byte boundary");
  return PDA_OK;
}

}  // namespace

extern "C" PDA_API pda_status pda_workspace_init(const pda_plan* plan, void* workspace,
                                         pda_stream_t stream) {
  pda::clear_error();
  if (plan == nullptr) return fail(PDA_ERR_INVALID_ARG, "plan is NULL");
  if (workspace == nullptr) return fail(PDA_ERR_WORKSPACE, "workspace is NULL");
  const cudaError_t e = cudaMemsetAsync(workspace, 0, plan->ws_bytes, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace)");
  return PDA_OK;
}

extern "C" PDA_API pda_status pda_read_device_error(void* workspace, pda_stream_t stream, int32_t* code) {
  pda::clear_error();
  if (workspace == nullptr || code == nullptr)
    return fail(PDA_ERR_INVALID_ARG, "workspace and code must be non-NULL");
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  *code = v;
  return PDA_OK;
}

namespace {

pda_status gqa_call(const void* q, const void* k_cache, const void* v_cache, float k_scale,
                    float v_scale, const int32_t* block_tables, const int32_t* context_lens,
                    float scale, void* out, float* lse, const pda_plan* plan, void* workspace,
                    pda_stream_t stream) {
  pda_status st = check_common(plan, PDA_KIND_GQA, q, block_tables, context_lens, scale, out,
                               workspace);
  if (st != PDA_OK || plan->prob.batch == 0) return st;
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale))
    return fail(PDA_ERR_INVALID_ARG, "k_scale and v_scale must be finite");
  if (k_cache == nullptr || v_cache == nullptr)
    return fail(PDA_ERR_INVALID_ARG, "k_cache and v_cache must be non-NULL");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(PDA_ERR_INVALID_ARG, "k_cache and v_cache must start on a 16-byte boundary");
  if (lse != nullptr && !aligned(lse, 4))
    return fail(PDA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  pda::GqaArgs args{q, k_cache, v_cache, block_tables, context_lens, scale, out, lse,
                    k_scale, v_scale};
  const int e = pda::launch_gqa_decode(*plan, args, pda::workspace_views(*plan, workspace),
                                       stream);
  if (e == -1) return fail(PDA_ERR_INVALID_ARG, "could not build the TMA descriptor of a cache");
  if (e != 0) return cuda_fail(e, "GQA decode launch");
  return PDA_OK;
}

}  // namespace

extern "C" PDA_API pda_status paged_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_tables, const int32_t* context_lens,
                                        float scale, void* out, float* lse, const pda_plan* plan,
                                        void* workspace, pda_stream_t stream) {
  pda::clear_error();
  if (plan != nullptr && plan->prob.kv_format != PDA_KV_SAME_AS_Q)
    return fail(PDA_ERR_INVALID_ARG,
                "the plan's caches are fp8: call paged_decode_attn_fp8 with their scales");
  return gqa_call(q, k_cache, v_cache, 1.f, 1.f, block_tables, context_lens, scale, out, lse, plan,
                  workspace, stream);
}

extern "C" PDA_API pda_status paged_decode_attn_fp8(const void* q, const void* k_cache,
                                                    const void* v_cache, float k_scale,
                                                    float v_scale, const int32_t* block_tables,
                                                    const int32_t* context_lens, float scale,
                                                    void* out, float* lse, const pda_plan* plan,
                                                    void* workspace, pda_stream_t stream) {
  pda::clear_error();
  if (plan != nullptr && plan->prob.kv_format != PDA_KV_FP8_E4M3)
    return fail(PDA_ERR_INVALID_ARG,
                "the plan's caches are not fp8 (kv_format PDA_KV_FP8_E4M3): call paged_decode_attn");
  return gqa_call(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale, out,
                  lse, plan, workspace, stream);
}

namespace {

pda_status mla_call(const void* q, const void* kv_cache, float kv_scale,
                    const int32_t* block_tables, const int32_t* context_lens, float scale,
                    void* out, float* lse, const pda_plan* plan, void* workspace,
                    pda_stream_t stream) {
  pda_status st = check_common(plan, PDA_KIND_MLA, q, block_tables, context_lens, scale, out,
                               workspace);
  if (st != PDA_OK || plan->prob.batch == 0) return st;
  if (!std::isfinite(kv_scale)) return fail(PDA_ERR_INVALID_ARG, "kv_scale must be finite");
  if (kv_cache == nullptr) return fail(PDA_ERR_INVALID_ARG, "kv_cache must be non-NULL");
  if (!aligned(kv_cache, 16))
    return fail(PDA_ERR_INVALID_ARG, "kv_cache must start on a 16-byte boundary");
  if (lse != nullptr && !aligned(lse, 4))
    return fail(PDA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  pda::MlaArgs args{q, kv_cache, block_tables, context_lens, scale, out, lse, kv_scale};
  const int e = pda::launch_mla_decode(*plan, args, pda::workspace_views(*plan, workspace),
                                       stream);
  if (e == -1) return fail(PDA_ERR_INVALID_ARG, "could not build the TMA descriptor of the cache");
  if (e != 0) return cuda_fail(e, "MLA decode launch");
  return PDA_OK;
}

}  // namespace

extern "C" PDA_API pda_status mla_decode(const void* q, const void* kv_cache, const int32_t* block_tables,
                                 const int32_t* context_lens, float scale, void* out, float* lse,
                                 const pda_plan* plan, void* workspace, pda_stream_t stream) {
  pda::clear_error();
  if (plan != nullptr && plan->prob.kv_format != PDA_KV_SAME_AS_Q)
    return fail(PDA_ERR_INVALID_ARG,
                "the plan's cache is fp8: call mla_decode_fp8 with its scale");
  return mla_call(q, kv_cache, 1.f, block_tables, context_lens, scale, out, lse, plan, workspace,
                  stream);
}

extern "C" PDA_API pda_status mla_decode_fp8(const void* q, const void* kv_cache, float kv_scale,
                                             const int32_t* block_tables,
                                             const int32_t* context_lens, float scale, void* out,
                                             float* lse, const pda_plan* plan, void* workspace,
                                             pda_stream_t stream) {
  pda::clear_error();
  if (plan != nullptr && plan->prob.kv_format != PDA_KV_FP8_E4M3)
    return fail(PDA_ERR_INVALID_ARG,
                "the plan's cache is not fp8 (kv_format PDA_KV_FP8_E4M3): call mla_decode");
  return mla_call(q, kv_cache, kv_scale, block_tables, context_lens, scale, out, lse, plan,
                  workspace, stream);
}

extern "C" PDA_API pda_status pda_combine_splits(const float* partial_out, const float* partial_lse,
                                         int32_t rows, int32_t num_splits, int32_t head_dim_v,
                                         void* out, int32_t out_dtype, float* lse,
                                         pda_stream_t stream) {
  pda::clear_error();
  if (rows < 0 || num_splits < 1) return fail(PDA_ERR_INVALID_ARG, "rows >= 0, num_splits >= 1");
  if (head_dim_v < 4 || head_dim_v > 1024 || head_dim_v % 4 != 0)
    return fail(PDA_ERR_UNSUPPORTED, "head_dim_v must be a multiple of 4 in [4, 1024]");
  if (out_dtype != PDA_FP16 && out_dtype != PDA_BF16)
    return fail(PDA_ERR_INVALID_ARG, "out_dtype must be PDA_FP16 or PDA_BF16");
  if (rows == 0) return PDA_OK;
  if (partial_out == nullptr || partial_lse == nullptr || out == nullptr)
    return fail(PDA_ERR_INVALID_ARG, "partial_out, partial_lse and out must be non-NULL");
  if (!aligned(partial_out, 16) || !aligned(partial_lse, 4) || !aligned(out, 8) ||
      (lse != nullptr && !aligned(lse, 4)))
    return fail(PDA_ERR_INVALID_ARG, "misaligned pointer (partial_out needs 16 bytes, out 8)");
  const int e = pda::launch_combine(partial_out, partial_lse, rows, num_splits, head_dim_v, out,
                                    out_dtype, lse, stream);
  if (e != 0) return cuda_fail(e, "combine launch");
  return PDA_OK;
}

namespace {

pda_status append_call(int kind, const void* k_new, const void* v_new, void* k_cache,
                       void* v_cache, float k_scale, float v_scale, const int32_t* block_tables,
                       const int32_t* context_lens, const pda_plan* plan, void* workspace,
                       pda_stream_t stream) {
  if (plan == nullptr) return fail(PDA_ERR_INVALID_ARG, "plan is NULL");
  if (plan->prob.kind != kind)
    return fail(PDA_ERR_INVALID_ARG, "plan was created for the other kernel kind");
  if (plan->prob.batch == 0) return PDA_OK;
  const bool gqa = kind == PDA_KIND_GQA;
  if (k_new == nullptr || k_cache == nullptr || (gqa && (v_new == nullptr || v_cache == nullptr)) ||
      block_tables == nullptr || context_lens == nullptr)
    return fail(PDA_ERR_INVALID_ARG, "a required tensor pointer is NULL");
  if (!aligned(k_new, 16) || !aligned(k_cache, 16) ||
      (gqa && (!aligned(v_new, 16) || !aligned(v_cache, 16))))
    return fail(PDA_ERR_INVALID_ARG, "new values and caches must start on a 16-byte boundary");
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4))
    return fail(PDA_ERR_INVALID_ARG, "block_tables and context_lens must be 4-byte aligned");
  if (workspace == nullptr) return fail(PDA_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 256))
    return fail(PDA_ERR_WORKSPACE, "workspace must start on a 256-byte boundary");
  pda::AppendArgs args{k_new, v_new, k_cache, v_cache, block_tables, context_lens, k_scale,
                       v_scale};
  const int e = pda::launch_append(*plan, args, pda::workspace_views(*plan, workspace), stream);
  if (e != 0) return cuda_fail(e, "append launch");
  return PDA_OK;
}

}  // namespace

extern "C" PDA_API pda_status pda_kv_append(const void* k_new, const void* v_new, void* k_cache,
                                            void* v_cache, const int32_t* block_tables,
                                            const int32_t* context_lens, const pda_plan* plan,
                                            void* workspace, pda_stream_t stream) {
  pda::clear_error();
  if (plan != nullptr && plan->prob.kv_format != PDA_KV_SAME_AS_Q)
    return fail(PDA_ERR_INVALID_ARG, "the plan's caches are fp8: call pda_kv_append_fp8");
  return append_call(PDA_KIND_GQA, k_new, v_new, k_cache, v_cache, 1.f, 1.f, block_tables,
                     context_lens, plan, workspace, stream);
}

extern "C" PDA_API pda_status pda_kv_append_fp8(const void* k_new, const void* v_new,
                                                void* k_cache, void* v_cache, float k_scale,
                                                float v_scale, const int32_t* block_tables,
                                                const int32_t* context_lens,
                                                const pda_plan* plan, void* workspace,
                                                pda_stream_t stream) {
  pda::clear_error();
  if (plan != nullptr && plan->prob.kv_format != PDA_KV_FP8_E4M3)
    return fail(PDA_ERR_INVALID_ARG, "the plan's caches are not fp8: call pda_kv_append");
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale) || k_scale == 0.f || v_scale == 0.f)
    return fail(PDA_ERR_INVALID_ARG, "k_scale and v_scale must be finite and nonzero");
  return append_call(PDA_KIND_GQA, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                     block_tables, context_lens, plan, workspace, stream);
}

extern "C" PDA_API pda_status pda_mla_append(const void* kv_new, void* kv_cache,
                                             const int32_t* block_tables,
                                             const int32_t* context_lens, const pda_plan* plan,
                                             void* workspace, pda_stream_t stream) {
  pda::clear_error();
  if (plan != nullptr && plan->prob.kv_format != PDA_KV_SAME_AS_Q)
    return fail(PDA_ERR_INVALID_ARG, "the plan's record cache is fp8: call pda_mla_append_fp8");
  return append_call(PDA_KIND_MLA, kv_new, nullptr, kv_cache, nullptr, 1.f, 1.f, block_tables,
                     context_lens, plan, workspace, stream);
}

extern "C" PDA_API pda_status pda_mla_append_fp8(const void* kv_new, void* kv_cache,
                                                 float kv_scale, const int32_t* block_tables,
                                                 const int32_t* context_lens,
                                                 const pda_plan* plan, void* workspace,
                                                 pda_stream_t stream) {
  pda::clear_error();
  if (plan != nullptr && plan->prob.kv_format != PDA_KV_FP8_E4M3)
    return fail(PDA_ERR_INVALID_ARG, "the plan's record cache is not fp8: call pda_mla_append");
  if (!std::isfinite(kv_scale) || kv_scale == 0.f)
    return fail(PDA_ERR_INVALID_ARG, "kv_scale must be finite and nonzero");
  return append_call(PDA_KIND_MLA, kv_new, nullptr, kv_cache, nullptr, kv_scale, 1.f,
                     block_tables, context_lens, plan, workspace, stream);
}
