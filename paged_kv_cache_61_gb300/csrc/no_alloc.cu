// paged_decode_attn_no_alloc: the GQA decode call for callers that cannot allocate
// device memory. The scratch space that paged_decode_attn takes from the caller's
// workspace (split pieces, merge counters, error word) is a library-owned device
// array here, so the call needs only its inputs and outputs.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>
#include <string>

#include "pda_internal.h"

namespace pda {
namespace {

// One array per device that loads the library, kept until the process exits.
static __device__ __align__(256) unsigned char g_no_alloc_workspace[PDA_NO_ALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_addr_mutex;
void* g_addr[kMaxDevices] = {};

// Device address of the array on the current device. In host code the array's
// name is only a stand-in, so the address is looked up once per device (with that
// device current) and remembered.
cudaError_t workspace_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_addr_mutex);
  if (g_addr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_no_alloc_workspace);
    if (e != cudaSuccess) return e;
    g_addr[dev] = ptr;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace pda

extern "C" PDA_API pda_status paged_decode_attn_no_alloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, float scale, void* out, float* lse, const pda_plan* plan,
    pda_stream_t stream) {
  pda::clear_error();
  if (plan == nullptr) return pda::fail(PDA_ERR_INVALID_ARG, "plan is NULL");
  if (plan->prob.kind != PDA_KIND_GQA)
    return pda::fail(PDA_ERR_INVALID_ARG, "plan was created for the other kernel kind");
  if (plan->prob.kv_format != PDA_KV_SAME_AS_Q)
    return pda::fail(PDA_ERR_INVALID_ARG, "this call takes 16-bit caches (kv_format PDA_KV_SAME_AS_Q)");
  if (!std::isfinite(scale)) return pda::fail(PDA_ERR_INVALID_ARG, "scale must be finite");
  if (plan->prob.batch == 0) return PDA_OK;
  if (plan->ws_bytes > size_t(PDA_NO_ALLOC_WORKSPACE_BYTES))
    return pda::fail(PDA_ERR_WORKSPACE,
                     "the plan needs " + std::to_string(plan->ws_bytes) +
                         " bytes of workspace, more than the library's " +
                         std::to_string(PDA_NO_ALLOC_WORKSPACE_BYTES) +
                         "-byte array; use paged_decode_attn with a workspace");
  void* ws = nullptr;
  cudaError_t e = pda::workspace_address(&ws);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return pda::fail(PDA_ERR_CUDA, std::string("looking up the library workspace: ") +
                                       cudaGetErrorString(e));
  }
  // The merge counters must start at zero (a kernel that gave up on a timed-out wait
  // may have left one behind); the split pieces are always written before they are
  // read. The error word is not cleared: it collects the device errors of every call
  // until pda_no_alloc_read_device_error reads it.
  e = cudaMemsetAsync(static_cast<unsigned char*>(ws) + plan->ws_counters, 0,
                      plan->ws_part_lse - plan->ws_counters, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return pda::fail(PDA_ERR_CUDA, std::string("clearing the library workspace: ") +
                                       cudaGetErrorString(e));
  }
  // Same validation and launch as paged_decode_attn, on the library's array.
  return paged_decode_attn(q, k_cache, v_cache, block_tables, context_lens, scale, out, lse, plan,
                           ws, stream);
}

extern "C" PDA_API pda_status pda_no_alloc_read_device_error(pda_stream_t stream, int32_t* code) {
  pda::clear_error();
  if (code == nullptr) return pda::fail(PDA_ERR_INVALID_ARG, "code must be non-NULL");
  void* ws = nullptr;
  cudaError_t e = pda::workspace_address(&ws);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return pda::fail(PDA_ERR_CUDA, std::string("looking up the library workspace: ") +
                                       cudaGetErrorString(e));
  }
  // Every plan keeps its error word at the start of the workspace.
  return pda_read_device_error(ws, stream, code);
}
