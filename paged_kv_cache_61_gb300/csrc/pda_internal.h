// Internal declarations shared by the host side (plan.cpp, api.cpp) and the kernel launchers.
#pragma once

#include <cuda.h>

#include <cstddef>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "pda.h"

namespace pda {

// Work decomposition shared by the GQA and MLA kernels.
//
// A "segment" is one (sequence b, KV head or head group) pair; it owns
// num_pages(b) = ceil(ctx_b / P) page tiles. Segments are laid out b-major,
// head-minor, so the step's tiles form one flattened list of `total_tiles`
// entries. CTA i owns tiles [i*tiles_per_cta, min((i+1)*tiles_per_cta, total)).
// A segment covered by several CTAs is a Flash-Decoding split: each piece
// writes a normalized partial (O_s, L_s) into a per-CTA slot and the last piece
// to finish merges them.
// A segment split over more CTAs than the decode kernel merges in-line. Its pieces
// are merged by the stand-alone split-merge kernel that follows the decode kernel.
struct HeavySegment {
  int32_t b;          // sequence
  int32_t seg;        // segment: KV head and row chunk (GQA) or head group (MLA)
  int32_t np;         // pages of the sequence
  int32_t pad;
  int64_t seg_start;  // flattened index of the segment's first tile
};
constexpr int kMaxHeavySegments = 64;
constexpr int kMaxCtas = 2048;
// GQA: query rows (S * Hq / Hkv) per KV head; more than 32 are cut into row chunks
constexpr int kMaxRowsPerKvHead = 1024;

// The TMA descriptors of the last call, keyed by the tensors they address: a plan's
// shapes are fixed, so a call on the same buffers (the caches, and q for the MLA kernels)
// reuses them instead of encoding them again.
struct MapCache {
  std::mutex mu;
  bool valid = false;
  const void* key[2] = {nullptr, nullptr};
  int32_t extra = 0;
  CUtensorMap maps[2];

  // Fill out[0..1] (and *extra) from the cache, or from encode(out, extra) when the keys
  // differ; returns false (and caches nothing) when encode fails.
  template <typename F>
  bool get(const void* k0, const void* k1, CUtensorMap* out, int32_t* extra_out, F encode) {
    std::lock_guard<std::mutex> lock(mu);
    if (!(valid && key[0] == k0 && key[1] == k1)) {
      valid = false;
      int32_t x = 0;
      if (!encode(maps, &x)) return false;
      key[0] = k0;
      key[1] = k1;
      extra = x;
      valid = true;
    }
    std::memcpy(out, maps, sizeof(maps));
    if (extra_out != nullptr) *extra_out = extra;
    return true;
  }
};

struct Plan {
  pda_problem prob{};
  int32_t group = 1;            // query rows per segment (GQA: a chunk of S * Hq/Hkv; MLA: heads per group)
  int32_t segs_per_seq = 1;     // segments per sequence (GQA: Hkv * row_chunks; MLA: head groups)
  int32_t row_chunks = 1;       // GQA: segments per KV head (its S*G rows cut into chunks of group)
  int32_t head_subtiles = 1;    // GQA: 8-head MMA column tiles per segment
  int32_t cluster = 1;          // CTAs per work unit (2: the MLA kernel for 128-head groups)
  int32_t seq_len_q = 1;        // query tokens per sequence (S)
  int32_t heads_per_seg = 1;    // heads of a segment (G); its rows are the S*G (token, head) pairs
  int64_t total_tiles = 0;
  int64_t tiles_per_cta = 0;
  int32_t num_ctas = 0;         // work units (CTA pairs when cluster == 2)
  std::vector<int32_t> context_lens;  // host copy used for planning
  std::vector<int32_t> splits;        // per sequence: max pieces over its segments
  int32_t heavy_min_pieces = 4;       // segments with more pieces than this are "heavy"
  std::vector<HeavySegment> heavy;    // at most kMaxHeavySegments
  // workspace layout (byte offsets)
  size_t ws_err = 0;        // int32 device error word
  size_t ws_counters = 0;   // int32 [B * segs_per_seq * cluster]
  size_t ws_part_lse = 0;   // float [num_ctas * 2 * group]
  size_t ws_part_out = 0;   // float [num_ctas * 2 * group * head_dim_v]
  size_t ws_bytes = 0;
  mutable MapCache map_cache;   // TMA descriptors of the last call's buffers
};

// Error reporting (thread-local last error string).
pda_status fail(pda_status s, const std::string& why);
void clear_error();

// Device workspace pointers derived from a plan.
struct Workspace {
  int32_t* err;
  int32_t* counters;
  float* part_lse;
  float* part_out;
};
Workspace workspace_views(const Plan& plan, void* base);

// Kernel launchers (return a CUDA error code as int; 0 = success).
struct GqaArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float scale;
  void* out;
  float* lse;
  float k_scale = 1.f;   // fp8 caches: per-tensor dequantization scales
  float v_scale = 1.f;
};
int launch_gqa_decode(const Plan& plan, const GqaArgs& args, const Workspace& ws, void* stream);

struct MlaArgs {
  const void* q;
  const void* kv_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float scale;
  void* out;
  float* lse;
  float kv_scale = 1.f;   // E4M3 caches: the record's dequantization scale
};
int launch_mla_decode(const Plan& plan, const MlaArgs& args, const Workspace& ws, void* stream);

// Append the S new tokens of each sequence to the caches (append.cu). GQA: k_new/v_new
// [B][S][Hkv][D] into k_cache/v_cache; MLA: k_new [B][S][Dqk] into k_cache (v unused).
struct AppendArgs {
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float k_scale = 1.f;
  float v_scale = 1.f;
};
int launch_append(const Plan& plan, const AppendArgs& args, const Workspace& ws, void* stream);

// Merge the pieces of the plan's heavy segments (launched after a decode kernel on the
// same stream, overlapping its tail through programmatic dependent launch).
int launch_split_merge(const Plan& plan, const Workspace& ws, void* out, float* lse, void* stream);

int launch_combine(const float* partial_out, const float* partial_lse, int rows, int num_splits,
                   int head_dim_v, void* out, int out_dtype, float* lse, void* stream);

// Shape support queries (host-side, for validation before launch).
bool gqa_supported(const pda_problem& p, std::string* why);
bool mla_supported(const pda_problem& p, std::string* why);

// CTA residency the planner assumes for each kernel (CTAs per SM).
int gqa_ctas_per_sm(const pda_problem& p);
int mla_ctas_per_sm(const pda_problem& p);
int mla_heads_per_cta(const pda_problem& p);

// MLA with head groups of 128: one group per two-CTA cluster (mla_pair.cu).
bool mla_uses_pairs(const pda_problem& p);
int mla_pair_units(int num_sms);   // co-resident CTA pairs (falls back to num_sms / 2)
int launch_mla_pair(const Plan& plan, const MlaArgs& args, const Workspace& ws, void* stream);

// MLA with the 320-wide record and head groups of 128: one group per CTA, the heads on
// the MMA's M axis (mla_rows.cu).
bool mla_uses_rows(const pda_problem& p);
int launch_mla_rows(const Plan& plan, const MlaArgs& args, const Workspace& ws, void* stream);

}  // namespace pda

// The opaque handle of the C ABI is the planner's record.
struct pda_plan : pda::Plan {};
