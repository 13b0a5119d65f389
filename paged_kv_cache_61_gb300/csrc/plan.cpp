// Host-side planning: validate a decode problem and divide its page tiles over CTAs.
//
// FlashMLA-ETAP "Usage": scheduling metadata is computed once per decoding step
// from cache_seqlens and reused by every layer. "From MHA to MLA", section 4: a
// production runtime picks the number of splits from batch size, head tiles,
// context length and the number of SMs. Here every CTA receives the same number
// of page tiles (to within one), so varlen batches and single long sequences
// both keep every SM busy; the splits of a sequence follow from where the
// equal ranges cut its segments.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>

#include "pda_internal.h"

namespace pda {

namespace {

thread_local std::string g_last_error;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

pda_status fail(pda_status s, const std::string& why) {
  g_last_error = why;
  return s;
}

void clear_error() { g_last_error.clear(); }

Workspace workspace_views(const Plan& plan, void* base) {
  char* b = static_cast<char*>(base);
  return Workspace{reinterpret_cast<int32_t*>(b + plan.ws_err),
                   reinterpret_cast<int32_t*>(b + plan.ws_counters),
                   reinterpret_cast<float*>(b + plan.ws_part_lse),
                   reinterpret_cast<float*>(b + plan.ws_part_out)};
}

}  // namespace pda

using pda::fail;

extern "C" PDA_API const char* pda_last_error(void) { return pda::g_last_error.c_str(); }

extern "C" PDA_API const char* pda_status_string(pda_status s) {
  switch (s) {
    case PDA_OK: return "PDA_OK";
    case PDA_ERR_INVALID_ARG: return "PDA_ERR_INVALID_ARG";
    case PDA_ERR_UNSUPPORTED: return "PDA_ERR_UNSUPPORTED";
    case PDA_ERR_WORKSPACE: return "PDA_ERR_WORKSPACE";
    case PDA_ERR_CUDA: return "PDA_ERR_CUDA";
    case PDA_ERR_OUT_OF_BLOCKS: return "PDA_ERR_OUT_OF_BLOCKS";
  }
  return "PDA_ERR_UNKNOWN";
}

extern "C" PDA_API pda_status pda_plan_create(pda_plan** out, const pda_problem* prob,
                                      const int32_t* ctx_host) {
  pda::clear_error();
  if (out == nullptr) return fail(PDA_ERR_INVALID_ARG, "plan output pointer is NULL");
  *out = nullptr;
  if (prob == nullptr) return fail(PDA_ERR_INVALID_ARG, "problem is NULL");
  const pda_problem& p = *prob;
  if (p.kind != PDA_KIND_GQA && p.kind != PDA_KIND_MLA)
    return fail(PDA_ERR_INVALID_ARG, "kind must be PDA_KIND_GQA or PDA_KIND_MLA");
  if (p.dtype != PDA_FP16 && p.dtype != PDA_BF16)
    return fail(PDA_ERR_INVALID_ARG, "dtype must be PDA_FP16 or PDA_BF16");
  if (p.batch < 0) return fail(PDA_ERR_INVALID_ARG, "batch must be >= 0");
  if (p.num_q_heads < 1 || p.num_kv_heads < 1)
    return fail(PDA_ERR_INVALID_ARG, "head counts must be >= 1");
  if (p.num_q_heads % p.num_kv_heads != 0)
    return fail(PDA_ERR_INVALID_ARG, "H_q must be divisible by H_kv");
  if (p.page_size < 1 || p.max_blocks_per_seq < 1 || p.num_blocks < 1)
    return fail(PDA_ERR_INVALID_ARG, "page_size, max_blocks_per_seq and num_blocks must be >= 1");
  if (p.head_dim_qk < 1 || p.head_dim_v < 1)
    return fail(PDA_ERR_INVALID_ARG, "head dims must be >= 1");
  if (p.num_sms < 0 || p.force_num_ctas < 0)
    return fail(PDA_ERR_INVALID_ARG, "num_sms and force_num_ctas must be >= 0");
  if (p.kv_format != PDA_KV_SAME_AS_Q && p.kv_format != PDA_KV_FP8_E4M3)
    return fail(PDA_ERR_INVALID_ARG, "kv_format must be PDA_KV_SAME_AS_Q or PDA_KV_FP8_E4M3");
  if (p.seq_len_q < 0) return fail(PDA_ERR_INVALID_ARG, "seq_len_q must be >= 0");
  const int32_t S = p.seq_len_q > 1 ? p.seq_len_q : 1;
  if (p.batch > 0 && ctx_host == nullptr)
    return fail(PDA_ERR_INVALID_ARG, "context_lens_host is NULL");

  std::string why;
  if (p.kind == PDA_KIND_GQA ? !pda::gqa_supported(p, &why) : !pda::mla_supported(p, &why))
    return fail(PDA_ERR_UNSUPPORTED, why);

  const int64_t max_ctx = int64_t(p.max_blocks_per_seq) * p.page_size;
  for (int32_t b = 0; b < p.batch; ++b) {
    if (ctx_host[b] < S)
      return fail(PDA_ERR_INVALID_ARG, "context_lens[" + std::to_string(b) + "] < " +
                                           (S > 1 ? "seq_len_q" : std::string("1")));
    if (ctx_host[b] > max_ctx)
      return fail(PDA_ERR_INVALID_ARG, "context_lens[" + std::to_string(b) +
                                           "] exceeds max_blocks_per_seq * page_size");
  }

  int num_sms = p.num_sms;
  if (num_sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return fail(PDA_ERR_CUDA, "could not query the SM count of the current device");
    }
  }

  pda_plan* plan = new (std::nothrow) pda_plan();
  if (plan == nullptr) return fail(PDA_ERR_INVALID_ARG, "out of host memory");
  plan->prob = p;
  plan->prob.num_sms = num_sms;
  plan->context_lens.assign(ctx_host, ctx_host + p.batch);
  plan->prob.seq_len_q = S;
  plan->seq_len_q = S;

  int ctas_per_sm;
  int64_t min_tiles_per_cta;
  if (p.kind == PDA_KIND_GQA) {
    // A KV head's S*G query rows go to one segment when they fit the kernel's four
    // 8-column MMA tiles (32 rows); more rows are cut into row_chunks segments of equal
    // size, each of which reads the KV head's pages (the chunks of one head are
    // neighbours in the tile order, so their CTAs read the same pages at about the same
    // time and the repeated reads are served by L2).
    plan->heads_per_seg = p.num_q_heads / p.num_kv_heads;
    const int64_t rows = int64_t(S) * plan->heads_per_seg;
    plan->row_chunks = int32_t(pda::cdiv(rows, 32));
    plan->group = int32_t(pda::cdiv(rows, plan->row_chunks));
    plan->segs_per_seq = p.num_kv_heads * plan->row_chunks;
    plan->head_subtiles = (plan->group + 7) / 8;
    ctas_per_sm = pda::gqa_ctas_per_sm(p);
    // A split piece writes a 4·group·D-byte fp32 partial (group: the segment's rows) and
    // reads 64·D bytes per tile: at least group/4 + 1 tiles keep the partial under a
    // quarter of what the piece reads. (A
    // starting floor: the cap on pieces per segment below and the aligned-piece search
    // may raise or lower a CTA's share from there.)
    min_tiles_per_cta = std::max<int64_t>(4, plan->group / 4 + 1);
  } else {
    // The S*Hq query rows of a sequence (row R = i*Hq + h: query token i, head h) form
    // groups of n consecutive rows: all of them (S*Hq <= 64), or n heads of one token.
    const int n = pda::mla_heads_per_cta(p);
    plan->group = n;
    plan->heads_per_seg = std::min(n, p.num_q_heads);
    plan->segs_per_seq = int32_t(int64_t(S) * p.num_q_heads / n);
    plan->head_subtiles = 1;
    plan->cluster = pda::mla_uses_pairs(p) ? 2 : 1;
    ctas_per_sm = pda::mla_ctas_per_sm(p);
    min_tiles_per_cta = 2;
  }

  int64_t pages_total = 0, pages_max = 0;
  for (int32_t b = 0; b < p.batch; ++b) {
    pages_total += pda::cdiv(ctx_host[b], p.page_size);
    pages_max = std::max<int64_t>(pages_max, pda::cdiv(ctx_host[b], p.page_size));
  }
  plan->total_tiles = pages_total * plan->segs_per_seq;
  // GQA: at most 32 pieces per segment. Every piece adds a partial to the split merge,
  // which runs after the decode grid; with consumers that attend before waiting for the
  // previous grid, a sweep of forced CTA counts on B=1, ctx 32K put the fastest plans at
  // 32 pieces per segment or fewer: MQA 12.3 us at 256 pieces -> 7.2 us at 32; Hq/Hkv =
  // 16 (two segments) 11.5 -> 6.5 us at 32; Hkv=8 unchanged at 32.
  if (p.kind == PDA_KIND_GQA)
    min_tiles_per_cta = std::max<int64_t>(min_tiles_per_cta, pda::cdiv(pages_max, 32));

  if (plan->total_tiles > 0) {
    int64_t q;
    if (p.force_num_ctas > 0) {
      q = pda::cdiv(plan->total_tiles, p.force_num_ctas);
    } else {
      const int64_t max_ctas = plan->cluster == 2 ? int64_t(pda::mla_pair_units(num_sms))
                                                  : int64_t(num_sms) * ctas_per_sm;
      q = std::max(min_tiles_per_cta, pda::cdiv(plan->total_tiles, max_ctas));
      // Uniform batches (every GQA segment has the same S pages): give each CTA whole
      // segments, so no segment is split and no CTA pays the split-piece fence, counter
      // and merge. 16-bit caches: the fewest segments per CTA that fit one wave, when
      // that adds at most half again to a CTA's tiles (B=64, ctx 1K: 2 segments per
      // CTA, 256 CTAs, 45.9 -> 42.7 us). fp8 caches, whose CTAs are bound by their own
      // issue rate rather than by HBM: one segment per CTA, up to two waves, so a
      // CTA's start and end overlap the other CTA on its SM (34.1 -> 29.2 us).
      if (p.kind == PDA_KIND_GQA && p.batch > 0) {
        const int64_t S = pda::cdiv(ctx_host[0], p.page_size);
        bool uniform = true;
        for (int32_t b = 1; b < p.batch && uniform; ++b)
          uniform = pda::cdiv(ctx_host[b], p.page_size) == S;
        const int64_t nseg = int64_t(p.batch) * plan->segs_per_seq;
        if (uniform && S > q) {
          // segments longer than a CTA's share: pieces of S / k pages (k integer), so
          // every CTA range lies inside one segment; the smallest such piece that is
          // at least the natural share, if it adds at most a quarter to it (B=1, ctx
          // 32K, Hkv=8: 64-page pieces, 256 CTAs instead of 304: 25.8 -> 25.1 us), else
          // the largest below it, down to four fifths of it, if the pieces still fit one
          // wave (B=1, ctx 32K, MQA: 8-page pieces, 256 CTAs instead of 228: 13.74 ->
          // 13.01 us; fp8 caches 15.68 -> 14.41 us)
          bool found = false;
          for (int64_t d = q; d <= S && d * 4 <= q * 5; ++d)
            if (S % d == 0) {
              q = d;
              found = true;
              break;
            }
          for (int64_t d = q - 1; !found && d >= 4 && d * 5 >= q * 4; --d)
            if (S % d == 0 && nseg * (S / d) <= max_ctas) {
              q = d;
              found = true;
            }
        } else if (uniform && S >= min_tiles_per_cta) {
          if (p.kv_format == PDA_KV_FP8_E4M3) {
            if (nseg >= max_ctas && nseg <= 2 * max_ctas) q = S;
          } else {
            const int64_t m = pda::cdiv(nseg, max_ctas);   // segments per CTA, one wave
            if (m * S * 2 <= q * 3) q = m * S;
          }
        }
        // At most one tile per SM the step is latency bound, and a split-merge launch
        // after the decode grid costs more than the extra pieces save: raise the share
        // until every segment has no more pieces than the decode kernel merges itself
        // (B=4, ctx U{1..256}, Hkv=2: 18 CTAs and a merge launch 8.95 us, 12 CTAs and
        // one launch 6.06 us).
        if (plan->total_tiles <= num_sms) {
          auto max_pieces = [&](int64_t share) {
            int64_t worst = 1, start = 0;
            for (int32_t b = 0; b < p.batch; ++b) {
              const int64_t np = pda::cdiv(ctx_host[b], p.page_size);
              for (int32_t s = 0; s < plan->segs_per_seq; ++s) {
                const int64_t s0 = start + s * np;
                worst = std::max(worst, (s0 + np - 1) / share - s0 / share + 1);
              }
              start += np * plan->segs_per_seq;
            }
            return worst;
          };
          while (max_pieces(q) > 4) ++q;
        }
      }
    }
    q = std::max(q, pda::cdiv(plan->total_tiles, pda::kMaxCtas));
    plan->tiles_per_cta = q;
    plan->num_ctas = int32_t(pda::cdiv(plan->total_tiles, q));
  }

  // Splits per sequence: how many CTA ranges cut each of its segments. A segment cut
  // into more than heavy_min_pieces pieces is merged by the split-merge kernel; the
  // threshold keeps that list within kMaxHeavySegments (each heavy segment spans more
  // than heavy_min_pieces CTAs, and neighbours share at most one CTA).
  plan->heavy_min_pieces = int32_t(std::max<int64_t>(
      4, pda::cdiv(plan->num_ctas, pda::kMaxHeavySegments)));
  plan->splits.assign(p.batch, 1);
  int64_t start = 0;
  for (int32_t b = 0; b < p.batch; ++b) {
    const int64_t np = pda::cdiv(ctx_host[b], p.page_size);
    int32_t worst = 1;
    for (int32_t s = 0; s < plan->segs_per_seq; ++s) {
      const int64_t s0 = start + s * np, s1 = s0 + np;
      const int32_t pieces =
          int32_t((s1 - 1) / plan->tiles_per_cta - s0 / plan->tiles_per_cta + 1);
      worst = std::max(worst, pieces);
      if (pieces > plan->heavy_min_pieces) {
        if (plan->heavy.size() >= size_t(pda::kMaxHeavySegments)) {
          delete plan;
          return fail(PDA_ERR_UNSUPPORTED, "too many heavily split segments");
        }
        plan->heavy.push_back(pda::HeavySegment{b, s, int32_t(np), 0, s0});
      }
    }
    plan->splits[b] = worst;
    start += np * plan->segs_per_seq;
  }

  size_t off = 0;
  plan->ws_err = off;
  off += 256;
  plan->ws_counters = off;
  off = pda::round_up(
      off + sizeof(int32_t) * size_t(p.batch) * plan->segs_per_seq * plan->cluster, 256);
  plan->ws_part_lse = off;
  off = pda::round_up(off + sizeof(float) * size_t(plan->num_ctas) * 2 * plan->group, 256);
  plan->ws_part_out = off;
  off = pda::round_up(
      off + sizeof(float) * size_t(plan->num_ctas) * 2 * plan->group * p.head_dim_v, 256);
  plan->ws_bytes = off;

  *out = plan;
  return PDA_OK;
}

extern "C" PDA_API void pda_plan_destroy(pda_plan* plan) { delete plan; }

extern "C" PDA_API size_t pda_plan_workspace_bytes(const pda_plan* plan) {
  return plan ? plan->ws_bytes : 0;
}

extern "C" PDA_API int32_t pda_plan_num_ctas(const pda_plan* plan) { return plan ? plan->num_ctas : 0; }

extern "C" PDA_API int32_t pda_plan_num_launches(const pda_plan* plan) {
  if (plan == nullptr || plan->num_ctas == 0) return 0;
  return plan->heavy.empty() ? 1 : 2;
}

extern "C" PDA_API int32_t pda_plan_num_splits(const pda_plan* plan, int32_t b) {
  if (plan == nullptr || b < 0 || b >= plan->prob.batch) return 0;
  return plan->splits[b];
}
