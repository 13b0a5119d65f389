/*
 * pda.h - paged decode attention for GB300 (sm_103a), C ABI.
 *
 * One new query token per sequence attends to that sequence's cached keys and
 * values, which live in a paged pool addressed through a block table:
 *
 *   for sequence b, query head h, logical token j < context_lens[b]:
 *     phys = block_tables[b][j / P], slot = j % P                  (paging)
 *     K_j  = k_cache[phys][slot][h / G][:], V_j likewise (G = Hq / Hkv, contiguous grouping)
 *     s_j  = scale * <q[b][h], K_j>
 *   out[b][h] = sum_j softmax(s)_j V_j,   lse[b][h] = ln sum_j exp(s_j)   (natural log, fp32)
 *
 * Sources: "From MHA to MLA: KV Caches and Attention Kernels" (g-u-n.github.io),
 * sections 2-6 (GQA head mapping, grouped-head decode, Flash-Decoding split and
 * combine, paged addressing, absorbed MLA); "L2 讲解：paged decode attention 与
 * GQA" (kzhou003.github.io gpu-kernel-drills), sections ③-⑤ (grid over
 * (batch, KV head), page loop, masking of the partial last page); FlashMLA-ETAP
 * README, sections "Usage" and "Supported configurations" (per-step scheduling
 * metadata, 576/512 and 320/256 latent layouts, page size 64, fp32 lse).
 *
 * Conventions for every call:
 *  - The caller owns every buffer and the stream. Device pointers are CUDA
 *    device (or managed) memory of the current device; "host" pointers are
 *    ordinary host memory.
 *  - Tensors are dense and row-major with the shapes given below; 16-bit
 *    tensors (q, caches, out) start on a 16-byte boundary, the workspace on a
 *    256-byte boundary.
 *  - Decode calls allocate nothing. They are asynchronous on `stream` (NULL =
 *    the legacy default stream) and return as soon as the work is enqueued.
 *  - Arguments are validated on the host; a failed check returns a status and
 *    enqueues nothing. pda_last_error() gives a one-line reason for the last
 *    failure on the calling thread. No C++ exception crosses this boundary.
 *  - A workspace may be used by one call at a time: two calls that overlap on
 *    the GPU (different streams, same workspace) race.
 */
#ifndef PDA_H_
#define PDA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PDA_API __attribute__((visibility("default")))
#else
#define PDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers. */
typedef struct CUstream_st* pda_stream_t;

typedef enum pda_status {
  PDA_OK = 0,
  PDA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, ctx < 1, plan/kind mismatch */
  PDA_ERR_UNSUPPORTED = 2,  /* a shape or dtype this build has no kernel for */
  PDA_ERR_WORKSPACE = 3,    /* workspace missing or too small for the plan */
  PDA_ERR_CUDA = 4,         /* a CUDA runtime call failed (launch, copy, device query) */
  PDA_ERR_OUT_OF_BLOCKS = 5 /* the block pool has too few free blocks (nothing allocated) */
} pda_status;

typedef enum pda_dtype { PDA_FP16 = 0, PDA_BF16 = 1 } pda_dtype;
typedef enum pda_kind { PDA_KIND_GQA = 0, PDA_KIND_MLA = 1 } pda_kind;

/* Storage format of the caches ("Attention Kernel Variants: MQA, GQA, and MLA",
 * KV-cache arithmetic table, fp8 row, and pitfall 5: an fp8 cache stores one byte
 * per value and the kernel dequantizes its tiles before the attention arithmetic).
 *   PDA_KV_SAME_AS_Q: the caches hold values of the problem's dtype.
 *   PDA_KV_FP8_E4M3:  the caches hold one E4M3 byte per value (OCP 8-bit format:
 *                     bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN);
 *                     value = e4m3(code) * scale, one scale per tensor, passed to
 *                     the *_fp8 decode calls. q, out and lse keep their types. */
typedef enum pda_kv_format { PDA_KV_SAME_AS_Q = 0, PDA_KV_FP8_E4M3 = 1 } pda_kv_format;

/* Shape of one decode problem. The plan keeps a copy. */
typedef struct pda_problem {
  int32_t kind;               /* pda_kind */
  int32_t dtype;              /* pda_dtype of q, the caches and out */
  int32_t batch;              /* B >= 0 sequences (B == 0: every call is a no-op) */
  int32_t num_q_heads;        /* Hq */
  int32_t num_kv_heads;       /* Hkv, Hq % Hkv == 0 ("H_q must be divisible by H_kv"); MLA: 1 */
  int32_t head_dim_qk;        /* GQA: 64 or 128; MLA: 576 (512 latent + 64 rope) or 320 (256 + 64) */
  int32_t head_dim_v;         /* GQA: == head_dim_qk; MLA: head_dim_qk - 64 (V = the latent dims) */
  int32_t page_size;          /* tokens per physical block P; GQA: 16; MLA: 64 */
  int32_t max_blocks_per_seq; /* columns of block_tables */
  int64_t num_blocks;         /* physical blocks in the cache pool */
  int32_t num_sms;            /* SMs to plan for; 0 = query the current device */
  int32_t force_num_ctas;     /* 0 = automatic; > 0 = split the work over exactly this many CTAs */
  int32_t kv_format;          /* pda_kv_format of the caches (0 = same type as q) */
  int32_t seq_len_q;          /* S, query tokens per sequence; 0 or 1 = single-token decode.
                                 S > 1 (speculative / MTP decoding): query token i of
                                 sequence b sits at position ctx_b - S + i and attends to
                                 tokens 0 .. ctx_b - S + i (causal, bottom-right aligned);
                                 every ctx_b >= S. GQA: S * Hq / Hkv <= 1024 (a KV
                                 head's rows beyond 32 are computed in equal chunks of
                                 at most 32 rows, each of which reads the KV head's
                                 pages). MLA (16-bit records): S * Hq in {16, 32, 64},
                                 or Hq a multiple of 64 */
} pda_problem;

typedef struct pda_plan pda_plan;  /* opaque, owned by the library */

/*
 * Plan one decode step (FlashMLA-ETAP "Usage": scheduling metadata is computed
 * once per step, whenever the context lengths change, and reused by every
 * layer's attention call).
 *
 * The work of a step is the list of (sequence, KV head, page) tiles; the plan
 * divides it into equal contiguous ranges, one per CTA, sized from the SM
 * count. A (sequence, KV head) whose pages land in more than one range is
 * computed as Flash-Decoding splits ("From MHA to MLA", section 4) and
 * combined on the GPU by the last CTA that finishes one of its splits.
 *
 * context_lens_host: [B] int32 on the host, every entry in
 * [1, max_blocks_per_seq * page_size]. The device context_lens passed to the
 * decode call MUST hold the same values.
 * Returns PDA_OK and *plan, or an error status (and *plan == NULL).
 */
PDA_API pda_status pda_plan_create(pda_plan** plan, const pda_problem* problem,
                           const int32_t* context_lens_host);

/* Frees a plan (NULL is ignored). */
PDA_API void pda_plan_destroy(pda_plan* plan);

/* Bytes of device workspace the decode call needs for this plan (>= 256). */
PDA_API size_t pda_plan_workspace_bytes(const pda_plan* plan);

/* CTAs the decode call launches. */
PDA_API int32_t pda_plan_num_ctas(const pda_plan* plan);

/* Number of Flash-Decoding splits of sequence b: the largest number of CTAs that
 * share one of its (KV head or head group) segments. 1 = computed by one CTA. */
PDA_API int32_t pda_plan_num_splits(const pda_plan* plan, int32_t b);

/* Kernel launches one decode call makes with this plan: 1, or 2 when heavily split
 * segments are merged by a separate split-merge kernel after the decode kernel. (An
 * append call is one more launch of its own.) */
PDA_API int32_t pda_plan_num_launches(const pda_plan* plan);

/*
 * Zero a workspace before its first use with any plan. The decode calls leave
 * the workspace's counters at zero when they complete, so this is needed once
 * per workspace allocation, not once per call. Asynchronous on `stream`.
 */
PDA_API pda_status pda_workspace_init(const pda_plan* plan, void* workspace, pda_stream_t stream);

/*
 * Read and clear the device error word of a workspace (synchronizes `stream`).
 * *code = 0: no error; bit 0: a block-table entry of a read page was outside
 * [0, num_blocks) (that page was read as zeros); bit 1: a pipeline wait timed
 * out and the kernel abandoned its work; bit 2: the MLA kernel for head groups of
 * 128 found its shared memory not 1024-byte aligned and did no work.
 */
PDA_API pda_status pda_read_device_error(void* workspace, pda_stream_t stream, int32_t* code);

/*
 * GQA / MQA / MHA paged decode ("From MHA to MLA", sections 3-5; drill page,
 * sections ③-⑤).
 *   q             device [B, Hq, D] dtype; [B, S, Hq, D] when the plan's seq_len_q S > 1
 *   k_cache       device [num_blocks, P, Hkv, D] dtype
 *   v_cache       device [num_blocks, P, Hkv, D] dtype
 *   block_tables  device [B, max_blocks_per_seq] int32; only the first
 *                 ceil(ctx_b / P) entries of row b are read
 *   context_lens  device [B] int32, equal to the plan's host copy
 *   scale         softmax scale applied to q.k (e.g. 1/sqrt(D)); finite
 *   out           device [B, Hq, D] dtype ([B, S, Hq, D] when S > 1; written; rows of
 *                 other sequences untouched)
 *   lse           device [B, Hq] float32 natural-log LSE of the scaled logits ([B, Hq, S]
 *                 when S > 1, FlashMLA-ETAP "Usage" order), or NULL
 *   plan          from pda_plan_create with kind PDA_KIND_GQA
 *   workspace     device, pda_plan_workspace_bytes(plan) bytes, zeroed once
 * Slots past ctx in a sequence's last page and blocks not referenced by the
 * first ceil(ctx/P) table entries are never used, whatever they hold.
 */
PDA_API pda_status paged_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens,
                             float scale, void* out, float* lse, const pda_plan* plan,
                             void* workspace, pda_stream_t stream);

/*
 * paged_decode_attn over fp8 caches (plan created with kv_format PDA_KV_FP8_E4M3).
 *   k_cache, v_cache  device [num_blocks, P, Hkv, D] uint8 E4M3 codes, 16-byte aligned
 *   k_scale, v_scale  per-tensor dequantization scales (finite): K_j = e4m3(k) * k_scale,
 *                     V_j = e4m3(v) * v_scale
 * Every other argument, and the result, as for paged_decode_attn (q, out in the plan's
 * 16-bit dtype). A stale slot or an unused block may hold any code, NaN included.
 */
PDA_API pda_status paged_decode_attn_fp8(const void* q, const void* k_cache, const void* v_cache,
                                         float k_scale, float v_scale,
                                         const int32_t* block_tables, const int32_t* context_lens,
                                         float scale, void* out, float* lse, const pda_plan* plan,
                                         void* workspace, pda_stream_t stream);

/*
 * Absorbed MLA decode ("From MHA to MLA", section 6; FlashMLA-ETAP "Usage" and
 * "Supported configurations"): every query head attends to one shared record
 * per token of Dqk = head_dim_qk values, Dv = head_dim_v latent then 64 rope,
 * with (Dqk, Dv) = (576, 512) (kv_lora_rank 512) or (320, 256) (kv_lora_rank
 * 256). Scores use all Dqk values, values are the first Dv.
 *   q             device [B, Hq, Dqk] dtype (absorbed content query then rope query);
 *                 [B, S, Hq, Dqk] when the plan's seq_len_q S > 1
 *   kv_cache      device [num_blocks, 64, Dqk] dtype (one KV head)
 *   block_tables, context_lens, scale, plan (kind PDA_KIND_MLA), workspace: as above
 *   out           device [B, Hq, Dv] dtype; [B, S, Hq, Dv] when S > 1
 *   lse           device [B, Hq] float32 or NULL; [B, Hq, S] when S > 1
 * Hq: 16, 32 or a multiple of 64. With S > 1: S * Hq in {16, 32, 64}, or Hq a multiple
 * of 64 (the heads of each query token are then separate head groups, each reading the
 * sequence's pages).
 */
PDA_API pda_status mla_decode(const void* q, const void* kv_cache, const int32_t* block_tables,
                      const int32_t* context_lens, float scale, void* out, float* lse,
                      const pda_plan* plan, void* workspace, pda_stream_t stream);

/*
 * mla_decode over an E4M3 record cache ("Attention Kernel Variants: MQA, GQA, and MLA",
 * KV-cache arithmetic table: the DeepSeek-V3 MLA row with an fp8 latent, 34.3 KiB per
 * token; plan created with kv_format PDA_KV_FP8_E4M3).
 *   kv_cache   device [num_blocks, 64, Dqk] uint8 E4M3 codes, 16-byte aligned
 *   kv_scale   the record's per-tensor dequantization scale (finite): rec = e4m3(code) * kv_scale,
 *              for the scores (all Dqk values) and the values (the first Dv) alike
 * Every other argument, and the result, as for mla_decode (q, out in the plan's 16-bit
 * dtype). Supported: seq_len_q * num_q_heads in {16, 32}. A stale slot or an unused block
 * may hold any code, NaN included.
 */
PDA_API pda_status mla_decode_fp8(const void* q, const void* kv_cache, float kv_scale,
                                  const int32_t* block_tables, const int32_t* context_lens,
                                  float scale, void* out, float* lse, const pda_plan* plan,
                                  void* workspace, pda_stream_t stream);

/*
 * Flash-Decoding combine on its own ("From MHA to MLA", section 4): for each
 * of `rows` rows, merge `num_splits` locally normalized partial outputs:
 *   L = max_s L_s + ln sum_s exp(L_s - max_s L_s),   out = sum_s exp(L_s - L) O_s
 * Splits with L_s = -inf carry no weight.
 *   partial_out  device [rows, num_splits, head_dim_v] float32
 *   partial_lse  device [rows, num_splits] float32 (natural log)
 *   out          device [rows, head_dim_v] in out_dtype (pda_dtype)
 *   lse          device [rows] float32, or NULL
 * head_dim_v: a multiple of 4, at most 1024. rows >= 0, num_splits >= 1.
 */
PDA_API pda_status pda_combine_splits(const float* partial_out, const float* partial_lse, int32_t rows,
                              int32_t num_splits, int32_t head_dim_v, void* out,
                              int32_t out_dtype, float* lse, pda_stream_t stream);

/*
 * GQA / MQA / MHA paged decode without a caller-provided workspace.
 *
 * The sources this library follows have no counterpart to this call: it exists
 * for callers that cannot allocate device memory when they decode, for example
 * code running inside another framework's memory pool, a plug-in that is only
 * handed input and output buffers, or a host that must not call cudaMalloc
 * after start-up. It computes exactly what paged_decode_attn computes, with the
 * same arguments minus `workspace`.
 *
 * Its split pieces, merge counters and error word live instead in one
 * library-owned device array of PDA_NO_ALLOC_WORKSPACE_BYTES (16 MiB) that every
 * GPU which loads this library keeps until the process exits. The call
 * allocates nothing and calls no allocating routine:
 *  - the first call on a device looks up that device's address of the array
 *    (once per device, with that device current) and keeps it for the life of
 *    the process; make that first call before any stream capture. The kept
 *    address is not valid after cudaDeviceReset on that device: a process that
 *    resets a device must not use this call (or its error reader) there again;
 *  - each call clears the array's merge counters on `stream` before its kernel
 *    runs; the split pieces need no clearing (they are written before read);
 *  - every call shares the one array, so calls that can overlap on the GPU
 *    (different streams, or several host threads) race and give wrong results;
 *    issue them on one stream, or serialize them;
 *  - a plan whose workspace exceeds the array (pda_plan_workspace_bytes(plan) >
 *    PDA_NO_ALLOC_WORKSPACE_BYTES) is rejected with PDA_ERR_WORKSPACE.
 * Device-side errors (a block id outside the pool, a timed-out wait: the codes of
 * pda_read_device_error) accumulate in the array's own error word across calls
 * until pda_no_alloc_read_device_error reads and clears it.
 */
#define PDA_NO_ALLOC_WORKSPACE_BYTES (16u << 20)
PDA_API pda_status paged_decode_attn_no_alloc(const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_tables,
                                              const int32_t* context_lens, float scale, void* out,
                                              float* lse, const pda_plan* plan,
                                              pda_stream_t stream);

/*
 * Read and clear the device error word of paged_decode_attn_no_alloc's library array
 * on the current device (synchronizes `stream`). *code as for pda_read_device_error:
 * 0 = no error; bit 0: a block-table entry of a read page was outside [0, num_blocks)
 * (that page was read as zeros); bit 1: a pipeline wait timed out and the kernel
 * abandoned its work. Like the decode call it allocates nothing, and it has no
 * counterpart in the sources this library follows.
 */
PDA_API pda_status pda_no_alloc_read_device_error(pda_stream_t stream, int32_t* code);

/*
 * Append the S new tokens of every sequence to the caches ("From MHA to MLA", section 2:
 * at each decode step the new key and value are appended to the cache; section 5: token
 * n of sequence b lives in block block_tables[b][n / P], slot n % P). S is the plan's
 * seq_len_q; the new tokens are sequence b's logical tokens context_lens[b] - S + i, so
 * context_lens already counts them (the same lengths the decode call then takes).
 *   GQA plan (pda_kv_append):
 *     k_new, v_new    device [B, S, Hkv, D] in the plan's dtype, 16-byte aligned
 *     k_cache, v_cache device [num_blocks, P, Hkv, D] (plan's dtype), written in place
 *   MLA plan (pda_mla_append): kv_new [B, S, Dqk] into kv_cache [num_blocks, 64, Dqk]
 *   block_tables, context_lens device, as for the decode calls; the entries that hold the
 *                   new tokens must already be assigned (see pda_pool_grow)
 *   workspace       the plan's workspace (only its error word is used)
 * A new token whose table entry is outside [0, num_blocks), or whose position is outside
 * the table or negative, is not written and sets bit 0 of the device error word.
 * Asynchronous on `stream`; no other cache entry is touched.
 */
PDA_API pda_status pda_kv_append(const void* k_new, const void* v_new, void* k_cache,
                                 void* v_cache, const int32_t* block_tables,
                                 const int32_t* context_lens, const pda_plan* plan,
                                 void* workspace, pda_stream_t stream);

/* pda_kv_append into E4M3 caches (plan kv_format PDA_KV_FP8_E4M3): each value x is
 * stored as the E4M3 code of x / scale, the division in fp32 (IEEE, round to nearest),
 * rounded once to nearest-even and saturated to +-448 (NaN stays NaN). k_scale and
 * v_scale (finite, nonzero) are the tensors' dequantization scales. */
PDA_API pda_status pda_kv_append_fp8(const void* k_new, const void* v_new, void* k_cache,
                                     void* v_cache, float k_scale, float v_scale,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     const pda_plan* plan, void* workspace, pda_stream_t stream);

/* pda_mla_append takes plans of 16-bit record caches (kv_format PDA_KV_SAME_AS_Q); an
 * E4M3 plan is refused with PDA_ERR_INVALID_ARG. */
PDA_API pda_status pda_mla_append(const void* kv_new, void* kv_cache,
                                  const int32_t* block_tables, const int32_t* context_lens,
                                  const pda_plan* plan, void* workspace, pda_stream_t stream);

/* pda_mla_append into an E4M3 record cache (MLA plan with kv_format PDA_KV_FP8_E4M3, the
 * variants page's fp8 latent): kv_new [B, S, Dqk] in the plan's dtype is stored as the
 * E4M3 codes of x / kv_scale into kv_cache [num_blocks, 64, Dqk] bytes, with the
 * quantization of pda_kv_append_fp8. kv_scale (finite, nonzero) is the record cache's
 * dequantization scale, the one mla_decode_fp8 takes. */
PDA_API pda_status pda_mla_append_fp8(const void* kv_new, void* kv_cache, float kv_scale,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      const pda_plan* plan, void* workspace,
                                      pda_stream_t stream);

/*
 * Physical block pool behind the block tables ("From MHA to MLA", section 5: requests'
 * logical pages map to one shared physical pool). Host memory only; one thread at a time
 * per pool. Blocks are ids in [0, num_blocks); a new pool hands them out as 0, 1, 2, ...
 * and a released block is handed out before the older free ones.
 */
typedef struct pda_block_pool pda_block_pool;  /* opaque, owned by the library */

PDA_API pda_status pda_pool_create(pda_block_pool** pool, int64_t num_blocks);
PDA_API void pda_pool_destroy(pda_block_pool* pool);
PDA_API int64_t pda_pool_num_free(const pda_block_pool* pool);

/* Grow one sequence from old_len to new_len tokens: assigns blocks to its logical pages
 * ceil(old_len / page_size) .. ceil(new_len / page_size) - 1, writing them into the host
 * table row (max_blocks_per_seq entries). All or nothing: PDA_ERR_OUT_OF_BLOCKS, with the
 * row and the pool unchanged, when too few blocks are free. */
PDA_API pda_status pda_pool_grow(pda_block_pool* pool, int32_t* table_row,
                                 int32_t max_blocks_per_seq, int32_t page_size,
                                 int32_t old_len, int32_t new_len);

/* Return the blocks of a finished sequence (its first ceil(len / page_size) entries) to
 * the pool and set those entries to -1. An entry that is not an in-use block of this pool,
 * or a block listed twice, fails with PDA_ERR_INVALID_ARG and changes nothing. */
PDA_API pda_status pda_pool_release(pda_block_pool* pool, int32_t* table_row,
                                    int32_t page_size, int32_t len);

/* Static name of a status code. */
PDA_API const char* pda_status_string(pda_status status);

/* One-line description of the last failed call on this thread ("" if none). */
PDA_API const char* pda_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PDA_H_ */
