/*
 * msa.h -- C ABI of libmsa, MSA block-sparse attention for GB300 (sm_103a).
 *
 * The method: every query token attends, for each KV head, only to the keys
 * of the 128-token KV-cache pages that an indexer selected for it (top-16
 * page ids per token and KV head), with a causal mask inside the page that
 * holds the query.  Sources:
 *   [P2] vLLM PR 60684, "MSA prefill takes the E4M3 query natively":
 *        Overview (E4M3 query over vLLM's packed K|V pages), Details /
 *        "Kernel capability" (E4M3 QK and PV MMAs), Details / "Scales"
 *        (q scale folds into the softmax scale, per-tensor K/V scales),
 *        Details / "Numerics" (probabilities rounded to E4M3), Validation
 *        (acceptance rule), Performance (build_k2q_csr + attention + combine
 *        timed per layer; top-k 16, page 128).
 *   [P4] vLLM docs, vllm.models.minimax_m3.nvidia.sparse_attention_msa,
 *        MiniMaxM3SparseMSAImpl.forward: build_k2q_csr(topk [H, T, 16],
 *        cu_seqlens_q, cu_seqlens_k, 128, total_rows=total_kv_blocks,
 *        qhead_per_kv) -> (row_ptr, q_indices, schedule), then
 *        sparse_atten_func(q, k_cache, v_cache, row_ptr, q_indices, topK=16,
 *        blk_kv=128, causal=True, softmax_scale, cu_seqlens_q/k,
 *        page_table=block_table, seqused_k=seq_lens, schedule, out=...).
 *   [P1] vLLM PR 60930, Details / "Host sync": the plan runs on the device,
 *        with no device-to-host copy, and the run call allocates nothing.
 *
 * Conventions for every call
 *   - All array arguments are DEVICE pointers unless stated otherwise; the
 *     caller owns every buffer (inputs, outputs and workspaces).  The library
 *     never allocates, frees or synchronises on the compute calls, so they
 *     can be captured in a CUDA graph.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *   - Return value: MSA_OK, or an MSA_ERR_* code detected on the host before
 *     anything is launched (then nothing was launched), or MSA_ERR_CUDA when
 *     a launch failed.
 *   - Problems that only the device can see (a page id past its request's
 *     pages, a block_table entry outside the pool, inconsistent cu_seqlens, a
 *     bounded wait that expired) never fault: the offending entry is skipped
 *     and a bit is set in the plan's device status word (MSA_STATUS_*), which
 *     msa_read_status() returns.
 *   - Fixed shape constants: head dim 128, page 128 tokens, top-k 16 ([P2]
 *     Performance; [P4] forward).  The GQA group G = Hq / Hkv may be any
 *     value from 1 to 128 (query head hq reads KV head hq / G).
 *   - E4M3 is the OCP float8 E4M3 ("fn") format, one byte per element.
 */
#ifndef MSA_H
#define MSA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MSA_API __attribute__((visibility("default")))
#else
#define MSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define MSA_HEAD_DIM 128
#define MSA_PAGE_SIZE 128
#define MSA_TOPK 16

/* host-side return codes */
#define MSA_OK 0
#define MSA_ERR_SHAPE 1       /* a size, count or stride is out of range     */
#define MSA_ERR_UNSUPPORTED 2 /* e.g. G outside 1..128, Hq not a multiple    */
#define MSA_ERR_ALIGN 3       /* a pointer is not aligned as documented       */
#define MSA_ERR_WORKSPACE 4   /* workspace NULL or smaller than required      */
#define MSA_ERR_CUDA 5        /* a CUDA runtime / driver call failed          */
#define MSA_ERR_NULL 6        /* a required pointer is NULL                   */
#define MSA_ERR_TOO_LARGE 7   /* beyond msa_decode_noalloc's fixed scratch    */
#define MSA_ERR_BUSY 8        /* msa_decode_noalloc entered from two threads  */

/* device status bits (msa_read_status) */
#define MSA_STATUS_BAD_PAGE_ID (1u << 0)  /* top-k id >= page count, or < -1 */
#define MSA_STATUS_BAD_BLOCK (1u << 1)    /* block_table entry not a page    */
#define MSA_STATUS_BAD_SEQLENS (1u << 2)  /* cu_seqlens inconsistent/too big */
#define MSA_STATUS_ROWS_OVERFLOW (1u << 3)/* sum of page counts > total_rows */
#define MSA_STATUS_TIMEOUT (1u << 4)      /* a bounded device wait expired   */
#define MSA_STATUS_BAD_WORK (1u << 5)     /* inconsistent work item skipped  */

/* element types of split partials (msa_combine) */
#define MSA_DTYPE_F32 0
#define MSA_DTYPE_BF16 1

/*
 * NVFP4 K/V pages ([P2] Details / "Kernel capability": with an E4M3 query,
 * each NVFP4 code times its block scale is dequantised to E4M3, the K global
 * scale is applied to the scores and the V global scale in the combine;
 * Details / "Numerics": K and V are rounded to E4M3.  [P4]
 * MiniMaxM3SparseMSANvfp4Backend: each KV head's K and V are two slots of
 * packed data plus block scales.)  The pages name the parts, not their byte
 * order; this library's layout, per (page, KV head), is the K slot then the
 * V slot, MSA_NVFP4_SLOT_BYTES each:
 *   codes   128 tokens x 64 bytes of E2M1 (OCP FP4: sign in bit 3, 2-bit
 *           exponent with bias 1, one mantissa bit); element 2i of a token
 *           in the low nibble of byte i, element 2i+1 in the high nibble
 *   scales  128 tokens x 8 E4M3 block scales, finite; scale b covers
 *           elements 16b .. 16b+15 of its token
 * so a pool is [num_pages][Hkv][MSA_NVFP4_PAGE_HEAD_BYTES] bytes.  Element
 * e of token t reads as E4M3(code x scale), rounded to nearest even and
 * saturated at 448; its real value is that times the K (or V) global scale.
 */
#define MSA_NVFP4_SLOT_BYTES 9216
#define MSA_NVFP4_PAGE_HEAD_BYTES 18432

/* KV page formats (AttnArgs::kv_format inside the library) */
#define MSA_KV_E4M3 0
#define MSA_KV_NVFP4 1

/*
 * The page-to-query plan.  msa_plan() fills this host struct; its pointers
 * point into the caller's plan workspace and at the caller's cu_seqlens
 * arrays, which must stay alive and unchanged until the last msa_prefill()
 * that uses the plan has run on the stream.  All fields are 64-bit so the
 * layout is the same for every compiler and for ctypes.
 *
 * CSR ([P4] build_k2q_csr): rows are (KV head h, request b, logical page p)
 * with row index r = h * total_rows + req_off[b] + p, where req_off[b] is the
 * sum of the page counts ceil(seq_len / 128) of requests before b.  Row r
 * lists, in ascending token order, the query tokens t whose top-k list for
 * head h holds page p (first occurrence, not after t's own page, valid id),
 * each with `slot` = the list position j of that first occurrence.
 * work (the schedule): 4 int32 per item {csr start, token count, b,
 * (h << 24) | p}; rows in ascending order, each cut into chunks of
 * chunk_tokens = floor(128 / G) tokens; the item count is counters[1].
 * records: the same items as the attention kernel reads them, record_bytes
 * each: an int4 header {KV row of the page in the pool, token count, first
 * key position of the page, first query head} and one int4 per token
 * {global token id, query position, slot j, 0}.
 */
typedef struct msa_plan {
  int64_t B, T, Hq, Hkv, total_rows, max_seqlen_q, max_seqlen_k, num_pages;
  int64_t bt_stride, bitmap_words, chunk_tokens, max_nnz, max_work, rows;
  int64_t record_bytes;
  const int32_t *cu_seqlens_q; /* caller's [B+1]                            */
  const int32_t *cu_seqlens_k; /* caller's [B+1]                            */
  int32_t *req_off;            /* [B+1]                                     */
  uint32_t *bitmap;            /* [rows * bitmap_words] token membership    */
  int32_t *word_pre;           /* [rows * bitmap_words] tokens before word  */
  int32_t *row_cnt;            /* [rows] entries of the row                 */
  int32_t *row_loc;            /* [rows][2] entries, work items before the
                                  row within its row tile                   */
  uint64_t *tile_state;        /* [row tiles] tile totals                   */
  int32_t *row_ptr;            /* [rows + 1]                                */
  int32_t *q_idx;              /* [max_nnz] global query token ids          */
  uint8_t *slot;               /* [max_nnz] top-k position j                */
  int32_t *work;               /* [max_work * 4]                            */
  void *records;               /* [max_work * record_bytes]                 */
  int32_t *counters;           /* [0] nnz, [1] work items, [2] plan valid   */
  uint16_t *slot_mask;         /* [T * Hkv] bit j: slot j holds a partial  */
  uint32_t *status;            /* [1] MSA_STATUS_* bits                     */
} msa_plan_t;

/* Library version (major * 10000 + minor * 100 + patch). */
MSA_API int msa_version(void);

/* Text for an MSA_ERR_* code. */
MSA_API const char *msa_status_string(int code);

/*
 * Bytes of device workspace msa_plan() needs for these bounds.
 *   B requests, T query tokens in total, Hq query heads, Hkv KV heads,
 *   total_rows >= the sum
 *   over requests of ceil(seq_len / 128) (vLLM's total_kv_blocks),
 *   max_seqlen_q >= every request's query length.
 * Returns MSA_ERR_SHAPE for negative sizes or a result that overflows,
 * MSA_ERR_UNSUPPORTED when Hq / Hkv is not an integer in 1..128.
 */
MSA_API int msa_plan_workspace_bytes(int64_t B, int64_t T, int64_t Hq, int64_t Hkv,
                             int64_t total_rows, int64_t max_seqlen_q,
                             size_t *bytes);

/*
 * build_k2q_csr + schedule on the device ([P4] forward; [P1] "Host sync":
 * plan on device, no device-to-host copy).
 *   topk          int32 [T][Hkv][16]  logical page ids of the token's own
 *                 request; -1 = padding.  Ids past the request's pages or
 *                 below -1 set MSA_STATUS_BAD_PAGE_ID and are skipped; a
 *                 repeated id counts once; an id after the token's own page
 *                 is dropped (fully masked by the causal rule).
 *   cu_seqlens_q  int32 [B+1]  prefix sums of query lengths, [0] = 0, [B] = T
 *   cu_seqlens_k  int32 [B+1]  prefix sums of sequence lengths (cached keys
 *                 plus this chunk); request b's queries are the LAST
 *                 q_len_b positions of its seq_len_b tokens.
 *   block_table   int32 [B][bt_stride]  logical -> physical page, bt_stride
 *                 >= ceil(max_seqlen_k / 128) (else MSA_ERR_SHAPE); an entry
 *                 used by a valid selection must lie in [0, num_pages), else
 *                 MSA_STATUS_BAD_BLOCK is set and that selection is skipped.
 *   Hq, Hkv       query / KV heads; Hq % Hkv == 0, 1 <= Hq / Hkv <= 128.
 *   total_rows, max_seqlen_q, max_seqlen_k: host-known bounds (see above);
 *                 a request exceeding them sets MSA_STATUS_BAD_SEQLENS (or
 *                 ROWS_OVERFLOW) and the whole plan comes out empty.
 *   workspace     device buffer of msa_plan_workspace_bytes() bytes,
 *                 256-byte aligned; it holds the plan until it is rebuilt.
 *   plan          host struct, filled on return.
 * Launches 4 kernels on `stream`; never synchronises.
 */
MSA_API int msa_plan(const int32_t *topk, const int32_t *cu_seqlens_q,
             const int32_t *cu_seqlens_k, const int32_t *block_table,
             int64_t bt_stride, int64_t num_pages, int64_t B, int64_t T,
             int64_t Hq, int64_t Hkv, int64_t total_rows,
             int64_t max_seqlen_q, int64_t max_seqlen_k, void *workspace,
             size_t workspace_bytes, msa_plan_t *plan, void *stream);

/*
 * msa_plan for one shard of KV heads: heads [h_begin, h_begin + Hkv) of a
 * top-k tensor that holds topk_hkv KV heads per token.  Under tensor
 * parallelism a rank owns num_attention_heads / tp_size query heads and
 * the KV heads of its own cache ([P4] MiniMaxM3SparseMSAMetadataBuilder:
 * num_q_heads = num_attention_heads // tp_size); the heads shard with no
 * exchange inside the attention.  With this plan the rank passes its own
 * tensors to msa_prefill / msa_prefill_attention / msa_prefill_combine:
 * q [T][Hq][128] and out [T][Hq][128] hold the shard's Hq = Hkv * G query
 * heads, the pool its Hkv KV heads.  Each shard's result is bit-identical
 * to the same heads of one unsharded call.
 *   topk       int32 [T][topk_hkv][16] (the whole tensor, not a copy of
 *              the slice)
 *   topk_hkv   KV heads in topk's layout, 1 .. 127
 *   h_begin    first KV head of the shard; h_begin + Hkv <= topk_hkv
 *   (the other arguments as msa_plan, Hq and Hkv those of the shard)
 * Returns MSA_ERR_SHAPE when the head range does not fit.  Launches the same
 * 4 kernels as msa_plan.
 */
MSA_API int msa_plan_heads(const int32_t *topk, int64_t topk_hkv, int64_t h_begin,
                   const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                   const int32_t *block_table, int64_t bt_stride, int64_t num_pages,
                   int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t total_rows,
                   int64_t max_seqlen_q, int64_t max_seqlen_k, void *workspace,
                   size_t workspace_bytes, msa_plan_t *plan, void *stream);

/*
 * Bytes of device workspace msa_prefill() needs: the split partials,
 * T * Hq * 16 * (128 E4M3 bytes + 1 fp32), plus the V scale for the combine.
 */
MSA_API int msa_prefill_workspace_bytes(int64_t T, int64_t Hq, size_t *bytes);

/*
 * Sparse attention over the planned pages, then the log-sum-exp combine
 * ([P4] sparse_atten_func; [P2] Overview and Details: E4M3 query over the
 * packed E4M3 K|V pages, E4M3 QK and PV MMAs, probabilities rounded to E4M3,
 * q scale folded into the softmax scale).
 *   q            E4M3 [T][Hq][128], 16-byte aligned
 *   kv           E4M3 [num_pages][Hkv][128][256]: per token, K in bytes
 *                0..127 and V in bytes 128..255 ([P4]: kv_cache.split(D));
 *                16-byte aligned; num_pages * Hkv * 128 < 2^31
 *   q_scale, k_scale, v_scale  per-tensor dequantisation scales (host)
 *   softmax_scale  e.g. 1/sqrt(128); score = (q.k) * q_scale * k_scale *
 *                softmax_scale
 *   block_table  as in msa_plan (the same table)
 *   plan         from msa_plan() for the same batch
 *   workspace    msa_prefill_workspace_bytes() bytes, 256-byte aligned
 *   out          bf16 [T][Hq][128] (round to nearest even); a (token, head)
 *                with no attended key gets zeros
 *   lse          fp32 [T][Hq] natural-log sum of exp(score), or NULL;
 *                -inf where no key is attended
 * Launches the attention kernel (tcgen05 / TMA / TMEM, persistent over the
 * plan's work list) and the combine kernel on `stream`.
 */
MSA_API int msa_prefill(const uint8_t *q, const uint8_t *kv, int64_t num_pages,
                float q_scale, float k_scale, float v_scale,
                float softmax_scale, const int32_t *block_table,
                int64_t bt_stride, const msa_plan_t *plan, void *workspace,
                size_t workspace_bytes, uint16_t *out, float *lse,
                void *stream);

/*
 * The two halves of msa_prefill, for callers that schedule or time them
 * separately; msa_prefill(...) is exactly msa_prefill_attention(...)
 * followed by msa_prefill_combine(...) on the same workspace.
 *   msa_prefill_attention: the attention kernel only; writes the split
 *     partials into `workspace`: one per token, query head and top-k slot,
 *     the normalised O in E4M3 in V's code units (a convex combination of
 *     E4M3 V codes, so always in range) and the lse in fp32, plus v_scale.
 *     Arguments as in msa_prefill.
 *   msa_prefill_combine: merges the partials that msa_prefill_attention left
 *     in `workspace` (slots the plan marked empty are skipped) into out / lse.
 */
MSA_API int msa_prefill_attention(const uint8_t *q, const uint8_t *kv,
                                  int64_t num_pages, float q_scale,
                                  float k_scale, float v_scale,
                                  float softmax_scale,
                                  const int32_t *block_table,
                                  int64_t bt_stride, const msa_plan_t *plan,
                                  void *workspace, size_t workspace_bytes,
                                  void *stream);
MSA_API int msa_prefill_combine(const msa_plan_t *plan, void *workspace,
                                size_t workspace_bytes, uint16_t *out,
                                float *lse, void *stream);

/*
 * NVFP4 page-heads -> E4M3 pool: the cache exactly as the NVFP4 attention
 * reads it (layout and rounding above).  kv8[ph][t][0..127] is token t's K,
 * kv8[ph][t][128..255] its V; page-head ph = page * Hkv + KV head.
 *   kv4   [page_heads][MSA_NVFP4_PAGE_HEAD_BYTES], 16-byte aligned
 *   kv8   E4M3 [page_heads][128][256], 16-byte aligned, not overlapping kv4
 * One HBM-bound kernel on `stream`.
 */
MSA_API int msa_nvfp4_to_e4m3(const uint8_t *kv4, int64_t page_heads,
                              uint8_t *kv8, void *stream);

/*
 * msa_prefill over an NVFP4 pool: the same arguments, with kv4 in place of
 * kv ([num_pages][Hkv][MSA_NVFP4_PAGE_HEAD_BYTES], 16-byte aligned) and
 * k_scale / v_scale the K and V global scales.  Each selected (page, KV
 * head) is read in its NVFP4 form (18 KB instead of 32 KB) and dequantised
 * to E4M3 in shared memory; the result is the one msa_prefill gives on the
 * E4M3 pool that msa_nvfp4_to_e4m3() writes, with the same scales.
 * Workspace: msa_prefill_workspace_bytes().
 */
MSA_API int msa_prefill_nvfp4(const uint8_t *q, const uint8_t *kv4,
                              int64_t num_pages, float q_scale, float k_scale,
                              float v_scale, float softmax_scale,
                              const int32_t *block_table, int64_t bt_stride,
                              const msa_plan_t *plan, void *workspace,
                              size_t workspace_bytes, uint16_t *out,
                              float *lse, void *stream);

/* The attention half of msa_prefill_nvfp4 (see msa_prefill_attention);
 * msa_prefill_combine() finishes it. */
MSA_API int msa_prefill_attention_nvfp4(const uint8_t *q, const uint8_t *kv4,
                                        int64_t num_pages, float q_scale,
                                        float k_scale, float v_scale,
                                        float softmax_scale,
                                        const int32_t *block_table,
                                        int64_t bt_stride,
                                        const msa_plan_t *plan,
                                        void *workspace,
                                        size_t workspace_bytes, void *stream);

/*
 * msa_prefill with a BF16 query ([P2] Details / "Kernel capability": the
 * BF16-Q x FP8-K/V mode stages K/V up to BF16 and runs BF16 MMAs; Overview:
 * the BF16 query is the E4M3 query dequantised, q_scale applied).
 *   q16   bf16 [T][Hq][128] (uint16 codes), 16-byte aligned; q_scale still
 *         multiplies the scores (1.0 for a query that carries its scale)
 * Every other argument, the workspace and the outputs as in msa_prefill
 * (E4M3 pool only).  Each selected page's K and V are widened to bf16 in
 * shared memory (exact), QK and PV run as bf16 tensor-core MMAs with fp32
 * accumulation, probabilities are rounded to bf16; the split partials and
 * the combine are msa_prefill's.
 */
MSA_API int msa_prefill_bf16q(const uint16_t *q16, const uint8_t *kv,
                              int64_t num_pages, float q_scale, float k_scale,
                              float v_scale, float softmax_scale,
                              const int32_t *block_table, int64_t bt_stride,
                              const msa_plan_t *plan, void *workspace,
                              size_t workspace_bytes, uint16_t *out,
                              float *lse, void *stream);

/* The attention half of msa_prefill_bf16q (see msa_prefill_attention);
 * msa_prefill_combine() finishes it. */
MSA_API int msa_prefill_attention_bf16q(const uint16_t *q16, const uint8_t *kv,
                                        int64_t num_pages, float q_scale,
                                        float k_scale, float v_scale,
                                        float softmax_scale,
                                        const int32_t *block_table,
                                        int64_t bt_stride,
                                        const msa_plan_t *plan,
                                        void *workspace,
                                        size_t workspace_bytes, void *stream);

/*
 * Merge split partials by log-sum-exp ([P2] Performance: "combine" is the
 * third step of the per-layer call; Validation: probabilities are rounded
 * per split).  For each row r:
 *   M = max_j lse[r][j];  L = M + ln sum_j exp(lse[r][j] - M);
 *   out[r] = sum_j exp(lse[r][j] - L) * part_o[r][j]   (bf16, nearest even)
 *   lse_out[r] = L
 *   part_o     [rows][splits][128], MSA_DTYPE_F32 or MSA_DTYPE_BF16, each
 *              partial already normalised by its own softmax sum
 *   part_lse   fp32 [rows][splits]; -inf marks an empty split; a row with
 *              no filled split gives zeros and lse -inf
 *   lse_out    fp32 [rows] or NULL
 * 1 <= splits <= 64.
 */
MSA_API int msa_combine(const void *part_o, int part_dtype, const float *part_lse,
                int64_t rows, int64_t splits, uint16_t *out, float *lse_out,
                void *stream);

/*
 * Bytes of device workspace msa_decode() needs for these bounds.
 */
MSA_API int msa_decode_workspace_bytes(int64_t B, int64_t n, int64_t Hq, int64_t Hkv,
                               int64_t max_seqlen_k, size_t *bytes);

/*
 * Decode / speculative verify ([P4] forward, decode branch: the E4M3 query
 * of n = 1..8 tokens per request -- one regular token, or k drafts plus
 * one -- attends over the same packed pages with per-token top-k lists).
 * Request b's n query tokens sit at positions seq_lens[b] - n .. seq_lens[b]-1
 * and are causal among themselves.  Built from the same plan, attention and
 * combine kernels as prefill: each (KV head, page) selected by the batch is
 * read once and its partials merged by log-sum-exp.
 *   q          E4M3 [B*n][Hq][128]
 *   topk       int32 [B*n][Hkv][16]
 *   seq_lens   int32 [B] (device), each in [n, max_seqlen_k]
 *   workspace  msa_decode_workspace_bytes() bytes, 256-byte aligned
 *   plan_out   optional host struct (NULL allowed) that receives the plan,
 *              e.g. for msa_read_status()
 *   out, lse   as in msa_prefill, [B*n][Hq][...]
 */
MSA_API int msa_decode(const uint8_t *q, const uint8_t *kv, int64_t num_pages,
               float q_scale, float k_scale, float v_scale,
               float softmax_scale, const int32_t *topk,
               const int32_t *block_table, int64_t bt_stride,
               const int32_t *seq_lens, int64_t B, int64_t n, int64_t Hq,
               int64_t Hkv, int64_t max_seqlen_k, void *workspace,
               size_t workspace_bytes, uint16_t *out, float *lse,
               msa_plan_t *plan_out, void *stream);

/*
 * msa_decode over an NVFP4 pool: kv4 as in msa_prefill_nvfp4, k_scale /
 * v_scale the global scales, everything else as in msa_decode.
 */
MSA_API int msa_decode_nvfp4(const uint8_t *q, const uint8_t *kv4,
                             int64_t num_pages, float q_scale, float k_scale,
                             float v_scale, float softmax_scale,
                             const int32_t *topk, const int32_t *block_table,
                             int64_t bt_stride, const int32_t *seq_lens,
                             int64_t B, int64_t n, int64_t Hq, int64_t Hkv,
                             int64_t max_seqlen_k, void *workspace,
                             size_t workspace_bytes, uint16_t *out, float *lse,
                             msa_plan_t *plan_out, void *stream);

/*
 * msa_decode for callers that cannot allocate device memory -- for example
 * code that only receives raw device pointers through a foreign-function
 * boundary and has no access to an allocator, or that runs where allocating
 * is not allowed.  It takes the same arguments as msa_decode except the
 * workspace and plan_out, and computes the same result with the same
 * kernels.  (The pages have no counterpart; this is a library convenience.)
 *
 * Its scratch -- the sequence prefix sums, the plan and the split partials
 * that msa_decode keeps in the caller's workspace -- lives in one fixed
 * array of MSA_NOALLOC_SCRATCH_BYTES (16 MiB) of device memory that every GPU
 * which loads this library holds until the process exits.  The call itself
 * allocates and frees nothing.
 *   - A batch whose msa_decode_workspace_bytes() exceeds that size is
 *     rejected with MSA_ERR_TOO_LARGE before anything is launched.
 *   - Every call outside stream capture looks up the array's device address
 *     in the current device's context (a runtime call; the first one on a
 *     device also loads the module).  A call made while `stream` is being
 *     captured reuses the address of that device's last call outside
 *     capture, so make one call on each device before capturing; without
 *     one the captured call returns MSA_ERR_CUDA.
 *   - All calls share the one array and each overwrites it (the parts that
 *     must start at zero are cleared by every call).  Calls whose work
 *     overlaps on the GPU -- on different streams, or from several host
 *     threads -- race and must not be issued.  A call entered while another
 *     host thread is inside this function returns MSA_ERR_BUSY without
 *     launching anything; the GPU-side overlap of calls enqueued one after
 *     another on different streams cannot be seen here and stays the
 *     caller's to avoid.
 *   - Device status bits are not returned (there is no plan_out).
 */
#define MSA_NOALLOC_SCRATCH_BYTES (16u << 20)
MSA_API int msa_decode_noalloc(const uint8_t *q, const uint8_t *kv,
                               int64_t num_pages, float q_scale,
                               float k_scale, float v_scale,
                               float softmax_scale, const int32_t *topk,
                               const int32_t *block_table, int64_t bt_stride,
                               const int32_t *seq_lens, int64_t B, int64_t n,
                               int64_t Hq, int64_t Hkv, int64_t max_seqlen_k,
                               uint16_t *out, float *lse, void *stream);

/*
 * For tests of the expiry path only: sets the wall-time limit, in
 * nanoseconds, of the attention kernel's pipeline waits for every later
 * launch in this process; 0 restores the default of about one second.  With
 * a limit shorter than a page load, a wait runs out: the kernel sets
 * MSA_STATUS_TIMEOUT, stops issuing work, lets the copies and MMAs it has
 * already started land (those drain waits keep the full limit), frees its
 * tensor memory and returns; the outputs of that call are not meaningful,
 * and the next call on the same workspaces computes normally.  (The pages
 * have no counterpart; this is a library test hook.)
 */
MSA_API int msa_test_set_wait_limit_ns(uint64_t ns);

/*
 * Copies the plan's device status word to *status.  This call synchronises
 * the device (it is meant for tests and debugging, not the hot path).
 */
MSA_API int msa_read_status(const msa_plan_t *plan, uint32_t *status);

/*
 * Copies the plan's device counters: *nnz = CSR entries, *num_work = work
 * items.  Synchronises the device (tests and debugging only).
 */
MSA_API int msa_read_counters(const msa_plan_t *plan, int64_t *nnz,
                      int64_t *num_work);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H */
