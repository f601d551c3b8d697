/*
 * mla_decode.h — C ABI of libmla_decode.so: paged FP8 multi-head latent
 * attention (MLA) decode with split-KV partials and an online-softmax merge,
 * for NVIDIA GB300 (sm_103a).
 *
 * The problem (TensorRT-LLM issue #20510, "CuTe DSL FP8 MLA decode
 * regression", sections "Setup" and "Repro 1/2"): each query row (head h of
 * query token qi of request b) attends over the request's paged KV cache.
 * A KV row is 576 E4M3 values: 512 latent + 64 rope.  K is the whole row, V is
 * its first 512 values.  Pages hold 32 tokens.  Q is E4M3; the output is BF16
 * with an optional fp32 log-sum-exp ("softmax stats").  The KV range of each
 * request is split across CTAs (split_kv); each split writes (max, sum, O)
 * partials that a merge kernel combines (TensorRT-LLM PR #20380, "split the
 * KV partials of a row across thread groups in fmhaReductionKernel",
 * "Description").
 *
 * Definition computed (all scales multiply the dequantised values):
 *   q   = q_scale * Q[b, qi, h, 0:576],  k_j = kv_scale * KV(token j),
 *   v_j = k_j[0:512],  s_j = softmax_scale * (q . k_j),
 *   visible keys j < n with n = L_b (or L_b - q_len + qi + 1 when causal:
 *   the MTP-verify block, query token i sees keys [0, L - q_len + i]),
 *   O = sum_j softmax(s)_j v_j  (BF16, round to nearest even),
 *   LSE = ln sum_j exp(s_j)     (natural log, fp32).
 *
 * Conventions for every function:
 *   - Return value is an mla_status_t.  Nothing throws, exits or aborts.
 *     On a non-OK return, mla_last_error() gives a message (thread-local).
 *   - Device pointers are plain CUDA device addresses; host pointers are
 *     marked "host".  The caller owns every buffer (including the workspace)
 *     and keeps it alive until the stream has passed the call.
 *   - The library never allocates device memory.  mla_decode and mla_merge
 *     enqueue work on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and return without synchronising, so they can be captured in a CUDA
 *     graph.
 *   - Conditions only the device can see (a page id outside [0, num_pages),
 *     inconsistent kv_lens/splits/chunks, a wait that ran out) are written to
 *     a status word at the head of the workspace; mla_decode_status() reads
 *     it.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,
  MLA_ERR_UNSUPPORTED = 2,
  MLA_ERR_WORKSPACE_TOO_SMALL = 3,
  MLA_ERR_CUDA = 4,
  MLA_ERR_TIMEOUT = 5
} mla_status_t;

#define MLA_HEAD_DIM 576
#define MLA_LATENT_DIM 512
#define MLA_ROPE_DIM 64
#define MLA_PAGE_SIZE 32
#define MLA_TILE_TOKENS 128 /* split chunks are multiples of this */
#define MLA_MAX_SPLITS 256  /* per-request split cap of the GB300 planner and the kernels */
#define MLA_PAGES_SPLIT_CAP 128 /* the pages' planner cap (issue #20510, "Repro 2") */
#define MLA_MAX_ROWS 1024   /* num_heads * q_len */

/*
 * Split planner (host only; issue #20510, "Repro 2": per-request plan
 * `block_split_kvs` with the split cap raised to 128, and the follow-up
 * comment on skewed batches and the minimum tiles per split).
 *
 * kv_lens      host int32[batch], each >= q_len >= 1.
 * num_heads    heads per request (H); num_heads * q_len <= MLA_MAX_ROWS.
 * sm_count     SMs of the target GPU (used when target_ctas <= 0).
 * target_ctas  > 0: reproduce the pages' planner: t = max(1, target/B)
 *              splits per request, chunk = roundup128(ceil(L/t)).  (A request
 *              with more than 96 rows runs each split as several row-group
 *              CTAs on top of that.)
 *              <= 0: GB300 planner: one common chunk for the whole batch,
 *              chosen to balance whole waves of one CTA per SM.
 * Outputs (host): splits_out[batch] (1..MLA_PAGES_SPLIT_CAP with a target,
 *              1..MLA_MAX_SPLITS for the GB300 planner: a single long request
 *              can then fill every SM), chunk_out[batch]
 *              (tokens per split, a multiple of 128, splits*chunk >= L),
 *              *kv_split_out (merge thread groups: the largest of 16, 8, 4, 2,
 *              1 with at least two partials per group and
 *              (num_heads * q_len * the requests with more than one split)
 *              * groups <= 6 * sm_count, with sm_count 152 when <= 0) and
 *              *workspace_bytes_out for mla_decode with max(splits).
 */
MLA_API int mla_decode_plan(const int32_t* kv_lens, int32_t batch, int32_t num_heads, int32_t q_len,
                    int32_t sm_count, int32_t target_ctas, int32_t* splits_out,
                    int32_t* chunk_out, int32_t* kv_split_out, size_t* workspace_bytes_out);

/*
 * CTA item list of a plan (host only): one entry per (request, split, row
 * group) that has work, packed as (b << MLA_ITEM_B_SHIFT) |
 * (split << MLA_ITEM_S_SHIFT) | row_group, in split-major order (every
 * request's split s before anyone's split s + 1).  Passed to the decode
 * through mla_decode_options_t.cta_items (a device copy) and num_ctas, it
 * replaces the batch x max_splits grid, whose empty slots (split >= splits[b])
 * a skewed batch has many of, by exactly the CTAs that have work (issue
 * #20510 follow-up: skewed batches, skip_empty_splits).
 *
 * splits      host int32[batch], as planned by mla_decode_plan.
 * items_out   host int32[capacity] or NULL (then only *n_items_out is set).
 * Errors: MLA_ERR_INVALID_ARG (null, batch > MLA_ITEM_MAX_BATCH, a split
 * count out of range, capacity too small), MLA_ERR_UNSUPPORTED (rows).
 */
#define MLA_ITEM_B_SHIFT 14
#define MLA_ITEM_S_SHIFT 5
#define MLA_ITEM_MAX_BATCH 65535
MLA_API int mla_decode_plan_items(const int32_t* splits, int32_t batch, int32_t num_heads,
                                  int32_t q_len, int32_t* items_out, int32_t capacity,
                                  int32_t* n_items_out);

/* The item list for the BF16 entry points (mla_decode_bf16_ex,
 * mla_decode_bf16_sparse): the same list, with the BF16 kernels' row groups
 * (at most 48 rows per CTA, where the FP8 kernels take up to 96).  Arguments
 * and errors as for mla_decode_plan_items. */
MLA_API int mla_decode_plan_items_bf16(const int32_t* splits, int32_t batch, int32_t num_heads,
                                       int32_t q_len, int32_t* items_out, int32_t capacity,
                                       int32_t* n_items_out);

/* Workspace bytes mla_decode needs: a 256-byte status header, then per
 * (row, split) an fp32 pair (m, l) and an fp32 O[512]. */
MLA_API size_t mla_decode_workspace_size(int32_t batch, int32_t q_len, int32_t num_heads,
                                 int32_t max_splits);

/*
 * Decode: split-KV kernel, then (if any request has more than one split) the
 * merge.  Row r = (b*q_len + qi)*num_heads + h.
 *
 * q_fp8          E4M3 [batch, q_len, num_heads, 576], contiguous, 16-byte aligned.
 * kv_pages_fp8   E4M3 [num_pages, 32, 576], contiguous, 16-byte aligned.
 * page_table     int32 [batch, max_pages_per_req]; entry i of request b is the
 *                page holding tokens [32i, 32i+32).  Only entries below
 *                ceil(kv_lens[b]/32) are read.
 * kv_lens, splits, chunks   int32 [batch] on the device, as planned by
 *                mla_decode_plan (splits[b] <= max_splits).
 * kv_split       merge thread groups (1, 2, 4, 8, 16).
 * causal         nonzero: MTP-verify mask inside the q_len block.
 * workspace      device buffer of >= mla_decode_workspace_size(...) bytes,
 *                256-byte aligned, its status header zeroed once by
 *                mla_decode_workspace_init.
 * out_bf16       BF16 [batch, q_len, num_heads, 512].
 * lse_f32        fp32 [batch, q_len, num_heads] or NULL.
 * out_f32_debug  fp32 [batch, q_len, num_heads, 512] or NULL: the output
 *                before the BF16 store (for tests).
 * Errors: MLA_ERR_INVALID_ARG (null or misaligned pointer, bad sizes),
 * MLA_ERR_WORKSPACE_TOO_SMALL, MLA_ERR_CUDA (launch failure).
 */
MLA_API int mla_decode(const void* q_fp8, const void* kv_pages_fp8, int64_t num_pages,
               const int32_t* page_table, int32_t max_pages_per_req, const int32_t* kv_lens,
               const int32_t* splits, const int32_t* chunks, int32_t max_splits,
               int32_t kv_split, int32_t batch, int32_t q_len, int32_t num_heads, int32_t causal,
               float q_scale, float kv_scale, float softmax_scale, void* workspace,
               size_t workspace_bytes, void* out_bf16, float* lse_f32, float* out_f32_debug,
               void* stream);

/*
 * Options of mla_decode_ex (issue #20510, "Repro 1/2" run() arguments and the
 * follow-up's device-side scales; PR #20380, "Description": sinks are handled
 * in the merge).
 *
 * q_scale_dev, kv_scale_dev, softmax_scale_dev  device fp32 pointers or NULL.
 *     When set, element 0 is read by the kernels instead of the host value, so
 *     a captured CUDA graph picks up new scales on replay without a host read.
 * output_scale  multiplies O (BF16 and fp32 outputs), not the LSE.  1 = off.
 * sinks  NULL or device fp32 [num_heads]: per-head attention-sink logit in the
 *     units of the scaled scores (natural log).  A sink acts as one more key
 *     with that logit and a zero value: it joins the softmax denominator, so
 *     O shrinks and LSE = ln(sum_j exp(s_j) + exp(sink)).
 * query_lens  NULL or device int32 [batch] (issue #20510, "Repro 1": the
 *     run() arguments is_var_q / query_lens; the pages do not define them, so
 *     this is the plain reading): request b has query_lens[b] query tokens,
 *     1 <= query_lens[b] <= q_len, in slots qi < query_lens[b] of the padded
 *     [batch, q_len, num_heads] row layout.  They are the request's last
 *     positions, so under causal slot qi sees keys j <= L - query_lens[b] + qi.
 *     Rows of the other slots see no key: O = 0, LSE = -inf (or the sink).
 *     Out-of-range values are reported as MLA_ERR_INVALID_ARG by the device.
 * kv_bounds  NULL or device int32 [batch][2] (issue #20510, "Repro 1": the
 *     run() argument kv_bounds; plain reading): keys restricted to
 *     lo <= j < hi for (lo, hi) = kv_bounds[b], intersected with [0, L) and
 *     the causal range.  Whole 128-token tiles below lo are skipped.
 * cta_items, num_ctas  NULL / 0, or the device copy of the item list of
 *     mla_decode_plan_items for this call's splits and its length: the
 *     split-KV kernel then launches exactly num_ctas CTAs.
 * persistent_ctas  0, or (with an item list) the number of persistent CTAs
 *     (issue #20510, "Repro 1": the run() argument is_persistent; plain
 *     reading): min(persistent_ctas, num_ctas) CTAs are launched and CTA c
 *     works on items c, c + grid, c + 2 grid, ... of the list, one after
 *     another, loading the next item's Q and first KV tiles while it
 *     finishes the current one, so each CTA's start-up is paid once.  The
 *     results are the same numbers as with one CTA per item.  FP8 entry
 *     points only (the BF16 ones return MLA_ERR_UNSUPPORTED).
 * phases  MLA_PHASE_ALL (0): the split-KV kernel, then the merge.
 *     MLA_PHASE_SPLIT: the split-KV kernel only (requests with one split get
 *     their final output, the others partials in the workspace).
 *     MLA_PHASE_MERGE: the merge only, of the partials that a MLA_PHASE_SPLIT
 *     call with the same arguments left in the workspace.  The two enqueued
 *     one after the other on one stream are the whole call, as
 *     mla_decode_splitkv and mla_decode_merge are for mla_decode (to time
 *     the kernels one by one, or to run other work between them).  Other
 *     values: MLA_ERR_INVALID_ARG.
 * Zero-initialise the structure: fields added later default to off.
 */
#define MLA_PHASE_ALL 0
#define MLA_PHASE_SPLIT 1
#define MLA_PHASE_MERGE 2
typedef struct {
  const float* q_scale_dev;
  const float* kv_scale_dev;
  const float* softmax_scale_dev;
  float output_scale;
  const float* sinks;
  const int32_t* query_lens;
  const int32_t* kv_bounds;
  const int32_t* cta_items;
  int32_t num_ctas;
  int32_t persistent_ctas;
  int32_t phases;
} mla_decode_options_t;

/* mla_decode with options (NULL options = mla_decode).  Same arguments,
 * checks and results otherwise. */
MLA_API int mla_decode_ex(const void* q_fp8, const void* kv_pages_fp8, int64_t num_pages,
                          const int32_t* page_table, int32_t max_pages_per_req,
                          const int32_t* kv_lens, const int32_t* splits, const int32_t* chunks,
                          int32_t max_splits, int32_t kv_split, int32_t batch, int32_t q_len,
                          int32_t num_heads, int32_t causal, float q_scale, float kv_scale,
                          float softmax_scale, void* workspace, size_t workspace_bytes,
                          void* out_bf16, float* lse_f32, float* out_f32_debug,
                          const mla_decode_options_t* options, void* stream);

/*
 * Sparse decode over selected pages (TensorRT-LLM PR #17441 "m3 decode perf":
 * the sparse MLA decode after the top-k block selector, which reads E4M3 q and
 * the paged FP8 cache directly).  Keys are restricted to the logical pages
 * listed per request:
 *
 * block_idx  device int32 [batch][topk]: logical page indices of request b
 *            (page p holds keys [32p, 32p + 32)), strictly increasing over
 *            the non-negative entries; negative entries are unused slots.
 *            Pages at or past ceil(L/32) hold no key and are skipped.  Order
 *            violations seen inside a split are reported as
 *            MLA_ERR_INVALID_ARG by the device.
 * topk       entries per request, >= 1.
 * kv_lens    the requests' true lengths L (the causal limit and the last
 *            page's tail come from them).
 * splits, chunks, max_splits, kv_split  the plan of mla_decode_plan for the
 *            compact lengths 32 * topk of every request: split s covers
 *            selection entries [s * chunk / 32, (s + 1) * chunk / 32).
 * options    as for mla_decode_ex (query_lens and kv_bounds also apply), or
 *            NULL.
 * Everything else is as for mla_decode.
 */
MLA_API int mla_decode_sparse(const void* q_fp8, const void* kv_pages_fp8, int64_t num_pages,
                              const int32_t* page_table, int32_t max_pages_per_req,
                              const int32_t* kv_lens, const int32_t* block_idx, int32_t topk,
                              const int32_t* splits, const int32_t* chunks, int32_t max_splits,
                              int32_t kv_split, int32_t batch, int32_t q_len, int32_t num_heads,
                              int32_t causal, float q_scale, float kv_scale, float softmax_scale,
                              void* workspace, size_t workspace_bytes, void* out_bf16,
                              float* lse_f32, float* out_f32_debug,
                              const mla_decode_options_t* options, void* stream);

/*
 * The two phases of mla_decode, for callers that schedule them separately
 * (to overlap other work, or to time the kernels one by one).  Same arguments
 * and checks as mla_decode.  mla_decode_splitkv launches the split-KV kernel:
 * requests with one split get their final output, the others get partials in
 * the workspace.  mla_decode_merge then launches the merge of those partials
 * (nothing when max_splits == 1).  mla_decode == splitkv followed by merge on
 * the same stream.
 */
MLA_API int mla_decode_splitkv(const void* q_fp8, const void* kv_pages_fp8, int64_t num_pages,
                               const int32_t* page_table, int32_t max_pages_per_req,
                               const int32_t* kv_lens, const int32_t* splits,
                               const int32_t* chunks, int32_t max_splits, int32_t kv_split,
                               int32_t batch, int32_t q_len, int32_t num_heads, int32_t causal,
                               float q_scale, float kv_scale, float softmax_scale,
                               void* workspace, size_t workspace_bytes, void* out_bf16,
                               float* lse_f32, float* out_f32_debug, void* stream);
MLA_API int mla_decode_merge(const void* q_fp8, const void* kv_pages_fp8, int64_t num_pages,
                             const int32_t* page_table, int32_t max_pages_per_req,
                             const int32_t* kv_lens, const int32_t* splits,
                             const int32_t* chunks, int32_t max_splits, int32_t kv_split,
                             int32_t batch, int32_t q_len, int32_t num_heads, int32_t causal,
                             float q_scale, float kv_scale, float softmax_scale,
                             void* workspace, size_t workspace_bytes, void* out_bf16,
                             float* lse_f32, float* out_f32_debug, void* stream);

/*
 * BF16-KV decode: the same method and split plan with a BF16 cache (issue
 * #20510, "Repro 2": the BF16 kernel mla_decode_fp16.py, 512 latent + 64 rope,
 * page size 32, BF16 output).  Q and KV are BF16, so there are no q/kv scales;
 * everything else (plan, workspace, status, row order, outputs, merge, error
 * codes) is as for mla_decode.
 *
 * q_bf16          BF16 [batch, q_len, num_heads, 576], contiguous, 16-byte aligned.
 * kv_pages_bf16   BF16 [num_pages, 32, 576], contiguous, 16-byte aligned.
 * The workspace size is mla_decode_workspace_size(...) for the same plan.
 */
MLA_API int mla_decode_bf16(const void* q_bf16, const void* kv_pages_bf16, int64_t num_pages,
                            const int32_t* page_table, int32_t max_pages_per_req,
                            const int32_t* kv_lens, const int32_t* splits, const int32_t* chunks,
                            int32_t max_splits, int32_t kv_split, int32_t batch, int32_t q_len,
                            int32_t num_heads, int32_t causal, float softmax_scale,
                            void* workspace, size_t workspace_bytes, void* out_bf16,
                            float* lse_f32, float* out_f32_debug, void* stream);

/* mla_decode_bf16 with options (NULL options = mla_decode_bf16): output_scale,
 * sinks, query_lens, kv_bounds and softmax_scale_dev as for mla_decode_ex;
 * cta_items / num_ctas as for mla_decode_ex with a list built by
 * mla_decode_plan_items_bf16.  q_scale_dev and kv_scale_dev are FP8-only
 * (BF16 Q and KV carry no scale): MLA_ERR_UNSUPPORTED. */
MLA_API int mla_decode_bf16_ex(const void* q_bf16, const void* kv_pages_bf16, int64_t num_pages,
                               const int32_t* page_table, int32_t max_pages_per_req,
                               const int32_t* kv_lens, const int32_t* splits,
                               const int32_t* chunks, int32_t max_splits, int32_t kv_split,
                               int32_t batch, int32_t q_len, int32_t num_heads, int32_t causal,
                               float softmax_scale, void* workspace, size_t workspace_bytes,
                               void* out_bf16, float* lse_f32, float* out_f32_debug,
                               const mla_decode_options_t* options, void* stream);

/* Sparse decode over selected pages with a BF16 cache: mla_decode_sparse's
 * selection (block_idx, topk, the plan over the compact lengths 32 * topk)
 * with mla_decode_bf16's Q, KV and outputs (PR #17441 "m3 decode perf": the
 * sparse MLA decode after the top-k block selector; here on the BF16 cache of
 * issue #20510's mla_decode_fp16.py).  options as for mla_decode_bf16_ex. */
MLA_API int mla_decode_bf16_sparse(const void* q_bf16, const void* kv_pages_bf16,
                                   int64_t num_pages, const int32_t* page_table,
                                   int32_t max_pages_per_req, const int32_t* kv_lens,
                                   const int32_t* block_idx, int32_t topk, const int32_t* splits,
                                   const int32_t* chunks, int32_t max_splits, int32_t kv_split,
                                   int32_t batch, int32_t q_len, int32_t num_heads,
                                   int32_t causal, float softmax_scale, void* workspace,
                                   size_t workspace_bytes, void* out_bf16, float* lse_f32,
                                   float* out_f32_debug, const mla_decode_options_t* options,
                                   void* stream);

/* Zero the 256-byte status header of a new workspace (async on `stream`).
 * Call once per workspace before its first mla_decode; after that the
 * header only changes when the device reports a condition, and
 * mla_decode_status clears it again after reading.  The partial area needs
 * no initialisation. */
MLA_API int mla_decode_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Merge alone (PR #20380, "Description": KvSplit thread groups, a shared-memory
 * combine rescaled by exp2(group max - max), empty groups skipped, padded loads
 * with weight 0).
 *
 * partial_o   fp32 [rows, num_ctas_kv, 512]: un-normalised outputs.
 * partial_ml  fp32 [rows, num_ctas_kv, 2]: (m in log2 units, l).  A slot with
 *             l == 0 (conventionally m = -inf) is empty and is skipped.
 * Result per row: M = max m_s, w_s = 2^(m_s - M),
 *   O = sum w_s O_s / sum w_s l_s (BF16 and optionally fp32),
 *   LSE = ln2 * (M + log2 sum w_s l_s).  A row with no non-empty slot gives
 *   O = 0 and LSE = -inf.
 */
MLA_API int mla_merge(const float* partial_o, const float* partial_ml, int32_t rows, int32_t num_ctas_kv,
              int32_t kv_split, void* out_bf16, float* lse_f32, float* out_f32_debug,
              void* stream);

/*
 * FP8 paged KV append: quantize n_tokens new latent rows and scatter them into
 * the paged cache that mla_decode reads (TensorRT-LLM PR #17273, "Fuse the DSv4
 * MLA prologue": a latent row is quantized to FP8 and scattered into the paged
 * cache; the model-specific RMSNorm and RoPE before it are not part of this
 * library).
 *
 * rows_bf16     BF16 [n_tokens, 576] (512 latent + 64 rope), 16-byte aligned.
 * req_idx       int32 [n_tokens]: request of each row (0 <= b < batch).
 * positions     int32 [n_tokens]: token index of each row within its request;
 *               it lands in slot pos % 32 of page page_table[b][pos / 32].
 * page_table    int32 [batch, max_pages_per_req].
 * kv_pages_fp8  E4M3 [num_pages, 32, 576], 8-byte aligned; written in place.
 * kv_scale      the stored code is e4m3(x / kv_scale): IEEE fp32 division,
 *               nearest E4M3 value with ties to even, magnitudes beyond 448
 *               saturate to 448, NaN stays NaN.
 * status        device int32 or NULL: set to MLA_ERR_INVALID_ARG if some row
 *               had an out-of-range request, position or page id (that row is
 *               skipped); never cleared by the call.
 * Rows with the same (request, position) race; the caller keeps them unique.
 */
MLA_API int mla_kv_append(const void* rows_bf16, int64_t n_tokens, const int32_t* req_idx,
                          const int32_t* positions, const int32_t* page_table,
                          int32_t max_pages_per_req, int32_t batch, void* kv_pages_fp8,
                          int64_t num_pages, float kv_scale, int32_t* status, void* stream);

/* Synchronously reads the status word at the head of `workspace` (MLA_OK,
 * MLA_ERR_INVALID_ARG for a bad page id or inconsistent plan arrays,
 * MLA_ERR_TIMEOUT for a wait that ran out) after `stream` has drained, and
 * clears it. */
MLA_API int mla_decode_status(const void* workspace, void* stream);

/*
 * Decode without a workspace argument, for callers that cannot allocate
 * device memory (a host runtime that owns every allocation and forbids side
 * allocations, or a latency-critical path that cannot afford cudaMalloc's
 * implicit synchronisation).  The pages have no counterpart to this call.
 *
 * Same arguments and results as mla_decode, minus workspace/workspace_bytes.
 * The scratch (status word and split partials) is a fixed, file-scope device
 * array of MLA_STATIC_WS_BYTES bytes inside the library, which every GPU that
 * loads the library holds until the process exits.  A call whose scratch
 * (mla_decode_workspace_size) would exceed it returns
 * MLA_ERR_WORKSPACE_TOO_SMALL.  The call allocates nothing.
 *
 * The first call on a device (and the first after the device's context has
 * been replaced, e.g. by cudaDeviceReset) resolves the array's device address
 * on that device (the current device) and zeroes its status header with a
 * synchronous cudaMemset, so make that first call before any stream capture.
 * All calls share the one array: calls that overlap on the GPU (on different
 * streams, or from different threads) race on it and must be serialised by
 * the caller.  Conditions the device detects (a bad page id, inconsistent
 * plan arrays, a wait that ran out) go to the array's status word, which
 * stays set across calls until mla_decode_static_ws_status reads and clears
 * it; the output of such a call is not valid.
 */
#define MLA_STATIC_WS_BYTES (16u * 1024u * 1024u)
MLA_API int mla_decode_static_ws(const void* q_fp8, const void* kv_pages_fp8, int64_t num_pages,
                                 const int32_t* page_table, int32_t max_pages_per_req,
                                 const int32_t* kv_lens, const int32_t* splits,
                                 const int32_t* chunks, int32_t max_splits, int32_t kv_split,
                                 int32_t batch, int32_t q_len, int32_t num_heads, int32_t causal,
                                 float q_scale, float kv_scale, float softmax_scale,
                                 void* out_bf16, float* lse_f32, float* out_f32_debug,
                                 void* stream);

/* Status of mla_decode_static_ws calls (no counterpart on the pages): waits
 * for `stream` to drain, then reads and clears the status word of the fixed
 * scratch array on the current device, like mla_decode_status does for a
 * caller-owned workspace.  Returns MLA_OK, MLA_ERR_INVALID_ARG (bad page id or
 * inconsistent plan arrays in some call since the last read) or
 * MLA_ERR_TIMEOUT.  Allocates nothing. */
MLA_API int mla_decode_static_ws_status(void* stream);

/* Test hook.  Sets the limit, in SM clock cycles, of the split-KV kernel's
 * pipeline waits for launches made after the call (0 restores the default of
 * about 2 s).  A tiny limit makes those waits run out: the kernel then records
 * MLA_ERR_TIMEOUT in the status word, lets its own copies and MMAs finish
 * (those drains keep the long limit), frees TMEM and exits, leaving the
 * context usable.  Not for production use. */
MLA_API void mla_debug_set_wait_limit(long long cycles);

/* Test hook.  For launches made after the call, the pipeline wait of `role`
 * at tile index `tile` of every split-KV CTA reads as expired without any
 * stall: 0 the producer's wait for a free KV stage, 1 the QK issuer's wait
 * for a landed tile, 2 the PV issuer's wait for P^T, 3 the softmax's wait
 * for S^T, 4 its wait for a free P^T buffer (FP8 configurations of 32 rows
 * or more), 5 its wait for the last MMAs before the epilogue (tile 0).  The
 * kernel then does what a wait that ran out does: records MLA_ERR_TIMEOUT,
 * stops the other roles, lets its own copies and MMAs finish, frees TMEM and
 * exits (the call's output is not valid).  role < 0 turns it off.  Not for
 * production use. */
MLA_API void mla_debug_set_expire(int32_t role, int32_t tile);

/* Message for the last non-OK status returned on this thread. */
MLA_API const char* mla_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MLA_DECODE_H_ */
