/*
 * nvfp4kv.h -- C ABI of the NVFP4 paged-KV attention library (GB300, sm_103a).
 *
 * Batched attention decode and short-query extend over a paged KV cache whose
 * K and V are stored as NVFP4: e2m1 values packed two per byte (low nibble =
 * even element), one FP8-E4M3 scale per 16 consecutive head-dim elements of a
 * token, and one FP32 global scale per tensor (page "Support NVFP4 KV cache
 * decode on SM120", Gemini changelog of csrc/xqa/mha.h: GMemCacheHeadSf and
 * the k_sf_cache / v_sf_cache / kv_cache_sf arguments of xqa and
 * xqa_batch_decode_with_kv_cache).
 *
 * Conventions shared by every entry point
 *  - Every function returns an nvfp4kv_status (0 = success).  On failure
 *    nvfp4kv_last_error_detail() returns a message for the calling thread.
 *    Nothing aborts, throws across the ABI, allocates device memory or
 *    synchronises a stream (nvfp4kv_workspace_flags excepted, which reads one
 *    word back).  Argument errors are detected on the host before anything is
 *    enqueued: a call that fails validation launches nothing.
 *  - The caller owns every buffer.  Device buffers (marked [dev]) must stay
 *    allocated until the work enqueued on `stream` has completed; host
 *    buffers (marked [host]) are read during the call, except `plan_host`,
 *    which is also the source of an asynchronous copy (see the plan).
 *  - Cache tensors use BYTE strides; the innermost row (the Dk/2 or Dv/2
 *    packed bytes, the Dk/16 or Dv/16 scale bytes of one (page, slot, head))
 *    is contiguous.  K, V, K-scale and V-scale each have their own stride
 *    triple, so K and V pools with different stride families are supported,
 *    not silently mis-addressed (page "Re-enable split-KV for NVFP4 KV cache
 *    in prefill path", commits on independent K/V strides and on the
 *    support-or-reject contract).  NHD ([page][slot][head][row]) and HND
 *    ([page][head][slot][row]) are both expressible.
 *  - Q strides are in elements; out [rows, Hq, Dv] bf16 and lse [rows, Hq]
 *    float32 are contiguous; the output is sized by head_dim_vo (same page,
 *    commit on the asymmetric-head dispatch and out_head_dim sizing).
 *  - lse is the natural log of the sum of exp of the scaled scores and is
 *    written for every (query row, head) (page "fix(attention): correct
 *    SM120 NVFP4 qk_correction layout, row-sum reduction, and lse", second
 *    commit).
 *  - Page table (FlashInfer convention): request b owns the pages
 *    kv_indices[kv_indptr[b] .. kv_indptr[b+1]) and holds
 *    L_b = (npages_b - 1) * page_size + last_page_len[b] tokens (0 when it
 *    owns no page); qo_indptr gives its n_b = qo_indptr[b+1]-qo_indptr[b]
 *    query rows, which sit at positions L_b - n_b .. L_b - 1 (bottom-right
 *    causal alignment: a new token sees the whole prefix, the earlier new
 *    tokens and itself).
 */
#ifndef NVFP4KV_H
#define NVFP4KV_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status ------------------------------------------------------------ */
typedef enum nvfp4kv_status {
  NVFP4KV_OK = 0,
  NVFP4KV_ERR_INVALID_ARGUMENT = 1,  /* null pointer, bad size/stride/index */
  NVFP4KV_ERR_UNSUPPORTED = 2,       /* valid but not implemented here      */
  NVFP4KV_ERR_WORKSPACE_TOO_SMALL = 3,
  NVFP4KV_ERR_CUDA = 4,              /* a CUDA runtime call failed          */
  NVFP4KV_ERR_DEVICE_CHECK = 5,      /* device flags report a bad index     */
  NVFP4KV_ERR_PLAN_MISMATCH = 6      /* run arguments differ from the plan  */
} nvfp4kv_status;

/* Bits of the device flag word (see nvfp4kv_workspace_flags). */
#define NVFP4KV_FLAG_BAD_PAGE_INDEX 0x1u   /* a kv_indices entry out of pool  */
#define NVFP4KV_FLAG_BAD_APPEND_TARGET 0x2u /* append token outside its request */
#define NVFP4KV_FLAG_COPY_TIMEOUT 0x4u  /* a pipeline wait of the tcgen05 kernel
                                           ran out (a copy or product did not
                                           complete in time); the affected
                                           rows are not valid                */
#define NVFP4KV_FLAG_BAD_LIVE_LENGTH 0x8u /* a live last_page_len was outside
                                           [1, 16] or left fewer tokens than
                                           query rows (clamped)              */
#define NVFP4KV_FLAG_PACE_TIMEOUT 0x10u /* a pacing wait between the units of
                                           a decode CTA ran out; pacing
                                           carries no data, results stand  */

const char* nvfp4kv_status_string(int status);
const char* nvfp4kv_last_error_detail(void);

/* ---- the paged cache ----------------------------------------------------- */
typedef struct nvfp4kv_paged_cache {
  uint8_t* k_data; /* [dev] packed e2m1, Dk/2 bytes per (page, slot, head)   */
  uint8_t* v_data; /* [dev] packed e2m1, Dv/2 bytes per (page, slot, head)   */
  uint8_t* k_sf;   /* [dev] E4M3 bytes, Dk/16 per (page, slot, head)         */
  uint8_t* v_sf;   /* [dev] E4M3 bytes, Dv/16 per (page, slot, head)         */
  int64_t k_stride_page, k_stride_slot, k_stride_head;          /* bytes */
  int64_t v_stride_page, v_stride_slot, v_stride_head;          /* bytes */
  int64_t k_sf_stride_page, k_sf_stride_slot, k_sf_stride_head; /* bytes */
  int64_t v_sf_stride_page, v_sf_stride_slot, v_sf_stride_head; /* bytes */
  int32_t num_pages;   /* pages in the pool                                  */
  int32_t page_size;   /* tokens per page: 16 or 1                           */
  int32_t num_kv_heads;
  int32_t head_dim_qk; /* (Dk, Dv) in {(64,64), (128,128), (256,256),        */
  int32_t head_dim_vo; /*  (256,128), (512,256)}; others: UNSUPPORTED         */
  float k_global_scale; /* dequantised K = e2m1 * E4M3 scale * k_global_scale;
                           in [2^-64, 2^64]                                  */
  float v_global_scale; /* dequantised V uses its own global scale (same range) */
} nvfp4kv_paged_cache;
/* Alignment: data pointers and data strides are multiples of 16 bytes; scale
 * pointers and scale strides are multiples of min(16, D/16) bytes. */

/* ---- quantise-append ----------------------------------------------------- */
/* Quantise nnz new tokens from bf16 and store them into their pages
 * (the in-tree NVFP4 KV quantisation kernel the prefill tests of page
 * "Re-enable split-KV for NVFP4 KV cache in prefill path" feed the cache
 * with; recipe per 16-element block of one token and head: scale byte
 * s = E4M3_RNE_satfinite(amax / (6 g)), codes e2m1_RNE_satfinite(x / (s g))
 * with ties to the even code, zero codes keeping the sign of x, low nibble =
 * even element; every rounding decision is the exact-real one).
 *   k_bf16 [dev]  element (t, h, d) at k_bf16[t*k_stride_tok + h*k_stride_head
 *                 + d]; strides in elements, multiples of 8; 16-byte aligned.
 *   v_bf16 [dev]  same with the V strides, d < head_dim_vo.
 *   batch_idx, positions [dev, nnz]  request and absolute position of token t.
 *   kv_indices, kv_indptr, last_page_len [dev]  page table AFTER the append
 *                 (every position must lie below L_b).
 *   device_flags [dev, optional]  a token whose request, position or page id
 *                 is out of range is skipped and sets
 *                 NVFP4KV_FLAG_BAD_APPEND_TARGET here.
 * Inputs must be finite.  nnz == 0 is a no-op. */
int nvfp4kv_quantize_append(const nvfp4kv_paged_cache* cache,
                            const void* k_bf16, int64_t k_stride_tok,
                            int64_t k_stride_head, const void* v_bf16,
                            int64_t v_stride_tok, int64_t v_stride_head,
                            int32_t nnz, const int32_t* batch_idx,
                            const int32_t* positions, const int32_t* kv_indices,
                            const int32_t* kv_indptr,
                            const int32_t* last_page_len, int32_t batch,
                            uint32_t* device_flags, cudaStream_t stream);

/* ---- plan ---------------------------------------------------------------- */
/* Split-KV (flash-decoding) work plan.  Chunk boundaries are multiples of 16
 * tokens: whole pages at page size 16, sixteen pages at page size 1 (page
 * "Re-enable split-KV for NVFP4 KV cache in prefill path": the commit gating
 * split-KV off for NVFP4 and its follow-up asking for 16-token-aligned
 * chunks; a later commit there notes that scale blocks run along head_dim, so
 * a token-axis split never cuts one; the tests there run page sizes 1 and
 * 16).  The
 * plan sizes the chunk so the attention grid fills the GPU in one wave,
 * reading the SM count and the per-block shared-memory opt-in of the device
 * (same page, commit on the shared-memory probe). */
typedef struct nvfp4kv_plan_options {
  int32_t causal;             /* nonzero: causal (bottom-right) within a row  */
  int32_t disable_split;      /* nonzero: one work unit per (request, head)  */
  int32_t max_splits;         /* >0: at most this many chunks per request    */
  int32_t force_chunk_tokens; /* >0: chunk size in tokens, multiple of 16    */
  int32_t kernel;             /* 0 auto (3 when head dims are 128 and a kv
                                 head has more than 16 query rows, else 1),
                                 1 tensor-core (mma.sync), 2 CUDA-core,
                                 3 tcgen05 (head dims 128 x 128 only),
                                 4 FP4 query and probabilities: the query
                                 quantised to NVFP4 per 16 dims, p = exp(s
                                 - m) against the row's maximum over all its
                                 keys (a first launch computes the maxima),
                                 scaled by 448 * 6 and quantised to NVFP4
                                 per 16 consecutive keys before the PV
                                 product; o divides by that scale times the
                                 unquantised sum of p, lse is the plain
                                 ln-sum-exp (page "fix(attention): correct
                                 SM120 NVFP4 qk_correction layout, row-sum
                                 reduction, and lse", description).  At most
                                 8 query rows per kv head; mma.sync with the
                                 FP4 operands expanded exactly to f16      */
  int32_t num_sms;            /* >0: override the device's SM count          */
  int32_t ctas_per_sm;        /* >0: override the occupancy query            */
  int32_t out_dtype;          /* output element: 0 bf16 (default), 1 f16      */
  /* [dev, may be NULL] live lengths: when set, every run of this plan reads
   * request b's current last_page_len from device_last_page_len[b] when its
   * kernel starts, instead of the planned one.  The plan then stays valid
   * across decode steps for as long as every request keeps its page count
   * (kv_indptr) and its query count; a step that opens a new page needs a
   * new plan.  The array must stay allocated while the plan is used. */
  const int32_t* device_last_page_len;
} nvfp4kv_plan_options;

typedef struct nvfp4kv_plan_info {
  uint32_t magic;
  int32_t batch, num_qo_heads, num_kv_heads, head_dim_qk, head_dim_vo;
  int32_t page_size, causal;
  int32_t kernel;          /* 1 tensor-core, 2 CUDA-core, 3 tcgen05, 4 FP4
                              query and probabilities (two launches)       */
  int32_t num_units;       /* attention work units (grid x)                  */
  int32_t row_blocks;      /* query-row blocks per unit (grid y)             */
  int32_t rows_per_block;  /* query rows (G x qo positions) per CTA          */
  int32_t warps;           /* warps per CTA                                  */
  int32_t split;           /* nonzero: partial states + merge                */
  int32_t chunk_pages;     /* pages per unit (the last one may be shorter)   */
  int32_t max_units_per_request;
  int32_t total_qo_rows;   /* sum of n_b                                     */
  int32_t num_sms, ctas_per_sm, smem_bytes, device;
  int32_t out_dtype;       /* 0 bf16, 1 f16 (the plan option)                */
  int64_t num_partials;    /* partial (o, lse) states when split             */
  int64_t total_kv_pages;  /* pages referenced by the batch                  */
  uint64_t workspace_bytes;  /* device workspace needed                      */
  uint64_t plan_host_bytes;  /* host bytes the plan writes into plan_host    */
  uint64_t off_flags, off_units, off_merge_indptr, off_partial_lse,
      off_partial_o;       /* byte offsets inside the workspace              */
  uint64_t off_counters;   /* merge arrival counters (self-resetting)        */
  const int32_t* device_last_page_len;  /* the plan option, or NULL          */
  uint64_t off_row_max;    /* kernel 4: f32 row maxima [rows][Hq][units per
                              request] written by the first launch (else 0) */
} nvfp4kv_plan_info;

/* Build the plan from HOST copies of the batch description.
 *   qo_indptr_h, kv_indptr_h [host, batch+1], last_page_len_h [host, batch].
 *   opts [host, may be NULL = defaults].
 *   device  CUDA device to plan for (<0: current device; when both num_sms
 *           and ctas_per_sm are given no device is queried at all).
 *   plan_host [host] receives the work list; it must hold
 *           info->plan_host_bytes.  When workspace is non-NULL the plan
 *           enqueues one cudaMemcpyAsync(workspace <- plan_host) and a
 *           cudaMemsetAsync of the flag word on `stream`: keep plan_host
 *           unchanged until that copy completes (use pinned memory to keep
 *           it asynchronous).
 *   workspace [dev, may be NULL]: NULL asks for sizes only (info filled,
 *           nothing enqueued); otherwise it must hold info->workspace_bytes
 *           and be 256-byte aligned.
 * Returns WORKSPACE_TOO_SMALL (with info sizes filled) when plan_host or the
 * workspace is too small. */
int nvfp4kv_decode_plan(const int32_t* qo_indptr_h, const int32_t* kv_indptr_h,
                        const int32_t* last_page_len_h, int32_t batch,
                        int32_t num_qo_heads, int32_t num_kv_heads,
                        int32_t head_dim_qk, int32_t head_dim_vo,
                        int32_t page_size, const nvfp4kv_plan_options* opts,
                        int32_t device, void* plan_host,
                        uint64_t plan_host_bytes, void* workspace,
                        uint64_t workspace_bytes, cudaStream_t stream,
                        nvfp4kv_plan_info* info);

/* ---- run ------------------------------------------------------------------ */
/* The output element is the plan's out_dtype: bf16 (default) or f16; every
 * `out_bf16` argument below points to elements of that type. */
/* Attention for the planned batch: GQA-grouped QK^T, online softmax and PV
 * over the dequantised pages.  When the plan split a request, every work unit
 * stores an f32 partial (o, lse) in the workspace and the last unit of each
 * (request, kv head, row block) to finish folds them by log-sum-exp (the merge
 * of nvfp4kv_merge_states) into out/lse; units find out who is last through
 * counters in the workspace and never wait for one another.  One kernel
 * launch; nothing else is enqueued, so the call can be captured in a CUDA
 * graph.  One workspace must not be used by two runs in flight at once.
 *   q_bf16 [dev]  element (row, head, d) at q[row*q_stride_tok +
 *                 head*q_stride_head + d]; strides in elements, multiples
 *                 of 8; 16-byte aligned.
 *   cache         the paged cache (dims must match the plan).
 *   kv_indices [dev]  the planned page table's page ids.
 *   sm_scale      scale of the scores; <= 0 selects 1/sqrt(head_dim_qk).
 *   workspace [dev]   the workspace the plan was uploaded into.
 *   out_bf16 [dev]    [rows, Hq, Dv]; lse [dev, may be NULL] [rows, Hq].
 * A page id outside the pool is read as page 0 and sets
 * NVFP4KV_FLAG_BAD_PAGE_INDEX in the workspace flag word. */
int nvfp4kv_decode_run(const nvfp4kv_plan_info* info, const void* q_bf16,
                       int64_t q_stride_tok, int64_t q_stride_head,
                       const nvfp4kv_paged_cache* cache,
                       const int32_t* kv_indices, float sm_scale,
                       void* workspace, uint64_t workspace_bytes,
                       void* out_bf16, float* lse, cudaStream_t stream);

/* Same as nvfp4kv_decode_run (kept as the name of the attention half). */
int nvfp4kv_decode_attend(const nvfp4kv_plan_info* info, const void* q_bf16,
                          int64_t q_stride_tok, int64_t q_stride_head,
                          const nvfp4kv_paged_cache* cache,
                          const int32_t* kv_indices, float sm_scale,
                          void* workspace, uint64_t workspace_bytes,
                          void* out_bf16, float* lse, cudaStream_t stream);
/* One decode / extend step in one launch: the step's new tokens are
 * quantised into their pages (the recipe of nvfp4kv_quantize_append) by the
 * attention kernel itself, just before the pages holding them are read, then
 * the attention runs as in nvfp4kv_decode_run.  Request b's new tokens are
 * its last n_b positions L_b - n_b .. L_b - 1, one per query row:
 *   new_k_bf16 [dev]  element (row, h, d) at new_k[row*k_stride_tok +
 *                     h*k_stride_head + d] for query row `row` (the token at
 *                     position L_b - n_b + i for row qo_indptr[b] + i), d < Dk;
 *   new_v_bf16 [dev]  the same with the V strides, d < Dv;
 * strides in elements, multiples of 8, 16-byte aligned.  The page table
 * must already cover the new positions (last_page_len counts them).  The
 * cache is written: afterwards it holds the new tokens exactly as
 * nvfp4kv_quantize_append would have stored them.  Requires a tensor-core
 * kernel (plan option kernel 0, 1 or 3).  A new token whose page id is out of
 * the pool is skipped and sets NVFP4KV_FLAG_BAD_APPEND_TARGET. */
int nvfp4kv_decode_append_run(const nvfp4kv_plan_info* info, const void* new_k_bf16,
                              int64_t k_stride_tok, int64_t k_stride_head,
                              const void* new_v_bf16, int64_t v_stride_tok,
                              int64_t v_stride_head, const void* q_bf16,
                              int64_t q_stride_tok, int64_t q_stride_head,
                              const nvfp4kv_paged_cache* cache,
                              const int32_t* kv_indices, float sm_scale,
                              void* workspace, uint64_t workspace_bytes,
                              void* out_bf16, float* lse, cudaStream_t stream);

/* Re-merge the partial states a split run left in the workspace with the
 * standalone merge kernel (nvfp4kv_merge_states over the plan's merge
 * indptr); rewrites out/lse with the same values.  A no-op without split. */
int nvfp4kv_decode_merge(const nvfp4kv_plan_info* info, void* workspace,
                         uint64_t workspace_bytes, void* out_bf16, float* lse,
                         cudaStream_t stream);

/* ---- dequantise ------------------------------------------------------------ */
/* Paged NVFP4 -> float32 for a list of pages (the cache format of page
 * "Support NVFP4 KV cache decode on SM120"; page "Re-enable split-KV for
 * NVFP4 KV cache in prefill path" checks attention against such a dequantised
 * copy): x_hat = e2m1(code) * E4M3(scale) * global_scale, the exact value
 * rounded to float32 (code * scale is exact; one rounding).
 *   page_ids [dev] int32 [num_ids]: physical page of each entry;
 *   k_out [dev, may be NULL] float32 [num_ids, page_size, num_kv_heads,
 *     head_dim_qk]: element (e, slot, h, d) = K of page page_ids[e], slot,
 *     head h, dim d;
 *   v_out [dev, may be NULL] float32 [num_ids, page_size, num_kv_heads,
 *     head_dim_vo];
 *   device_flags [dev, may be NULL]: NVFP4KV_FLAG_BAD_PAGE_INDEX is or-ed in
 *     for an id outside [0, num_pages); that entry's slots are written as 0.
 * Every slot of a page is converted, including slots past a request's
 * length (they hold whatever the pool held).  Outputs are 16-byte aligned;
 * any cache accepted by nvfp4kv_quantize_append is accepted.  Enqueued on
 * `stream`; nothing is allocated. */
int nvfp4kv_dequantize_paged(const nvfp4kv_paged_cache* cache, const int32_t* page_ids,
                             int32_t num_ids, float* k_out, float* v_out,
                             uint32_t* device_flags, cudaStream_t stream);

/* ---- merge ---------------------------------------------------------------- */
/* Fold partial attention states (the flash-decoding split of page
 * "Re-enable split-KV for NVFP4 KV cache in prefill path"; the pages give no
 * formula, this is the standard one): for entry e with partials
 * i in [merge_indptr[e], merge_indptr[e+1]):
 *   M = max_i lse_i;  lse = M + ln sum_i exp(lse_i - M);
 *   o = sum_i exp(lse_i - lse) * o_i   (o_i already normalised);
 * all lse_i = -inf, or no partial, gives o = 0 and lse = -inf.
 *   o_partial [dev] float32 [num_partials, head_dim_vo];
 *   lse_partial [dev] float32 [num_partials], natural log;
 *   merge_indptr [dev] int32 [num_entries + 1];
 *   out_bf16 [dev] [num_entries, head_dim_vo]; lse [dev, may be NULL]
 *   [num_entries].  head_dim_vo is a multiple of 32, at most 512. */
int nvfp4kv_merge_states(const float* o_partial, const float* lse_partial,
                         const int32_t* merge_indptr, int32_t num_entries,
                         int32_t head_dim_vo, void* out_bf16, float* lse,
                         cudaStream_t stream);

/* ---- allocation-free variant -------------------------------------------- */
/* nvfp4kv_decode_run for callers that cannot allocate device memory where
 * they run attention (device memory fully reserved up front, for example by a
 * KV-cache pool sized to the GPU; a host framework that provides no scratch
 * buffer; a path that must not call cudaMalloc because it synchronises the
 * device).  The pages have no counterpart of it: it exists for deployment.
 * The workspace is a fixed 16 MiB array inside the library, held by every GPU
 * that loads the library until the process exits; the call allocates
 * nothing.  The caller still passes the inputs and the outputs.
 *   info, plan_host [host]  a plan made by nvfp4kv_decode_plan with
 *           workspace = NULL (sizes only); info->workspace_bytes must not
 *           exceed 16 MiB (otherwise WORKSPACE_TOO_SMALL and nothing is
 *           enqueued).  plan_host is the source of an asynchronous copy: keep
 *           it unchanged until the work on `stream` has completed.
 *   the other arguments are those of nvfp4kv_decode_run.
 * Every argument is checked first (as nvfp4kv_decode_run checks them, plus
 * info->device against the current device): a call that fails enqueues
 * nothing and leaves the array as it was.  An accepted call clears the
 * array's flag word and merge counters and copies the plan's work list into
 * it before the attention kernel, all on `stream`.  Outside a stream
 * capture every call looks up the array's device address on the current
 * device; inside a capture the address found by that device's last
 * uncaptured call is used, so make one call before capturing (otherwise
 * INVALID_ARGUMENT).  All calls share the one array: calls whose work
 * overlaps on the GPU (different streams, or different plans in flight at
 * once) race and must be serialised by the caller.  A bad page id sets
 * NVFP4KV_FLAG_BAD_PAGE_INDEX in the array's flag word: read it with
 * nvfp4kv_static_workspace_flags before the next call clears it. */
int nvfp4kv_decode_run_static(const nvfp4kv_plan_info* info, const void* plan_host,
                              const void* q_bf16, int64_t q_stride_tok,
                              int64_t q_stride_head, const nvfp4kv_paged_cache* cache,
                              const int32_t* kv_indices, float sm_scale,
                              void* out_bf16, float* lse, cudaStream_t stream);

/* The device flag word of the static workspace (the flags of the last
 * nvfp4kv_decode_run_static call on the current device), read as
 * nvfp4kv_workspace_flags reads a caller workspace: synchronises `stream`,
 * optionally clears the word, and returns NVFP4KV_ERR_DEVICE_CHECK when a
 * flag is set (*flags is written either way).  info is the plan of that
 * call.  No counterpart on the pages, like the entry point it serves. */
int nvfp4kv_static_workspace_flags(const nvfp4kv_plan_info* info, uint32_t* flags,
                                   int32_t clear, cudaStream_t stream);

/* ---- flags ---------------------------------------------------------------- */
/* Read (and optionally clear) the device flag word of a planned workspace.
 * Synchronises `stream`.  Returns NVFP4KV_ERR_DEVICE_CHECK when a flag is set
 * (the word is still written to *flags). */
int nvfp4kv_workspace_flags(const nvfp4kv_plan_info* info,
                            const void* workspace, uint32_t* flags,
                            int32_t clear, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4KV_H */
