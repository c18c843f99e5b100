/*
 * nvfp4_oracle.h -- plain, slow, single-threaded float64 CPU oracle for NVFP4
 * paged-KV attention decode/extend.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or execute this code: only the test suite, the smoke check of the
 * build entry point and the CPU-baseline leg of the benchmark use it.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * What it computes, and from where:
 *  - NVFP4 storage (page "Support NVFP4 KV cache decode on SM120", Gemini
 *    changelog for csrc/xqa/mha.h and csrc/xqa/defines.h): K and V are e2m1
 *    values packed two per uint8 ("ElemsPerContainer == 2"), every 16
 *    consecutive head-dim elements of one token carry one FP8-E4M3 scale
 *    (GMemCacheHeadSf), and each tensor has one FP32 global scale
 *    (CodeRabbit review of tests/attention/test_xqa_batch_decode.py: V must
 *    be dequantised with the V global scale, not K's).
 *  - Quantisation recipe (the pages name nvfp4_quantize / to_nvfp4 but give
 *    no formula; the plain reading adopted here): block scale
 *    s = E4M3_RNE_satfinite(amax / (6 g)), element code
 *    c = e2m1_RNE_satfinite(x / (s g)), low nibble = even element.
 *  - Attention (page "fix(attention): correct SM120 NVFP4 qk_correction
 *    layout, row-sum reduction, and lse", description item 3): lse is the
 *    plain natural-log sum-exp of the scaled scores; exact softmax
 *    attention otherwise.
 *  - Split-KV + merge (page "Re-enable split-KV for NVFP4 KV cache in prefill
 *    path", commit gating split-KV for NVFP4, and its follow-up "16-token-
 *    aligned chunk boundaries"): per-chunk (o, lse) states folded by the
 *    log-sum-exp merge.  The pages give no merge formula; the standard one
 *    is written out in orc_merge_states.
 */
#ifndef NVFP4_ORACLE_H
#define NVFP4_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes of the oracle (independent of the library's codes). */
#define ORC_OK 0
#define ORC_BAD_ARGUMENT 1
#define ORC_BAD_INDEX 2

/* ---- scalar formats --------------------------------------------------- */
double orc_e2m1_value(uint8_t code);          /* 4-bit code -> value        */
double orc_e4m3_value(uint8_t byte);          /* 8-bit E4M3 (fn) -> value   */
uint8_t orc_e2m1_encode(double x);            /* RNE, satfinite, keeps sign */
uint8_t orc_e4m3_encode(double x);            /* RNE, satfinite, keeps sign */
double orc_bf16_value(uint16_t bits);         /* bf16 bit pattern -> value  */

/* Quantise one 16-element block with global scale g (> 0).
 * packed[k] = code(x[2k]) | code(x[2k+1]) << 4;  *sf = E4M3 scale byte. */
void orc_quantize_block16(const double x[16], double g, uint8_t packed[8],
                          uint8_t* sf);

/* ---- paged cache ------------------------------------------------------ */
/* Byte strides; the innermost dimension (packed bytes / scale bytes of one
 * (page, slot, head)) is contiguous. */
typedef struct {
  uint8_t* k_data;
  uint8_t* v_data;
  uint8_t* k_sf;
  uint8_t* v_sf;
  int64_t k_stride_page, k_stride_slot, k_stride_head;
  int64_t v_stride_page, v_stride_slot, v_stride_head;
  int64_t k_sf_stride_page, k_sf_stride_slot, k_sf_stride_head;
  int64_t v_sf_stride_page, v_sf_stride_slot, v_sf_stride_head;
  int32_t num_pages, page_size, num_kv_heads, head_dim_qk, head_dim_vo;
  float k_global_scale, v_global_scale;
} orc_cache;

/* Page-table view of a batch (FlashInfer convention): request b owns pages
 * kv_indices[kv_indptr[b] .. kv_indptr[b+1]); its length is
 * (npages - 1) * page_size + last_page_len[b] (0 when it owns no page). */
typedef struct {
  const int32_t* kv_indices;
  const int32_t* kv_indptr;     /* [batch + 1] */
  const int32_t* last_page_len; /* [batch]     */
  int32_t batch;
} orc_page_table;

int64_t orc_kv_len(const orc_page_table* pt, int32_t b, int32_t page_size);

/* Quantise nnz new tokens and store them into their pages.
 * k_bf16 element (t, h, d) is at k_bf16[t*k_stride_tok + h*k_stride_head + d]
 * (strides in elements); same for v.  Token t belongs to request batch_idx[t]
 * at absolute position positions[t]. Returns ORC_BAD_INDEX (and writes
 * nothing more) if a token maps outside its request's pages or the pool. */
int orc_quantize_append(const orc_cache* c, const uint16_t* k_bf16,
                        int64_t k_stride_tok, int64_t k_stride_head,
                        const uint16_t* v_bf16, int64_t v_stride_tok,
                        int64_t v_stride_head, int32_t nnz,
                        const int32_t* batch_idx, const int32_t* positions,
                        const orc_page_table* pt);

/* Dequantise one stored token row: which = 0 for K (head_dim_qk values),
 * 1 for V (head_dim_vo values). */
void orc_dequant_row(const orc_cache* c, int which, int32_t page, int32_t slot,
                     int32_t head, double* out);

/* Exact attention for request b, kv head h_kv: the G = Hq/Hkv query heads
 * h_kv*G .. h_kv*G+G-1 and every query row i of the request.
 *   q      bf16 bits, element (row, head, d) at
 *          q[(qo_indptr[b]+i)*q_stride_tok + head*q_stride_head + d]
 *   out    fp64, element (row, head, d) at out[((row)*Hq + head)*Dv + d]
 *   lse    fp64 natural log, at lse[row*Hq + head]
 * Query row i of request b sits at absolute position L_b - n_b + i; with
 * causal != 0 it sees keys j <= that position, otherwise all L_b keys.
 * chunk_tokens > 0 evaluates the split variant: per chunk of that many
 * tokens, then merged with orc_merge_states (for split-invariance tests).
 * A row that sees no key gets o = 0 and lse = -inf. */
int orc_attention_unit(const orc_cache* c, const orc_page_table* pt,
                       const int32_t* qo_indptr, const uint16_t* q_bf16,
                       int64_t q_stride_tok, int64_t q_stride_head,
                       int32_t num_qo_heads, int32_t causal, double sm_scale,
                       int32_t b, int32_t h_kv, int64_t chunk_tokens,
                       double* out, double* lse);

/* Attention with the query and the probabilities quantised to FP4 (page
 * "fix(attention): correct SM120 NVFP4 qk_correction layout, row-sum
 * reduction, and lse", description: the SM120 NVFP4 attention it fixes, a
 * SageAttention3 port, quantises Q, K, V and P to FP4; its row sum carries
 * the factor 2^fp8_scalexfp4_scale_log2 of the FP4 P quantisation, which lse
 * drops, and a uniform-score V = ones probe returns the V-quantisation value
 * 1.031).  The pages print no formula; the readings taken here:
 *  - each query row is quantised per 16 dims with E4M3 block scales and
 *    global scale 1 (orc_quantize_block16 with g = 1) and used dequantised;
 *    no block-mean smoothing (one query token per request and head in
 *    decode, whose mean is the row itself);
 *  - p_j = exp(s_j - m), m the row's maximum over all its visible keys (two
 *    passes: an online kernel's running maximum would tie the codes to its
 *    tile order), is scaled by 448 * 6 (the E4M3 maximum times the e2m1
 *    maximum, 2^fp8_scalexfp4_scale_log2) and quantised per 16 consecutive
 *    key positions 16b .. 16b + 15 with global scale 1 (masked keys count 0);
 *  - o = sum_j P_hat_j v_hat_j / (448 * 6 * sum_j p_j): the denominator is the
 *    softmax's own, from the unquantised p; lse = m + ln sum_j p_j.
 * Arguments and output layout as orc_attention_unit (no split variant). */
int orc_attention_unit_fp4qp(const orc_cache* c, const orc_page_table* pt,
                             const int32_t* qo_indptr, const uint16_t* q_bf16,
                             int64_t q_stride_tok, int64_t q_stride_head,
                             int32_t num_qo_heads, int32_t causal,
                             double sm_scale, int32_t b, int32_t h_kv,
                             double* out, double* lse);

/* Fold n partial states (o_i normalised, lse_i natural log) into one:
 * M = max lse_i; lse = M + ln sum exp(lse_i - M); o = sum exp(lse_i - lse) o_i.
 * All lse_i = -inf (or n = 0) gives o = 0, lse = -inf. */
void orc_merge_states(int32_t n, int32_t dim, const double* o_partial,
                      const double* lse_partial, double* o_out,
                      double* lse_out);

#ifdef __cplusplus
}
#endif
#endif
