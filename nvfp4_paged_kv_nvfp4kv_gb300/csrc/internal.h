// internal.h -- types shared by the host code and the kernels of the library
// (not part of the public ABI; see include/nvfp4kv.h for that).
#pragma once

#include <cstdint>

#include <cuda_runtime_api.h>

namespace nvfp4kv {

constexpr uint32_t kPlanMagic = 0x4E564B50u;  // "NVKP"
constexpr int kPageSize = 16;  // tokens of one tile (one page at page size 16)
constexpr int kBlock = 16;  // elements per E4M3 scale

// One attention work unit: the pages [page_begin, page_begin + num_pages)
// of kv_indices belong to request b; the unit covers its tokens
// [tok_begin, tok_begin + page_size*num_pages) clipped to kv_len, walked in
// tiles of 16 tokens (one page at page size 16, sixteen at page size 1;
// tok_begin is a multiple of 16).  The partial state
// of query row i, head h (of the unit's kv head) lives at
//   partial_base + (i * Hq + h) * num_splits + split      (when split),
// and `pair` numbers the (request, kv head) for the merge counters.
struct alignas(16) WorkUnit {
  int32_t b;
  int32_t h_kv;
  int32_t page_begin;   // absolute index into kv_indices
  int32_t num_pages;
  int32_t tok_begin;    // first token (request-relative) of the unit
  int32_t kv_len;       // L_b
  int32_t qo_begin;     // first query row of request b
  int32_t qo_len;       // n_b
  int32_t split;        // chunk index of this unit within the request
  int32_t num_splits;   // chunks of the request
  int32_t partial_base; // first partial index of request b
  int32_t pair;         // index of (b, h_kv) among the split groups
};
static_assert(sizeof(WorkUnit) == 48, "WorkUnit layout");

struct CacheView {
  const uint8_t* k_data;
  const uint8_t* v_data;
  const uint8_t* k_sf;
  const uint8_t* v_sf;
  int64_t k_sp, k_ss, k_sh;
  int64_t v_sp, v_ss, v_sh;
  int64_t ksf_sp, ksf_ss, ksf_sh;
  int64_t vsf_sp, vsf_ss, vsf_sh;
  int32_t num_pages;
};

struct AttendParams {
  const uint16_t* q;  // bf16 bits
  int64_t q_stride_tok, q_stride_head;
  CacheView cache;
  const int32_t* kv_indices;
  const WorkUnit* units;
  int32_t num_units;    // work units of the launch
  int32_t num_qo_heads, group, causal, split;
  int32_t page_size;    // 16 or 1
  int32_t out_f16;      // output element: 0 bf16, 1 f16
  float qk_scale_log2;  // sm_scale * k_global_scale * log2(e)
  float v_scale;        // v_global_scale
  uint16_t* out;        // bf16 or f16 [rows, Hq, Dv]
  float* lse;           // [rows, Hq] or null
  float* partial_o;     // [num_partials, Dv]
  float* partial_lse;   // [num_partials]
  int* counters;        // [pairs * row_blocks] arrival counters (split)
  uint32_t* flags;
  // when set, request b's current last_page_len (device); the planned page
  // and query counts still hold, kv_len follows it
  const int32_t* live_last_page_len;
  // fused append (null when not fused): bf16 K/V of the step's new tokens,
  // row-aligned with the query rows (row qo_begin + i is position
  // kv_len - qo_len + i), and the writable cache with its global scales
  const uint16_t* new_k;
  const uint16_t* new_v;
  int64_t nk_stride_tok, nk_stride_head, nv_stride_tok, nv_stride_head;
  float k_global_scale, v_global_scale;
  // FP4 query and probabilities (kernel 4): the row maxima (log2 domain) of
  // query row i, head h over split s of its request, at
  //   row_max[((qo_begin + i) * Hq + h) * row_max_splits + s]
  float* row_max;
  int32_t row_max_splits;
};

struct AppendParams {
  uint8_t* k_data;
  uint8_t* v_data;
  uint8_t* k_sf;
  uint8_t* v_sf;
  int64_t k_sp, k_ss, k_sh, v_sp, v_ss, v_sh;
  int64_t ksf_sp, ksf_ss, ksf_sh, vsf_sp, vsf_ss, vsf_sh;
  int32_t num_pages, num_kv_heads, head_dim_qk, head_dim_vo, page_size;
  float k_global_scale, v_global_scale;
  const uint16_t* k;
  const uint16_t* v;
  int64_t k_stride_tok, k_stride_head, v_stride_tok, v_stride_head;
  int32_t nnz, batch;
  const int32_t* batch_idx;
  const int32_t* positions;
  const int32_t* kv_indices;
  const int32_t* kv_indptr;
  const int32_t* last_page_len;
  uint32_t* flags;
};

struct DequantParams {
  const uint8_t* k_data;
  const uint8_t* v_data;
  const uint8_t* k_sf;
  const uint8_t* v_sf;
  int64_t k_sp, k_ss, k_sh, v_sp, v_ss, v_sh;
  int64_t ksf_sp, ksf_ss, ksf_sh, vsf_sp, vsf_ss, vsf_sh;
  int32_t num_pages, num_kv_heads, head_dim_qk, head_dim_vo, page_size;
  float k_global_scale, v_global_scale;
  const int32_t* page_ids;
  int32_t num_ids;
  float* k_out;  // [num_ids, page_size, Hkv, Dk] or null
  float* v_out;  // [num_ids, page_size, Hkv, Dv] or null
  uint32_t* flags;
};

// Kernel families and their launch descriptions (defined in the .cu files).
enum KernelKind { kKernelTensorCore = 1, kKernelCudaCore = 2, kKernelTcgen05 = 3,
                  kKernelFp4QP = 4 };

struct AttendConfig {
  int kind;       // KernelKind
  int dk, dv;
  int rows;       // query rows per CTA (8 or 16; 16, 32 or 64 for tcgen05)
  int warps;
  int smem_bytes;
  int units_per_cta;  // work units one CTA runs (0 or 1: one)
  const void* func;  // kernel entry (for occupancy queries)
};

// Look up the kernel for (kind, dk, dv, rows); false when not instantiated.
bool attend_config(int kind, int dk, int dv, int rows, AttendConfig* cfg);
cudaError_t launch_attend(const AttendConfig& cfg, const AttendParams& p,
                          int grid_x, int grid_y, cudaStream_t stream);
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_dequantize(const DequantParams& p, cudaStream_t stream);
cudaError_t launch_merge(const float* o_partial, const float* lse_partial,
                         const int32_t* merge_indptr, int32_t num_entries,
                         int32_t head_dim_vo, uint16_t* out, float* lse, bool out_f16,
                         cudaStream_t stream);

}  // namespace nvfp4kv
