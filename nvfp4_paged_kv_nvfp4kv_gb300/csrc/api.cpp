// api.cpp -- host side of the C ABI declared in include/nvfp4kv.h:
// argument validation, the split-KV planner and kernel dispatch.
#include "nvfp4kv.h"

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include <cuda_runtime_api.h>

#include "internal.h"

namespace nvfp4kv {
bool attend_config_tc(int dk, int dv, int rows, AttendConfig* cfg);
bool attend_config_simt(int dk, int dv, int rows, AttendConfig* cfg);
bool attend_config_tcgen05(int dk, int dv, int rows, AttendConfig* cfg);
bool attend_config_dec(int dk, int dv, int rows, int quads, AttendConfig* cfg);
bool attend_config_tc_fp4qp(int dk, int dv, int rows, int pass, AttendConfig* cfg);
cudaError_t prepare_kernel(const AttendConfig& cfg);
}  // namespace nvfp4kv

using namespace nvfp4kv;

namespace {
int fail(int status, const char* fmt, ...);
}

namespace nvfp4kv {
// Record a message for nvfp4kv_last_error_detail() and return `status`.
int set_error_detail(int status, const char* message) { return fail(status, "%s", message); }
}  // namespace nvfp4kv

namespace {

thread_local std::string g_detail;

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_detail = buf;
  return status;
}

int ok() {
  g_detail.clear();
  return NVFP4KV_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(NVFP4KV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, uint64_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

bool attention_dims_supported(int dk, int dv) {
  return (dk == 64 && dv == 64) || (dk == 128 && dv == 128) ||
         (dk == 256 && dv == 256) || (dk == 256 && dv == 128) ||
         (dk == 512 && dv == 256);
}

// Common cache checks.  `for_attention` adds the head-dim whitelist and the
// cp.async alignment rules.
int check_cache(const nvfp4kv_paged_cache* c, bool for_attention) {
  if (!c) return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "cache is null");
  if (!c->k_data || !c->v_data || !c->k_sf || !c->v_sf)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "cache buffer pointer is null");
  if (c->page_size != kPageSize && c->page_size != 1)
    return fail(NVFP4KV_ERR_UNSUPPORTED, "page_size %d (16 and 1 are supported)", c->page_size);
  if (c->num_pages <= 0 || c->num_kv_heads <= 0)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "num_pages %d / num_kv_heads %d must be > 0",
                c->num_pages, c->num_kv_heads);
  if (c->head_dim_qk <= 0 || c->head_dim_vo <= 0 || c->head_dim_qk % 32 ||
      c->head_dim_vo % 32 || c->head_dim_qk > 512 || c->head_dim_vo > 512)
    return fail(NVFP4KV_ERR_UNSUPPORTED,
                "head dims (%d, %d): each must be a multiple of 32 and at most 512",
                c->head_dim_qk, c->head_dim_vo);
  if (for_attention && !attention_dims_supported(c->head_dim_qk, c->head_dim_vo))
    return fail(NVFP4KV_ERR_UNSUPPORTED,
                "attention head dims (%d, %d) not built; supported: (64,64), "
                "(128,128), (256,256), (256,128), (512,256)",
                c->head_dim_qk, c->head_dim_vo);
  const float gmin = std::ldexp(1.0f, -64), gmax = std::ldexp(1.0f, 64);
  if (!(c->k_global_scale >= gmin && c->k_global_scale <= gmax) ||
      !(c->v_global_scale >= gmin && c->v_global_scale <= gmax))
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "global scales must lie in [2^-64, 2^64]");
  const int64_t kd[3] = {c->k_stride_page, c->k_stride_slot, c->k_stride_head};
  const int64_t vd[3] = {c->v_stride_page, c->v_stride_slot, c->v_stride_head};
  const int64_t ks[3] = {c->k_sf_stride_page, c->k_sf_stride_slot, c->k_sf_stride_head};
  const int64_t vs[3] = {c->v_sf_stride_page, c->v_sf_stride_slot, c->v_sf_stride_head};
  const int64_t ksa = std::min(16, c->head_dim_qk / 16), vsa = std::min(16, c->head_dim_vo / 16);
  for (int i = 0; i < 3; ++i) {
    if (kd[i] < 0 || vd[i] < 0 || ks[i] < 0 || vs[i] < 0)
      return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "negative cache stride");
    if (kd[i] % 16 || vd[i] % 16)
      return fail(NVFP4KV_ERR_INVALID_ARGUMENT,
                  "K/V data strides must be multiples of 16 bytes");
    if (ks[i] % ksa || vs[i] % vsa)
      return fail(NVFP4KV_ERR_INVALID_ARGUMENT,
                  "scale strides must be multiples of min(16, D/16) bytes");
  }
  if (!aligned(c->k_data, 16) || !aligned(c->v_data, 16) || !aligned(c->k_sf, ksa) ||
      !aligned(c->v_sf, vsa))
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "cache buffer misaligned");
  // the innermost row must not overlap the next slot/head (rows are contiguous)
  if (std::min(c->k_stride_slot, c->k_stride_head) < c->head_dim_qk / 2 ||
      std::min(c->v_stride_slot, c->v_stride_head) < c->head_dim_vo / 2 ||
      std::min(c->k_sf_stride_slot, c->k_sf_stride_head) < c->head_dim_qk / 16 ||
      std::min(c->v_sf_stride_slot, c->v_sf_stride_head) < c->head_dim_vo / 16)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "cache strides overlap a row");
  return NVFP4KV_OK;
}

CacheView view_of(const nvfp4kv_paged_cache* c) {
  CacheView v;
  v.k_data = c->k_data;
  v.v_data = c->v_data;
  v.k_sf = c->k_sf;
  v.v_sf = c->v_sf;
  v.k_sp = c->k_stride_page; v.k_ss = c->k_stride_slot; v.k_sh = c->k_stride_head;
  v.v_sp = c->v_stride_page; v.v_ss = c->v_stride_slot; v.v_sh = c->v_stride_head;
  v.ksf_sp = c->k_sf_stride_page; v.ksf_ss = c->k_sf_stride_slot; v.ksf_sh = c->k_sf_stride_head;
  v.vsf_sp = c->v_sf_stride_page; v.vsf_ss = c->v_sf_stride_slot; v.vsf_sh = c->v_sf_stride_head;
  v.num_pages = c->num_pages;
  return v;
}

bool lookup_kernel(int kind, int dk, int dv, int rows, AttendConfig* cfg) {
  if (kind == kKernelTensorCore) return attend_config_tc(dk, dv, rows, cfg);
  if (kind == kKernelCudaCore) return attend_config_simt(dk, dv, rows, cfg);
  if (kind == kKernelTcgen05) return attend_config_tcgen05(dk, dv, rows, cfg);
  if (kind == kKernelFp4QP) return attend_config_tc_fp4qp(dk, dv, rows, 2, cfg);
  return false;
}

constexpr int kMinChunkPages = 8;

// The bulk-copy decode kernel reads each (page, head) region of the four
// buffers with one copy: the 16 slots' rows must be contiguous, every region
// must start 16-byte aligned, and a page offset must fit 32 bits.
bool bulk_decode_layout(const nvfp4kv_paged_cache* c) {
  const int64_t kr = c->head_dim_qk / 2, vr = c->head_dim_vo / 2;
  const int64_t ksr = c->head_dim_qk / 16, vsr = c->head_dim_vo / 16;
  const int64_t lim = (int64_t)1 << 32;
  return c->k_stride_slot == kr && c->v_stride_slot == vr && c->k_sf_stride_slot == ksr &&
         c->v_sf_stride_slot == vsr && aligned(c->k_sf, 16) && aligned(c->v_sf, 16) &&
         c->k_sf_stride_page % 16 == 0 && c->k_sf_stride_head % 16 == 0 &&
         c->v_sf_stride_page % 16 == 0 && c->v_sf_stride_head % 16 == 0 &&
         c->k_stride_page < lim && c->v_stride_page < lim && c->k_sf_stride_page < lim &&
         c->v_sf_stride_page < lim;
}

}  // namespace

extern "C" {

const char* nvfp4kv_status_string(int status) {
  switch (status) {
    case NVFP4KV_OK: return "ok";
    case NVFP4KV_ERR_INVALID_ARGUMENT: return "invalid argument";
    case NVFP4KV_ERR_UNSUPPORTED: return "unsupported";
    case NVFP4KV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case NVFP4KV_ERR_CUDA: return "CUDA error";
    case NVFP4KV_ERR_DEVICE_CHECK: return "device check failed";
    case NVFP4KV_ERR_PLAN_MISMATCH: return "arguments do not match the plan";
    default: return "unknown status";
  }
}

const char* nvfp4kv_last_error_detail(void) { return g_detail.c_str(); }

int nvfp4kv_dequantize_paged(const nvfp4kv_paged_cache* cache, const int32_t* page_ids,
                             int32_t num_ids, float* k_out, float* v_out,
                             uint32_t* device_flags, cudaStream_t stream) {
  if (int st = check_cache(cache, false)) return st;
  if (num_ids < 0) return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "num_ids %d negative", num_ids);
  if (num_ids == 0 || (!k_out && !v_out)) return ok();
  if (!page_ids) return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "page_ids is null");
  if ((k_out && !aligned(k_out, 16)) || (v_out && !aligned(v_out, 16)))
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "outputs must be 16-byte aligned");
  DequantParams p{};
  p.k_data = cache->k_data; p.v_data = cache->v_data;
  p.k_sf = cache->k_sf; p.v_sf = cache->v_sf;
  p.k_sp = cache->k_stride_page; p.k_ss = cache->k_stride_slot; p.k_sh = cache->k_stride_head;
  p.v_sp = cache->v_stride_page; p.v_ss = cache->v_stride_slot; p.v_sh = cache->v_stride_head;
  p.ksf_sp = cache->k_sf_stride_page; p.ksf_ss = cache->k_sf_stride_slot;
  p.ksf_sh = cache->k_sf_stride_head;
  p.vsf_sp = cache->v_sf_stride_page; p.vsf_ss = cache->v_sf_stride_slot;
  p.vsf_sh = cache->v_sf_stride_head;
  p.num_pages = cache->num_pages;
  p.num_kv_heads = cache->num_kv_heads;
  p.head_dim_qk = cache->head_dim_qk;
  p.head_dim_vo = cache->head_dim_vo;
  p.page_size = cache->page_size;
  p.k_global_scale = cache->k_global_scale;
  p.v_global_scale = cache->v_global_scale;
  p.page_ids = page_ids;
  p.num_ids = num_ids;
  p.k_out = k_out;
  p.v_out = v_out;
  p.flags = device_flags;
  cudaError_t e = launch_dequantize(p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dequantize launch");
  return ok();
}

int nvfp4kv_quantize_append(const nvfp4kv_paged_cache* cache, const void* k_bf16,
                            int64_t k_stride_tok, int64_t k_stride_head,
                            const void* v_bf16, int64_t v_stride_tok,
                            int64_t v_stride_head, int32_t nnz,
                            const int32_t* batch_idx, const int32_t* positions,
                            const int32_t* kv_indices, const int32_t* kv_indptr,
                            const int32_t* last_page_len, int32_t batch,
                            uint32_t* device_flags, cudaStream_t stream) {
  if (int st = check_cache(cache, false)) return st;
  if (nnz < 0 || batch < 0)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "nnz %d / batch %d negative", nnz, batch);
  if (nnz == 0) return ok();
  if (!k_bf16 || !v_bf16 || !batch_idx || !positions || !kv_indices || !kv_indptr ||
      !last_page_len)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "null input pointer");
  if (!aligned(k_bf16, 16) || !aligned(v_bf16, 16) || k_stride_tok % 8 ||
      k_stride_head % 8 || v_stride_tok % 8 || v_stride_head % 8 || k_stride_tok < 0 ||
      k_stride_head < 0 || v_stride_tok < 0 || v_stride_head < 0)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT,
                "bf16 inputs must be 16-byte aligned with strides multiple of 8 elements");
  AppendParams p{};
  p.k_data = cache->k_data; p.v_data = cache->v_data;
  p.k_sf = cache->k_sf; p.v_sf = cache->v_sf;
  p.k_sp = cache->k_stride_page; p.k_ss = cache->k_stride_slot; p.k_sh = cache->k_stride_head;
  p.v_sp = cache->v_stride_page; p.v_ss = cache->v_stride_slot; p.v_sh = cache->v_stride_head;
  p.ksf_sp = cache->k_sf_stride_page; p.ksf_ss = cache->k_sf_stride_slot;
  p.ksf_sh = cache->k_sf_stride_head;
  p.vsf_sp = cache->v_sf_stride_page; p.vsf_ss = cache->v_sf_stride_slot;
  p.vsf_sh = cache->v_sf_stride_head;
  p.num_pages = cache->num_pages;
  p.num_kv_heads = cache->num_kv_heads;
  p.head_dim_qk = cache->head_dim_qk;
  p.head_dim_vo = cache->head_dim_vo;
  p.page_size = cache->page_size;
  p.k_global_scale = cache->k_global_scale;
  p.v_global_scale = cache->v_global_scale;
  p.k = static_cast<const uint16_t*>(k_bf16);
  p.v = static_cast<const uint16_t*>(v_bf16);
  p.k_stride_tok = k_stride_tok; p.k_stride_head = k_stride_head;
  p.v_stride_tok = v_stride_tok; p.v_stride_head = v_stride_head;
  p.nnz = nnz;
  p.batch = batch;
  p.batch_idx = batch_idx;
  p.positions = positions;
  p.kv_indices = kv_indices;
  p.kv_indptr = kv_indptr;
  p.last_page_len = last_page_len;
  p.flags = device_flags;
  cudaError_t e = launch_append(p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "quantize_append launch");
  return ok();
}

int nvfp4kv_decode_plan(const int32_t* qo_indptr_h, const int32_t* kv_indptr_h,
                        const int32_t* last_page_len_h, int32_t batch,
                        int32_t num_qo_heads, int32_t num_kv_heads,
                        int32_t head_dim_qk, int32_t head_dim_vo, int32_t page_size,
                        const nvfp4kv_plan_options* opts_in, int32_t device,
                        void* plan_host, uint64_t plan_host_bytes, void* workspace,
                        uint64_t workspace_bytes, cudaStream_t stream,
                        nvfp4kv_plan_info* info) {
  if (!info) return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "info is null");
  std::memset(info, 0, sizeof *info);
  nvfp4kv_plan_options opts{};
  if (opts_in) opts = *opts_in;
  if (batch < 0) return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "batch %d < 0", batch);
  if (batch > 0 && (!qo_indptr_h || !kv_indptr_h || !last_page_len_h))
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "null indptr / last_page_len");
  if (num_qo_heads <= 0 || num_kv_heads <= 0 || num_qo_heads % num_kv_heads)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT,
                "num_qo_heads %d must be a positive multiple of num_kv_heads %d",
                num_qo_heads, num_kv_heads);
  if (page_size != kPageSize && page_size != 1)
    return fail(NVFP4KV_ERR_UNSUPPORTED, "page_size %d (16 and 1 are supported)", page_size);
  if (opts.out_dtype != 0 && opts.out_dtype != 1)
    return fail(NVFP4KV_ERR_UNSUPPORTED, "out_dtype %d (0 bf16, 1 f16)", opts.out_dtype);
  if (!attention_dims_supported(head_dim_qk, head_dim_vo))
    return fail(NVFP4KV_ERR_UNSUPPORTED, "attention head dims (%d, %d) not built",
                head_dim_qk, head_dim_vo);
  if (opts.force_chunk_tokens < 0 || opts.force_chunk_tokens % kPageSize)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT,
                "force_chunk_tokens %d must be a non-negative multiple of 16",
                opts.force_chunk_tokens);
  if (opts.max_splits < 0 || opts.num_sms < 0 || opts.ctas_per_sm < 0 || opts.kernel < 0 ||
      opts.kernel > 4)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "bad plan option");
  const int G = num_qo_heads / num_kv_heads;

  // ---- batch description ------------------------------------------------
  if (batch > 0 && qo_indptr_h[0] != 0)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "qo_indptr[0] must be 0");
  // the planner counts 16-token tiles: one page at page size 16, PT pages
  // at page size 1
  const int PT = kPageSize / page_size;
  std::vector<int32_t> np(batch), nq(batch), nt(batch);
  int64_t total_pages = 0;
  int max_rows = 0, max_np = 0;
  for (int b = 0; b < batch; ++b) {
    nq[b] = qo_indptr_h[b + 1] - qo_indptr_h[b];
    np[b] = kv_indptr_h[b + 1] - kv_indptr_h[b];
    if (nq[b] < 0 || np[b] < 0)
      return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "indptr decreases at request %d", b);
    if (kv_indptr_h[b] < 0)
      return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "kv_indptr[%d] < 0", b);
    int64_t L = 0;
    if (np[b] > 0) {
      if (last_page_len_h[b] < 1 || last_page_len_h[b] > page_size)
        return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "last_page_len[%d] = %d not in [1, %d]", b,
                    last_page_len_h[b], page_size);
      L = static_cast<int64_t>(np[b] - 1) * page_size + last_page_len_h[b];
    }
    nt[b] = (np[b] + PT - 1) / PT;
    if (L < nq[b])
      return fail(NVFP4KV_ERR_INVALID_ARGUMENT,
                  "request %d has %d query rows but only %lld kv tokens", b, nq[b],
                  static_cast<long long>(L));
    if (L > (int64_t)1 << 30)
      return fail(NVFP4KV_ERR_UNSUPPORTED, "request %d longer than 2^30 tokens", b);
    if (nq[b] > 0) {
      total_pages += np[b];
      max_np = std::max(max_np, nt[b]);  // in tiles from here on
      max_rows = std::max(max_rows, nq[b] * G);
    }
  }
  const int32_t total_rows = batch > 0 ? qo_indptr_h[batch] : 0;

  // ---- kernel choice and occupancy --------------------------------------
  int kind = opts.kernel;
  AttendConfig cfg{};
  // auto: the tcgen05 kernel where a kv head has many query rows (extend):
  // it dequantises each page once for all of them and its products grow
  // with the rows; for a few rows (decode) the mma.sync register path is
  // cheaper (a tcgen05 product costs ~54 cycles to issue whatever its N)
  if (kind == 0)
    kind = (head_dim_qk == 128 && head_dim_vo == 128 && max_rows > 16) ? kKernelTcgen05
                                                                       : kKernelTensorCore;
  const int want_rows = kind == kKernelTcgen05 ? std::max(max_rows, 1) : (max_rows <= 8 ? 8 : 16);
  if (!lookup_kernel(kind, head_dim_qk, head_dim_vo, want_rows, &cfg))
    return fail(NVFP4KV_ERR_UNSUPPORTED, "no %s kernel for head dims (%d, %d)%s",
                kind == kKernelTensorCore ? "tensor-core"
                : kind == kKernelTcgen05  ? "tcgen05"
                : kind == kKernelFp4QP    ? "FP4 query/probability"
                                          : "CUDA-core",
                head_dim_qk, head_dim_vo,
                kind == kKernelFp4QP && want_rows > 8 ? " and more than 8 query rows per kv head"
                                                      : "");
  const int rows_per_block = cfg.rows;
  // A tensor-core plan of one block of <= 8 rows at page size 16 runs the
  // decode kernel where the cache layout allows it; that kernel takes several
  // units per CTA, so its occupancy (in units) sizes the wave.
  AttendConfig occ = cfg;
  int units_per_cta = 1;
  {
    AttendConfig dcfg{};
    if (kind == kKernelTensorCore && rows_per_block == 8 && page_size == kPageSize &&
        attend_config_dec(head_dim_qk, head_dim_vo, 8, 4, &dcfg)) {
      occ = dcfg;
      units_per_cta = std::max(1, dcfg.units_per_cta);
    }
  }
  int num_sms = opts.num_sms, ctas_per_sm = opts.ctas_per_sm;
  if (num_sms == 0 || ctas_per_sm == 0) {
    int dev = device;
    cudaError_t e = cudaSuccess;
    if (dev < 0) e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    // the device's SM count and the kernel's resident CTAs per SM do not
    // change: query them once per (device, kernel) and keep them (a plan is
    // built every serving step)
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, std::pair<int, int>> known;
    std::pair<int, int> sm_occ{0, 0};
    {
      std::lock_guard<std::mutex> lock(mu);
      auto it = known.find({dev, occ.func});
      if (it != known.end()) sm_occ = it->second;
    }
    if (sm_occ.first == 0) {
      e = cudaDeviceGetAttribute(&sm_occ.first, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return cuda_fail(e, "SM count");
      int optin = 0;
      e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
      if (e != cudaSuccess) return cuda_fail(e, "shared-memory opt-in");
      if (occ.smem_bytes > optin)
        return fail(NVFP4KV_ERR_UNSUPPORTED,
                    "kernel needs %d bytes of shared memory, device allows %d per block",
                    occ.smem_bytes, optin);
      int cur = -1;
      e = cudaGetDevice(&cur);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
      if (cur != dev && (e = cudaSetDevice(dev)) != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
      e = prepare_kernel(occ);
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&sm_occ.second, occ.func,
                                                          occ.warps * 32, occ.smem_bytes);
      if (cur != dev) cudaSetDevice(cur);
      if (e != cudaSuccess) return cuda_fail(e, "occupancy");
      if (sm_occ.second < 1) sm_occ.second = 1;
      sm_occ.second *= units_per_cta;  // unit slots per SM
      std::lock_guard<std::mutex> lock(mu);
      known[{dev, occ.func}] = sm_occ;
    }
    if (num_sms == 0) num_sms = sm_occ.first;
    if (ctas_per_sm == 0) ctas_per_sm = sm_occ.second;
    info->device = dev;
  } else {
    info->device = device;
  }

  // ---- chunk size (tiles per unit) --------------------------------------
  auto row_blocks_of = [&](int b) { return (nq[b] * G + rows_per_block - 1) / rows_per_block; };
  auto ctas_for = [&](int64_t c) {
    int64_t n = 0;
    for (int b = 0; b < batch; ++b)
      if (nq[b] > 0) n += (int64_t)num_kv_heads * ((nt[b] + c - 1) / c) * row_blocks_of(b);
    return n;
  };
  int64_t chunk = std::max(max_np, 1);
  if (!opts.disable_split) {
    if (opts.force_chunk_tokens > 0) {
      chunk = opts.force_chunk_tokens / kPageSize;
    } else if (max_np > kMinChunkPages) {
      const int64_t slots = (int64_t)num_sms * ctas_per_sm;
      int64_t work = 0;
      for (int b = 0; b < batch; ++b)
        if (nq[b] > 0) work += (int64_t)num_kv_heads * nt[b] * row_blocks_of(b);
      int64_t lo = std::max<int64_t>(kMinChunkPages, (work + slots - 1) / std::max<int64_t>(slots, 1));
      int64_t hi = max_np;
      if (lo >= hi || ctas_for(hi) > slots) {
        chunk = hi;  // already one unit per request suffices / cannot fit one wave
      } else {
        while (lo < hi) {  // smallest chunk whose grid fits one wave
          const int64_t mid = (lo + hi) / 2;
          if (ctas_for(mid) <= slots) hi = mid; else lo = mid + 1;
        }
        chunk = lo;
      }
    }
    if (opts.max_splits > 0)
      chunk = std::max<int64_t>(chunk, (max_np + opts.max_splits - 1) / opts.max_splits);
    // the tcgen05 kernel streams tiles of 8 pages: whole tiles per unit
    if (kind == kKernelTcgen05 && opts.force_chunk_tokens == 0 && chunk < max_np)
      chunk = std::min<int64_t>((chunk + 7) / 8 * 8, max_np);
  }
  chunk = std::max<int64_t>(chunk, 1);

  // ---- units, partial bases, merge indptr -------------------------------
  std::vector<WorkUnit> units;
  int32_t max_units = 0;
  bool split = false;
  int64_t n_units = 0;
  for (int b = 0; b < batch; ++b)
    if (nq[b] > 0) {
      if (nt[b] > chunk) split = true;
      n_units += (int64_t)num_kv_heads * ((nt[b] + chunk - 1) / chunk);
    }
  units.reserve(static_cast<size_t>(n_units));
  int64_t partial = 0;
  std::vector<int64_t> pbase(batch, 0);
  std::vector<int32_t> nsplit(batch, 0);
  for (int b = 0; b < batch; ++b) {
    if (nq[b] == 0) continue;
    const int S = static_cast<int>((nt[b] + chunk - 1) / chunk);
    nsplit[b] = S;
    max_units = std::max(max_units, S);
    pbase[b] = partial;
    if (split) partial += (int64_t)nq[b] * num_qo_heads * S;
    const int64_t L = static_cast<int64_t>(np[b] - 1) * page_size + last_page_len_h[b];
    const int64_t cp = chunk * PT;  // pages per unit
    for (int h = 0; h < num_kv_heads; ++h)
      for (int s = 0; s < S; ++s) {
        WorkUnit u{};
        u.b = b;
        u.h_kv = h;
        u.page_begin = kv_indptr_h[b] + static_cast<int32_t>(s * cp);
        u.num_pages = static_cast<int32_t>(std::min<int64_t>(cp, np[b] - s * cp));
        u.tok_begin = static_cast<int32_t>(s * chunk * kPageSize);
        u.kv_len = static_cast<int32_t>(L);
        u.qo_begin = qo_indptr_h[b];
        u.qo_len = nq[b];
        u.split = s;
        u.num_splits = S;
        u.partial_base = static_cast<int32_t>(pbase[b]);
        u.pair = b * num_kv_heads + h;
        units.push_back(u);
      }
  }
  // Longest units first when the grid takes more than one wave: the block
  // scheduler then starts the long units early (longest-processing-time
  // order); partial indices do not depend on the unit order.  A grid of one
  // wave starts every unit at once, and its order is left as built.
  int row_blocks = 0;
  for (int b = 0; b < batch; ++b)
    if (nq[b] > 0) row_blocks = std::max(row_blocks, row_blocks_of(b));
  if ((int64_t)units.size() * row_blocks > (int64_t)num_sms * ctas_per_sm)
    std::stable_sort(units.begin(), units.end(), [](const WorkUnit& a, const WorkUnit& b) {
      return a.num_pages > b.num_pages;
    });
  if (partial > INT32_MAX)
    return fail(NVFP4KV_ERR_UNSUPPORTED, "too many partial states (%lld)", (long long)partial);
  const int64_t entries = split ? (int64_t)total_rows * num_qo_heads : 0;

  // ---- layout ------------------------------------------------------------
  const uint64_t off_flags = 0;
  const uint64_t off_counters = 256;
  const uint64_t n_counters = split ? (uint64_t)batch * num_kv_heads * row_blocks : 0;
  const uint64_t off_units = align_up(off_counters + n_counters * 4, 256);
  const uint64_t off_merge = align_up(off_units + units.size() * sizeof(WorkUnit), 256);
  const uint64_t off_plse = align_up(off_merge + (split ? (entries + 1) * 4 : 0), 256);
  const uint64_t off_po = align_up(off_plse + partial * 4, 256);
  const uint64_t off_rm = align_up(off_po + (uint64_t)partial * head_dim_vo * 4, 256);
  const uint64_t n_row_max = kind == kKernelFp4QP
                                 ? (uint64_t)total_rows * num_qo_heads * std::max(max_units, 1)
                                 : 0;
  const uint64_t ws_bytes = align_up(off_rm + n_row_max * 4, 256);
  const uint64_t host_bytes = off_plse - off_units;

  info->magic = kPlanMagic;
  info->batch = batch;
  info->num_qo_heads = num_qo_heads;
  info->num_kv_heads = num_kv_heads;
  info->head_dim_qk = head_dim_qk;
  info->head_dim_vo = head_dim_vo;
  info->page_size = page_size;
  info->causal = opts.causal ? 1 : 0;
  info->kernel = kind;
  info->num_units = static_cast<int32_t>(units.size());
  info->row_blocks = row_blocks;
  info->rows_per_block = rows_per_block;
  info->warps = cfg.warps;
  info->split = split ? 1 : 0;
  info->chunk_pages = static_cast<int32_t>(std::min<int64_t>(chunk, INT32_MAX));
  info->max_units_per_request = max_units;
  info->total_qo_rows = total_rows;
  info->num_sms = num_sms;
  info->ctas_per_sm = ctas_per_sm;
  info->out_dtype = opts.out_dtype;
  info->smem_bytes = cfg.smem_bytes;
  info->num_partials = partial;
  info->total_kv_pages = total_pages;
  info->workspace_bytes = ws_bytes;
  info->plan_host_bytes = host_bytes;
  info->off_flags = off_flags;
  info->off_units = off_units;
  info->off_merge_indptr = off_merge;
  info->off_partial_lse = off_plse;
  info->off_partial_o = off_po;
  info->off_counters = off_counters;
  info->off_row_max = n_row_max ? off_rm : 0;
  info->device_last_page_len = opts.device_last_page_len;

  if (host_bytes > 0 && (!plan_host || plan_host_bytes < host_bytes))
    return fail(NVFP4KV_ERR_WORKSPACE_TOO_SMALL, "plan_host needs %llu bytes",
                (unsigned long long)host_bytes);
  uint8_t* hb = static_cast<uint8_t*>(plan_host);
  if (host_bytes > 0) std::memset(hb, 0, host_bytes);
  if (!units.empty()) std::memcpy(hb, units.data(), units.size() * sizeof(WorkUnit));
  if (split) {
    int32_t* mi = reinterpret_cast<int32_t*>(hb + (off_merge - off_units));
    for (int b = 0; b < batch; ++b)
      for (int i = 0; i < nq[b]; ++i)
        for (int h = 0; h < num_qo_heads; ++h) {
          const int64_t e = (int64_t)(qo_indptr_h[b] + i) * num_qo_heads + h;
          mi[e] = static_cast<int32_t>(pbase[b] + ((int64_t)i * num_qo_heads + h) * nsplit[b]);
        }
    mi[entries] = static_cast<int32_t>(partial);
  }
  if (!workspace) return ok();
  if (workspace_bytes < ws_bytes)
    return fail(NVFP4KV_ERR_WORKSPACE_TOO_SMALL, "workspace needs %llu bytes",
                (unsigned long long)ws_bytes);
  if (!aligned(workspace, 256))
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaSuccess;
  if (host_bytes > 0)
    e = cudaMemcpyAsync(ws + off_units, hb, host_bytes, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return cuda_fail(e, "plan upload");
  e = cudaMemsetAsync(ws + off_flags, 0, off_units - off_flags, stream);  // flags, counters
  if (e != cudaSuccess) return cuda_fail(e, "flag reset");
  return ok();
}

}  // extern "C"

namespace {

int check_run(const nvfp4kv_plan_info* info, const void* q, int64_t qst, int64_t qsh,
              const nvfp4kv_paged_cache* cache, const int32_t* kv_indices,
              const void* workspace, uint64_t workspace_bytes, const void* out) {
  if (!info || info->magic != kPlanMagic)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "info is not a plan");
  if (int st = check_cache(cache, true)) return st;
  if (cache->num_kv_heads != info->num_kv_heads || cache->head_dim_qk != info->head_dim_qk ||
      cache->head_dim_vo != info->head_dim_vo || cache->page_size != info->page_size)
    return fail(NVFP4KV_ERR_PLAN_MISMATCH, "cache dims differ from the plan");
  if (!workspace || workspace_bytes < info->workspace_bytes || !aligned(workspace, 256))
    return fail(NVFP4KV_ERR_WORKSPACE_TOO_SMALL, "workspace needs %llu bytes, 256-aligned",
                (unsigned long long)info->workspace_bytes);
  if (info->device >= 0) {  // the plan's SM count, occupancy and smem sizing
    int cur = -1;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (cur != info->device)
      return fail(NVFP4KV_ERR_PLAN_MISMATCH, "plan made for device %d, current device is %d",
                  info->device, cur);
  }
  if (info->num_units == 0) return NVFP4KV_OK;
  if (!q || !kv_indices || !out)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "null q / kv_indices / out");
  if (!aligned(q, 16) || qst % 8 || qsh % 8 || qst < 0 || qsh < 0 || !aligned(out, 4))
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT,
                "q must be 16-byte aligned with strides multiple of 8 elements");
  return NVFP4KV_OK;
}

}  // namespace

namespace nvfp4kv {
// The argument checks of nvfp4kv_decode_run, for entry points that must
// validate before they enqueue anything of their own.
int validate_run(const nvfp4kv_plan_info* info, const void* q, int64_t qst, int64_t qsh,
                 const nvfp4kv_paged_cache* cache, const int32_t* kv_indices,
                 const void* workspace, uint64_t workspace_bytes, const void* out) {
  return check_run(info, q, qst, qsh, cache, kv_indices, workspace, workspace_bytes, out);
}
}  // namespace nvfp4kv

namespace {

struct NewTokens {
  const void* k = nullptr;
  const void* v = nullptr;
  int64_t k_stride_tok = 0, k_stride_head = 0, v_stride_tok = 0, v_stride_head = 0;
};

int attend(const nvfp4kv_plan_info* info, const void* q_bf16, int64_t q_stride_tok,
           int64_t q_stride_head, const nvfp4kv_paged_cache* cache, const int32_t* kv_indices,
           float sm_scale, void* workspace, uint64_t workspace_bytes, void* out_bf16,
           float* lse, cudaStream_t stream, const NewTokens* nt) {
  if (int st = check_run(info, q_bf16, q_stride_tok, q_stride_head, cache, kv_indices,
                         workspace, workspace_bytes, out_bf16))
    return st;
  if (nt) {
    if (info->kernel != kKernelTensorCore && info->kernel != kKernelTcgen05 &&
        info->kernel != kKernelFp4QP)
      return fail(NVFP4KV_ERR_UNSUPPORTED, "the fused append runs in the tensor-core kernels");
    if (info->num_units > 0 &&
        (!nt->k || !nt->v || !aligned(nt->k, 16) || !aligned(nt->v, 16) ||
         nt->k_stride_tok % 8 || nt->k_stride_head % 8 || nt->v_stride_tok % 8 ||
         nt->v_stride_head % 8 || nt->k_stride_tok < 0 || nt->k_stride_head < 0 ||
         nt->v_stride_tok < 0 || nt->v_stride_head < 0))
      return fail(NVFP4KV_ERR_INVALID_ARGUMENT,
                  "new K/V must be 16-byte aligned with strides multiple of 8 elements");
  }
  if (info->num_units == 0) return ok();
  AttendConfig cfg{};
  // a tensor-core plan of one block of <= 8 rows runs the bulk-copy decode
  // kernel when the cache layout allows it (same arithmetic, same occupancy
  // or better: the plan's one-wave grid stays one wave)
  const bool dec = info->kernel == kKernelTensorCore && info->rows_per_block == 8 &&
                   info->page_size == kPageSize && bulk_decode_layout(cache) &&
                   attend_config_dec(info->head_dim_qk, info->head_dim_vo, 8,
                                     info->num_units <= info->num_sms ? 1 : 4, &cfg);
  if (!dec && !lookup_kernel(info->kernel, info->head_dim_qk, info->head_dim_vo,
                             info->rows_per_block, &cfg))
    return fail(NVFP4KV_ERR_UNSUPPORTED, "planned kernel not available");
  cudaError_t e = prepare_kernel(cfg);
  if (e != cudaSuccess) return cuda_fail(e, "kernel attributes");
  if (!(sm_scale > 0.f)) sm_scale = 1.0f / std::sqrt(static_cast<float>(info->head_dim_qk));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  AttendParams p{};
  p.q = static_cast<const uint16_t*>(q_bf16);
  p.q_stride_tok = q_stride_tok;
  p.q_stride_head = q_stride_head;
  p.cache = view_of(cache);
  p.kv_indices = kv_indices;
  p.units = reinterpret_cast<const WorkUnit*>(ws + info->off_units);
  p.num_units = info->num_units;
  p.num_qo_heads = info->num_qo_heads;
  p.group = info->num_qo_heads / info->num_kv_heads;
  p.causal = info->causal;
  p.split = info->split;
  p.page_size = info->page_size;
  p.out_f16 = info->out_dtype == 1;
  p.qk_scale_log2 = static_cast<float>(static_cast<double>(sm_scale) *
                                       cache->k_global_scale * 1.4426950408889634);
  p.v_scale = cache->v_global_scale;
  p.out = static_cast<uint16_t*>(out_bf16);
  p.lse = lse;
  p.partial_o = reinterpret_cast<float*>(ws + info->off_partial_o);
  p.partial_lse = reinterpret_cast<float*>(ws + info->off_partial_lse);
  p.counters = reinterpret_cast<int*>(ws + info->off_counters);
  p.flags = reinterpret_cast<uint32_t*>(ws + info->off_flags);
  p.live_last_page_len = info->device_last_page_len;
  if (nt) {
    p.new_k = static_cast<const uint16_t*>(nt->k);
    p.new_v = static_cast<const uint16_t*>(nt->v);
    p.nk_stride_tok = nt->k_stride_tok;
    p.nk_stride_head = nt->k_stride_head;
    p.nv_stride_tok = nt->v_stride_tok;
    p.nv_stride_head = nt->v_stride_head;
    p.k_global_scale = cache->k_global_scale;
    p.v_global_scale = cache->v_global_scale;
  }
  if (info->kernel == kKernelFp4QP) {
    // FP4 query and probabilities: the row-maximum pass (which also stores
    // the fused append's tokens), then the attention pass with those maxima
    AttendConfig mcfg{};
    if (!attend_config_tc_fp4qp(info->head_dim_qk, info->head_dim_vo, info->rows_per_block, 1,
                                &mcfg))
      return fail(NVFP4KV_ERR_UNSUPPORTED, "planned kernel not available");
    e = prepare_kernel(mcfg);
    if (e != cudaSuccess) return cuda_fail(e, "kernel attributes");
    p.row_max = reinterpret_cast<float*>(ws + info->off_row_max);
    p.row_max_splits = std::max(info->max_units_per_request, 1);
    e = launch_attend(mcfg, p, info->num_units, info->row_blocks, stream);
    if (e != cudaSuccess) return cuda_fail(e, "row-maximum launch");
    p.new_k = nullptr;
    p.new_v = nullptr;
  }
  e = launch_attend(cfg, p, info->num_units, info->row_blocks, stream);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return ok();
}

}  // namespace

extern "C" {

int nvfp4kv_decode_attend(const nvfp4kv_plan_info* info, const void* q_bf16,
                          int64_t q_stride_tok, int64_t q_stride_head,
                          const nvfp4kv_paged_cache* cache, const int32_t* kv_indices,
                          float sm_scale, void* workspace, uint64_t workspace_bytes,
                          void* out_bf16, float* lse, cudaStream_t stream) {
  return attend(info, q_bf16, q_stride_tok, q_stride_head, cache, kv_indices, sm_scale,
                workspace, workspace_bytes, out_bf16, lse, stream, nullptr);
}

int nvfp4kv_decode_append_run(const nvfp4kv_plan_info* info, const void* new_k_bf16,
                              int64_t k_stride_tok, int64_t k_stride_head,
                              const void* new_v_bf16, int64_t v_stride_tok,
                              int64_t v_stride_head, const void* q_bf16,
                              int64_t q_stride_tok, int64_t q_stride_head,
                              const nvfp4kv_paged_cache* cache, const int32_t* kv_indices,
                              float sm_scale, void* workspace, uint64_t workspace_bytes,
                              void* out_bf16, float* lse, cudaStream_t stream) {
  NewTokens nt;
  nt.k = new_k_bf16;
  nt.v = new_v_bf16;
  nt.k_stride_tok = k_stride_tok;
  nt.k_stride_head = k_stride_head;
  nt.v_stride_tok = v_stride_tok;
  nt.v_stride_head = v_stride_head;
  return attend(info, q_bf16, q_stride_tok, q_stride_head, cache, kv_indices, sm_scale,
                workspace, workspace_bytes, out_bf16, lse, stream, &nt);
}

int nvfp4kv_decode_merge(const nvfp4kv_plan_info* info, void* workspace,
                         uint64_t workspace_bytes, void* out_bf16, float* lse,
                         cudaStream_t stream) {
  if (!info || info->magic != kPlanMagic)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "info is not a plan");
  if (!info->split) return ok();
  if (!workspace || workspace_bytes < info->workspace_bytes || !aligned(workspace, 256))
    return fail(NVFP4KV_ERR_WORKSPACE_TOO_SMALL, "workspace needs %llu bytes",
                (unsigned long long)info->workspace_bytes);
  if (!out_bf16) return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "out is null");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = launch_merge(
      reinterpret_cast<const float*>(ws + info->off_partial_o),
      reinterpret_cast<const float*>(ws + info->off_partial_lse),
      reinterpret_cast<const int32_t*>(ws + info->off_merge_indptr),
      static_cast<int32_t>((int64_t)info->total_qo_rows * info->num_qo_heads),
      info->head_dim_vo, static_cast<uint16_t*>(out_bf16), lse, info->out_dtype == 1, stream);
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return ok();
}

int nvfp4kv_decode_run(const nvfp4kv_plan_info* info, const void* q_bf16,
                       int64_t q_stride_tok, int64_t q_stride_head,
                       const nvfp4kv_paged_cache* cache, const int32_t* kv_indices,
                       float sm_scale, void* workspace, uint64_t workspace_bytes,
                       void* out_bf16, float* lse, cudaStream_t stream) {
  // the split-KV merge is fused into the attention kernel
  return nvfp4kv_decode_attend(info, q_bf16, q_stride_tok, q_stride_head, cache, kv_indices,
                               sm_scale, workspace, workspace_bytes, out_bf16, lse, stream);
}

int nvfp4kv_merge_states(const float* o_partial, const float* lse_partial,
                         const int32_t* merge_indptr, int32_t num_entries,
                         int32_t head_dim_vo, void* out_bf16, float* lse,
                         cudaStream_t stream) {
  if (num_entries < 0) return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "num_entries < 0");
  if (head_dim_vo <= 0 || head_dim_vo % 32 || head_dim_vo > 512)
    return fail(NVFP4KV_ERR_UNSUPPORTED, "head_dim_vo %d: multiple of 32, at most 512",
                head_dim_vo);
  if (num_entries == 0) return ok();
  if (!o_partial || !lse_partial || !merge_indptr || !out_bf16)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "null pointer");
  if (!aligned(o_partial, 16) || !aligned(out_bf16, 2))
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "o_partial must be 16-byte aligned");
  cudaError_t e = launch_merge(o_partial, lse_partial, merge_indptr, num_entries, head_dim_vo,
                               static_cast<uint16_t*>(out_bf16), lse, false, stream);
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return ok();
}

int nvfp4kv_workspace_flags(const nvfp4kv_plan_info* info, const void* workspace,
                            uint32_t* flags, int32_t clear, cudaStream_t stream) {
  if (!info || info->magic != kPlanMagic || !workspace || !flags)
    return fail(NVFP4KV_ERR_INVALID_ARGUMENT, "bad arguments");
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws + info->off_flags, 4, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "flag read");
  if (clear) {
    e = cudaMemsetAsync(const_cast<uint8_t*>(ws) + info->off_flags, 0, 4, stream);
    if (e != cudaSuccess) return cuda_fail(e, "flag clear");
  }
  *flags = v;
  if (v) return fail(NVFP4KV_ERR_DEVICE_CHECK, "device flags 0x%x", v);
  return ok();
}

}  // extern "C"
