// append_fused.cuh -- the append step inside an attention launch: a work
// unit quantises the step's new tokens of its kv head that fall in its pages
// (token positions [lo, hi)) and stores them into the cache, with the same
// exact recipe as the standalone quantize_append kernel.  The new tokens'
// bf16 rows are row-aligned with the query rows: row qo_begin + i holds the
// token at position kv_len - qo_len + i.
#pragma once

#include <cstdint>

#include "device_common.cuh"
#include "internal.h"
#include "quantize.cuh"

namespace nvfp4kv {

// With owners > 1 only the tokens of the unit's pages rel with
// rel % owners == owner are handled (the pages one warp of a CTA streams).
template <int DK, int DV>
__device__ __forceinline__ void append_unit_tokens(const AttendParams& p, const WorkUnit& u,
                                                   int lo, int hi, int tid, int nthreads,
                                                   int owner = 0, int owners = 1) {
  const int first_new = u.kv_len - u.qo_len;
  constexpr int NB = DK / 16 + DV / 16;
  for (int idx = tid; idx < (hi - lo) * NB; idx += nthreads) {
    const int tok = lo + idx / NB, blk = idx % NB, i = tok - first_new;
    if (owners > 1 && ((tok - u.tok_begin) / 16) % owners != owner) continue;
    const bool isv = blk >= DK / 16;
    const int jb = isv ? blk - DK / 16 : blk;
    const uint16_t* src =
        isv ? p.new_v + (int64_t)(u.qo_begin + i) * p.nv_stride_tok +
                  (int64_t)u.h_kv * p.nv_stride_head
            : p.new_k + (int64_t)(u.qo_begin + i) * p.nk_stride_tok +
                  (int64_t)u.h_kv * p.nk_stride_head;
    const uint4 lo16 = *reinterpret_cast<const uint4*>(src + 16 * jb);
    const uint4 hi16 = *reinterpret_cast<const uint4*>(src + 16 * jb + 8);
    const int32_t page = p.kv_indices[u.page_begin + (tok - u.tok_begin) / p.page_size];
    if (page < 0 || page >= p.cache.num_pages) {
      atomicOr(p.flags, 0x2u);
      continue;
    }
    const int slot = tok % p.page_size;
    uint2 packed;
    const uint32_t sfb =
        quantize_block16(lo16, hi16, isv ? p.v_global_scale : p.k_global_scale, &packed);
    const CacheView& c = p.cache;
    uint8_t* drow = const_cast<uint8_t*>(
        isv ? c.v_data + page * c.v_sp + slot * c.v_ss + u.h_kv * c.v_sh
            : c.k_data + page * c.k_sp + slot * c.k_ss + u.h_kv * c.k_sh);
    uint8_t* srow = const_cast<uint8_t*>(
        isv ? c.v_sf + page * c.vsf_sp + slot * c.vsf_ss + u.h_kv * c.vsf_sh
            : c.k_sf + page * c.ksf_sp + slot * c.ksf_ss + u.h_kv * c.ksf_sh);
    *reinterpret_cast<uint2*>(drow + 8 * jb) = packed;
    srow[jb] = static_cast<uint8_t>(sfb);
  }
  __threadfence();  // before other CTAs' copies of the page read them
}

}  // namespace nvfp4kv
