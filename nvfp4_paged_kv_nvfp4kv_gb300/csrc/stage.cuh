// stage.cuh -- shared-memory stage of one page (16 tokens of one kv head)
// and the cp.async copies that fill it; shared by the attention kernels.
#pragma once

#include <cstdint>

#include "device_common.cuh"
#include "internal.h"

namespace nvfp4kv {

// Stage layout: packed K rows [16][Dk/2], K scale rows [16][Dk/16], packed V
// rows [16][Dv/2 + 16], V scale rows [16][Dv/16]; every section starts
// 16-byte aligned.  Filled by per-lane cp.async: odd K rows are xor-swizzled
// by 4 chunks when Dk >= 256 (a lane quad's 16-byte reads of two rows then
// hit different banks) and V rows are padded by 16 bytes (the PV reads of
// lane group g at tokens 2t.. hit distinct banks).  Bulk copies of a page's
// contiguous bytes (no padding, no swizzle) measured slower.
template <int DK, int DV>
struct PageStage {
  static constexpr int KROW = DK / 2;
  static constexpr bool KSWZ = DK >= 256;
  static constexpr int KSFROW = DK / 16;
  static constexpr int VC = DV / 16;
  static constexpr int VROW = DV / 2 + 16;
  static constexpr int VSFROW = DV / 16;
  static constexpr int K_BYTES = 16 * KROW;
  static constexpr int KSF_BYTES = 16 * KSFROW;
  static constexpr int V_BYTES = 16 * VROW;
  static constexpr int VSF_BYTES = 16 * VSFROW;
  static constexpr int OFF_KSF = K_BYTES;
  static constexpr int OFF_V = (OFF_KSF + KSF_BYTES + 15) / 16 * 16;
  static constexpr int OFF_VSF = OFF_V + V_BYTES;
  static constexpr int STAGE_BYTES = (OFF_VSF + VSF_BYTES + 15) / 16 * 16;
  static_assert(DK % 64 == 0 && DV % 64 == 0, "head dims");
  static_assert(VROW % 16 == 0, "V rows must stay 16-byte aligned");

  __device__ static __forceinline__ int k_pos(int row, int chunk) {
    return KSWZ ? (chunk ^ ((row & 1) << 2)) : chunk;
  }
};

// Copy one page (16 tokens of kv head h, page id pid) into a warp's stage
// (without WITH_V: its K rows and K scales only).
template <class S, bool WITH_V = true>
__device__ __forceinline__ void issue_page(uint8_t* st, const CacheView& c, int32_t pid,
                                           int h, int lane) {
  using namespace dev;
  const uint8_t* kb = c.k_data + pid * c.k_sp + h * c.k_sh;
  const uint8_t* vb = c.v_data + pid * c.v_sp + h * c.v_sh;
  const uint8_t* ksb = c.k_sf + pid * c.ksf_sp + h * c.ksf_sh;
  const uint8_t* vsb = c.v_sf + pid * c.vsf_sp + h * c.vsf_sh;
  constexpr int KCH = S::KROW / 16;       // 16-byte chunks per K row
  constexpr int VCHR = (S::VC * 8) / 16;  // 16-byte chunks per V row
#pragma unroll
  for (int ci = lane; ci < 16 * KCH; ci += 32) {
    const int r = ci / KCH, ch = ci % KCH;
    cp_async_16(st + r * S::KROW + S::k_pos(r, ch) * 16, kb + r * c.k_ss + ch * 16);
  }
#pragma unroll
  for (int ci = lane; WITH_V && ci < 16 * VCHR; ci += 32) {
    const int r = ci / VCHR, ch = ci % VCHR;
    cp_async_16(st + S::OFF_V + r * S::VROW + ch * 16, vb + r * c.v_ss + ch * 16);
  }
  constexpr int KSU = S::KSFROW < 16 ? S::KSFROW : 16;
  constexpr int KSN = S::KSFROW / KSU;
#pragma unroll
  for (int ci = lane; ci < 16 * KSN; ci += 32) {
    const int r = ci / KSN, u = ci % KSN;
    cp_async_small<KSU>(st + S::OFF_KSF + r * S::KSFROW + u * KSU,
                        ksb + r * c.ksf_ss + u * KSU);
  }
  constexpr int VSU = S::VSFROW < 16 ? S::VSFROW : 16;
  constexpr int VSN = S::VSFROW / VSU;
#pragma unroll
  for (int ci = lane; WITH_V && ci < 16 * VSN; ci += 32) {
    const int r = ci / VSN, u = ci % VSN;
    cp_async_small<VSU>(st + S::OFF_VSF + r * S::VSFROW + u * VSU,
                        vsb + r * c.vsf_ss + u * VSU);
  }
}

// Page size 1: the 16 token rows of a tile come from 16 pages (slot 0 each).
// pid_lane: lane r (r < 16) holds the page id of row r (lanes 16-31 repeat
// lanes 0-15); every lane takes the id of the row it copies by a shuffle,
// executed by all lanes before the copy's own condition.
template <class S, bool WITH_V = true>
__device__ __forceinline__ void issue_tile_rows(uint8_t* st, const CacheView& c,
                                                int32_t pid_lane, int h, int lane) {
  using namespace dev;
  constexpr int KCH = S::KROW / 16;
  constexpr int VCHR = (S::VC * 8) / 16;
#pragma unroll
  for (int k = 0; k < (16 * KCH + 31) / 32; ++k) {
    const int ci = lane + 32 * k;
    const int r = ci / KCH, ch = ci % KCH;
    const int32_t pr = __shfl_sync(0xffffffffu, pid_lane, r & 15);
    if (ci < 16 * KCH)
      cp_async_16(st + r * S::KROW + S::k_pos(r, ch) * 16,
                  c.k_data + pr * c.k_sp + h * c.k_sh + ch * 16);
  }
#pragma unroll
  for (int k = 0; k < (WITH_V ? (16 * VCHR + 31) / 32 : 0); ++k) {
    const int ci = lane + 32 * k;
    const int r = ci / VCHR, ch = ci % VCHR;
    const int32_t pr = __shfl_sync(0xffffffffu, pid_lane, r & 15);
    if (ci < 16 * VCHR)
      cp_async_16(st + S::OFF_V + r * S::VROW + ch * 16,
                  c.v_data + pr * c.v_sp + h * c.v_sh + ch * 16);
  }
  constexpr int KSU = S::KSFROW < 16 ? S::KSFROW : 16;
  constexpr int KSN = S::KSFROW / KSU;
#pragma unroll
  for (int k = 0; k < (16 * KSN + 31) / 32; ++k) {
    const int ci = lane + 32 * k;
    const int r = ci / KSN, u = ci % KSN;
    const int32_t pr = __shfl_sync(0xffffffffu, pid_lane, r & 15);
    if (ci < 16 * KSN)
      cp_async_small<KSU>(st + S::OFF_KSF + r * S::KSFROW + u * KSU,
                          c.k_sf + pr * c.ksf_sp + h * c.ksf_sh + u * KSU);
  }
  constexpr int VSU = S::VSFROW < 16 ? S::VSFROW : 16;
  constexpr int VSN = S::VSFROW / VSU;
#pragma unroll
  for (int k = 0; k < (WITH_V ? (16 * VSN + 31) / 32 : 0); ++k) {
    const int ci = lane + 32 * k;
    const int r = ci / VSN, u = ci % VSN;
    const int32_t pr = __shfl_sync(0xffffffffu, pid_lane, r & 15);
    if (ci < 16 * VSN)
      cp_async_small<VSU>(st + S::OFF_VSF + r * S::VSFROW + u * VSU,
                          c.v_sf + pr * c.vsf_sp + h * c.vsf_sh + u * VSU);
  }
}

}  // namespace nvfp4kv
