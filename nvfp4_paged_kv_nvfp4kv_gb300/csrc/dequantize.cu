// dequantize.cu -- paged NVFP4 -> float32, sm_103a.
//
// The inverse of the cache format (page "Support NVFP4 KV cache decode on
// SM120": packed e2m1 codes, one E4M3 scale per 16 head-dim elements, one
// float32 global scale per tensor): x_hat = e2m1(code) * E4M3(scale) * g.
// code * scale is exact in float32 (at most 2 + 4 significant bits), so the
// one rounding is that of the product with g: the result is the exact value
// rounded to float32.  The prefill tests of page "Re-enable split-KV for
// NVFP4 KV cache in prefill path" compare attention against a dequantised
// copy of the cache; this kernel gives that copy on the device.
//
// A warp takes one (page, slot, head) row at a time; lane l converts the
// 4-element groups l, l + 32, ... of the row's K and of its V: 2 code bytes
// and the block's scale byte in, one 16-byte float4 out, so a warp's stores
// are 512 contiguous bytes.  A CTA takes whole page entries (grid-stride).
// A page id outside the pool writes zeros and sets flag 0x1.
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace nvfp4kv {
namespace {

// 4 elements from 2 code bytes: code * scale (exact in float32) times g, one
// rounding
__device__ __forceinline__ float4 dequant4(uint32_t codes, float sc, float g) {
  uint32_t h4[4];
  dev::e2m1x8_to_f16x8(codes, h4);  // byte j -> h4[j], even element in the low half
  auto f = [](uint32_t h) { return __half2float(__ushort_as_half(static_cast<unsigned short>(h))); };
  return make_float4((f(h4[0] & 0xFFFFu) * sc) * g, (f(h4[0] >> 16) * sc) * g,
                     (f(h4[1] & 0xFFFFu) * sc) * g, (f(h4[1] >> 16) * sc) * g);
}

__global__ void __launch_bounds__(256) dequantize_kernel(const DequantParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int rows = p.page_size * p.num_kv_heads;
  for (int e = blockIdx.x; e < p.num_ids; e += gridDim.x) {
    const int32_t page = p.page_ids[e];
    const bool bad = page < 0 || page >= p.num_pages;
    if (bad && threadIdx.x == 0 && p.flags) atomicOr(p.flags, 0x1u);
    for (int r = warp; r < rows; r += nwarps) {
      const int slot = r / p.num_kv_heads, h = r % p.num_kv_heads;
      const int64_t orow = (static_cast<int64_t>(e) * p.page_size + slot) * p.num_kv_heads + h;
      if (p.k_out) {
        float* dst = p.k_out + orow * p.head_dim_qk;
        const uint8_t* row = p.k_data + page * p.k_sp + slot * p.k_ss + h * p.k_sh;
        const uint8_t* sfp = p.k_sf + page * p.ksf_sp + slot * p.ksf_ss + h * p.ksf_sh;
        for (int gg = lane; gg < p.head_dim_qk / 4; gg += 32) {
          float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
          if (!bad) {
            const uint32_t s2 = dev::e4m3x2_to_f16x2(sfp[gg / 4]);
            const float sc = __half2float(__ushort_as_half(static_cast<unsigned short>(s2 & 0xFFFFu)));
            o = dequant4(*reinterpret_cast<const uint16_t*>(row + 2 * gg), sc, p.k_global_scale);
          }
          reinterpret_cast<float4*>(dst)[gg] = o;
        }
      }
      if (p.v_out) {
        float* dst = p.v_out + orow * p.head_dim_vo;
        const uint8_t* row = p.v_data + page * p.v_sp + slot * p.v_ss + h * p.v_sh;
        const uint8_t* sfp = p.v_sf + page * p.vsf_sp + slot * p.vsf_ss + h * p.vsf_sh;
        for (int gg = lane; gg < p.head_dim_vo / 4; gg += 32) {
          float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
          if (!bad) {
            const uint32_t s2 = dev::e4m3x2_to_f16x2(sfp[gg / 4]);
            const float sc = __half2float(__ushort_as_half(static_cast<unsigned short>(s2 & 0xFFFFu)));
            o = dequant4(*reinterpret_cast<const uint16_t*>(row + 2 * gg), sc, p.v_global_scale);
          }
          reinterpret_cast<float4*>(dst)[gg] = o;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_dequantize(const DequantParams& p, cudaStream_t stream) {
  if (p.num_ids == 0 || (!p.k_out && !p.v_out)) return cudaSuccess;
  const int blocks = p.num_ids < 152 * 8 ? p.num_ids : 152 * 8;
  dequantize_kernel<<<blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace nvfp4kv
