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
// One thread per 16-element block of one (page, slot, head): 8 code bytes and
// one scale byte in, 64 bytes of float32 out.  A page id outside the pool
// writes zeros and sets flag 0x1.
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace nvfp4kv {
namespace {

__global__ void __launch_bounds__(256) dequantize_kernel(const DequantParams p) {
  const int bpk = p.k_out ? p.head_dim_qk / 16 : 0;
  const int bpv = p.v_out ? p.head_dim_vo / 16 : 0;
  const int per = bpk + bpv;
  const int64_t total = static_cast<int64_t>(p.num_ids) * p.page_size * p.num_kv_heads * per;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int blk = static_cast<int>(idx % per);
    const int64_t rest = idx / per;
    const int h = static_cast<int>(rest % p.num_kv_heads);
    const int64_t ps = rest / p.num_kv_heads;  // page entry * page_size + slot
    const int slot = static_cast<int>(ps % p.page_size);
    const int64_t e = ps / p.page_size;
    const bool isv = blk >= bpk;
    const int jb = isv ? blk - bpk : blk;
    const int d = isv ? p.head_dim_vo : p.head_dim_qk;
    float* dst = (isv ? p.v_out : p.k_out) + (ps * p.num_kv_heads + h) * d + 16 * jb;
    const int32_t page = p.page_ids[e];
    float4 o[4];
    if (page < 0 || page >= p.num_pages) {
      if (p.flags) atomicOr(p.flags, 0x1u);
      for (int k = 0; k < 4; ++k) o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      const uint8_t* row = isv ? p.v_data + page * p.v_sp + slot * p.v_ss + h * p.v_sh
                               : p.k_data + page * p.k_sp + slot * p.k_ss + h * p.k_sh;
      const uint8_t* sfp = isv ? p.v_sf + page * p.vsf_sp + slot * p.vsf_ss + h * p.vsf_sh
                               : p.k_sf + page * p.ksf_sp + slot * p.ksf_ss + h * p.ksf_sh;
      const uint2 codes = *reinterpret_cast<const uint2*>(row + 8 * jb);
      const uint32_t s2 = dev::e4m3x2_to_f16x2(sfp[jb]);
      const float sc = __half2float(__ushort_as_half(static_cast<unsigned short>(s2 & 0xFFFFu)));
      const float g = isv ? p.v_global_scale : p.k_global_scale;
      uint32_t h8[8];
      dev::e2m1x8_to_f16x8(codes.x, *reinterpret_cast<uint32_t(*)[4]>(h8));
      dev::e2m1x8_to_f16x8(codes.y, *reinterpret_cast<uint32_t(*)[4]>(h8 + 4));
      float v[16];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h8[k] & 0xFFFFu)));
        const float hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h8[k] >> 16)));
        v[2 * k] = (lo * sc) * g;  // lo * sc exact; one rounding
        v[2 * k + 1] = (hi * sc) * g;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) o[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) reinterpret_cast<float4*>(dst)[k] = o[k];
  }
}

}  // namespace

cudaError_t launch_dequantize(const DequantParams& p, cudaStream_t stream) {
  const int per = (p.k_out ? p.head_dim_qk / 16 : 0) + (p.v_out ? p.head_dim_vo / 16 : 0);
  const int64_t total = static_cast<int64_t>(p.num_ids) * p.page_size * p.num_kv_heads * per;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  dequantize_kernel<<<static_cast<int>(blocks), threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace nvfp4kv
