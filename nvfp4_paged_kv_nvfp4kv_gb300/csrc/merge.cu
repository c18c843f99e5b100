// merge.cu -- log-sum-exp merge of split-KV partial states, sm_103a.
//
// For entry e with partials i in [indptr[e], indptr[e+1]) (flash-decoding of
// page "Re-enable split-KV for NVFP4 KV cache in prefill path"; the pages
// give no formula, this is the standard one):
//   M = max_i lse_i, lse = M + ln sum_i exp(lse_i - M),
//   o = sum_i exp(lse_i - lse) o_i;  no finite lse_i -> o = 0, lse = -inf.
// One warp per entry; each lane owns DV/32 consecutive dims.
#include <cstdint>

#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace nvfp4kv {
namespace {

template <int PER>
__global__ void __launch_bounds__(256)
    merge_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                 const int32_t* __restrict__ indptr, int32_t n, int32_t dv,
                 uint16_t* __restrict__ out, float* __restrict__ lse, bool out_f16) {
  const int lane = threadIdx.x & 31;
  const int64_t e = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (e >= n) return;
  const int beg = indptr[e], end = indptr[e + 1];
  float M = -INFINITY;
  for (int i = beg + lane; i < end; i += 32) M = fmaxf(M, lse_part[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
  float L = -INFINITY;
  if (M != -INFINITY) {
    float S = 0.f;
    for (int i = beg + lane; i < end; i += 32) S += expf(lse_part[i] - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    L = M + logf(S);
#pragma unroll 4
    for (int i = beg; i < end; ++i) {
      const float w = expf(lse_part[i] - L);
      const float* src = o_part + static_cast<int64_t>(i) * dv + lane * PER;
      if constexpr (PER % 4 == 0) {
#pragma unroll
        for (int k = 0; k < PER; k += 4) {
          const float4 v = *reinterpret_cast<const float4*>(src + k);
          acc[k] += w * v.x;
          acc[k + 1] += w * v.y;
          acc[k + 2] += w * v.z;
          acc[k + 3] += w * v.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < PER; ++k) acc[k] += w * src[k];
      }
    }
  }
  uint16_t* dst = out + e * dv + lane * PER;
#pragma unroll
  for (int k = 0; k < PER; ++k) dst[k] = pack_out1(acc[k], out_f16);
  if (lane == 0 && lse) lse[e] = L;
}

}  // namespace

cudaError_t launch_merge(const float* o_partial, const float* lse_partial,
                         const int32_t* merge_indptr, int32_t num_entries,
                         int32_t head_dim_vo, uint16_t* out, float* lse, bool out_f16,
                         cudaStream_t stream) {
  if (num_entries == 0) return cudaSuccess;
  const int warps = 8;
  const int blocks = (num_entries + warps - 1) / warps;
  const int per = head_dim_vo / 32;
#define NVFP4KV_MERGE(PER_)                                                          \
  case PER_:                                                                       \
    merge_kernel<PER_><<<blocks, warps * 32, 0, stream>>>(                         \
        o_partial, lse_partial, merge_indptr, num_entries, head_dim_vo, out, lse, out_f16); \
    break;
  switch (per) {
    NVFP4KV_MERGE(1)
    NVFP4KV_MERGE(2)
    NVFP4KV_MERGE(3)
    NVFP4KV_MERGE(4)
    NVFP4KV_MERGE(5)
    NVFP4KV_MERGE(6)
    NVFP4KV_MERGE(7)
    NVFP4KV_MERGE(8)
    NVFP4KV_MERGE(12)
    NVFP4KV_MERGE(16)
    default:
      return cudaErrorInvalidValue;
  }
#undef NVFP4KV_MERGE
  return cudaGetLastError();
}

}  // namespace nvfp4kv
