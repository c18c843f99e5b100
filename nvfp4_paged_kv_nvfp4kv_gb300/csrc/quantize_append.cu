// quantize_append.cu -- bf16 -> NVFP4 quantise-into-page kernel, sm_103a.
//
// Per 16-element block of one token and kv head (the NVFP4 KV layout of page
// "Support NVFP4 KV cache decode on SM120": packed e2m1 + one E4M3 scale per
// 16 head-dim elements + one FP32 global scale per tensor):
//   s = E4M3_RNE_satfinite(amax / (6 g)),
//   code_i = e2m1_RNE_satfinite(x_i / (s g)) with ties to the even code and
//   the sign of x_i kept on zero codes, packed low nibble = even element.
// Every rounding decision is the exact-real one:
//  * amax / (6 g) is formed in float64 (6g exact; one rounding, which cannot
//    cross or land on an E4M3 midpoint since the numerator has 8 significant
//    bits) and rounded to E4M3 by an integer rint on its binade;
//  * instead of dividing x by s g, |x| is compared with the seven e2m1
//    midpoints times s g.  Each threshold T = mid * s * g is exact in
//    float64; it is rounded DOWN to float32 (Tf) with a flag saying whether
//    that was exact, so |x| > T  <=>  |x| > Tf and |x| == T  <=>  (exact and
//    |x| == Tf), all in float32 compares.  A tie takes the even code.
// One thread per block; a token whose request, position or page id is out of
// range is skipped and flagged.
#include <cstdint>

#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace nvfp4kv {
namespace {

// E4M3 (bias 7, 3 mantissa bits, subnormal spacing 2^-9, max 448) code of a
// positive finite double, round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3_code_rne_sat(double v) {
  if (!(v > 0.0)) return 0u;
  if (v > 448.0) return 0x7Eu;
  if (v < 0.015625) {                    // below 2^-6: grid m * 2^-9
    return static_cast<uint32_t>(rint(v * 512.0));  // 8 is the code of 2^-6
  }
  const long long bits = __double_as_longlong(v);
  const int e = static_cast<int>((bits >> 52) & 0x7FF) - 1023;  // v in [2^e, 2^e+1)
  const double up = __longlong_as_double(static_cast<long long>(1023 + 3 - e) << 52);
  const uint32_t r = static_cast<uint32_t>(rint(v * up));      // 8 .. 16
  const uint32_t code = (static_cast<uint32_t>(e + 7) << 3) + (r - 8u);  // 16 carries
  return code > 0x7Eu ? 0x7Eu : code;
}

__device__ __forceinline__ float e4m3_code_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xF, m = code & 7;
  if (e == 0) return static_cast<float>(m) * (1.0f / 512.0f);
  return __uint_as_float(((e - 7 + 127) << 23) | (m << 20));
}

__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
  const int bpk = p.head_dim_qk / 16, bpv = p.head_dim_vo / 16;
  const int per = bpk + bpv;
  const int64_t total = static_cast<int64_t>(p.nnz) * p.num_kv_heads * per;
  const double mids[7] = {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0};
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       idx < total; idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int blk = static_cast<int>(idx % per);
    const int64_t th = idx / per;
    const int h = static_cast<int>(th % p.num_kv_heads);
    const int t = static_cast<int>(th / p.num_kv_heads);
    const bool isv = blk >= bpk;
    const int jb = isv ? blk - bpk : blk;

    // locate the token's page
    const int b = p.batch_idx[t];
    const int pos = p.positions[t];
    int page = -1;
    bool ok = b >= 0 && b < p.batch && pos >= 0;
    if (ok) {
      const int beg = p.kv_indptr[b];
      const int np = p.kv_indptr[b + 1] - beg;
      const int64_t L = np > 0 ? static_cast<int64_t>(np - 1) * kPageSize + p.last_page_len[b] : 0;
      ok = pos < L;
      if (ok) {
        page = p.kv_indices[beg + pos / kPageSize];
        ok = page >= 0 && page < p.num_pages;
      }
    }
    if (!ok) {
      if (p.flags && blk == 0 && h == 0) atomicOr(p.flags, 0x2u);
      continue;
    }
    const int slot = pos % kPageSize;

    const uint16_t* src = isv ? p.v + t * p.v_stride_tok + h * p.v_stride_head
                              : p.k + t * p.k_stride_tok + h * p.k_stride_head;
    src += 16 * jb;
    const uint4 lo = *reinterpret_cast<const uint4*>(src);
    const uint4 hi = *reinterpret_cast<const uint4*>(src + 8);
    const uint32_t wv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    float x[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      x[2 * k] = __uint_as_float(wv[k] << 16);
      x[2 * k + 1] = __uint_as_float(wv[k] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(x[k]));

    const double g = isv ? static_cast<double>(p.v_global_scale)
                         : static_cast<double>(p.k_global_scale);
    const uint32_t sfb = e4m3_code_rne_sat(static_cast<double>(amax) / (6.0 * g));
    const float s = e4m3_code_value(sfb);
    const double sg = static_cast<double>(s) * g;  // exact
    float tf[7];
    bool ex[7];
#pragma unroll
    for (int k = 0; k < 7; ++k) {
      const double T = mids[k] * sg;  // exact
      tf[k] = __double2float_rd(T);
      ex[k] = static_cast<double>(tf[k]) == T;
    }
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float ax = fabsf(x[k]);
      uint32_t c = 0;
      if (s != 0.f) {
#pragma unroll
        for (int m = 0; m < 7; ++m) c += (ax > tf[m]) ? 1u : 0u;
#pragma unroll
        for (int m = 1; m < 7; m += 2)  // ties at odd midpoints round up to even
          if (ex[m] && ax == tf[m]) c = m + 1;
      }
      c |= (__float_as_uint(x[k]) >> 31) << 3;
      packed[k / 8] |= c << (4 * (k % 8));
    }
    uint8_t* drow = isv ? p.v_data + page * p.v_sp + slot * p.v_ss + h * p.v_sh
                        : p.k_data + page * p.k_sp + slot * p.k_ss + h * p.k_sh;
    uint8_t* srow = isv ? p.v_sf + page * p.vsf_sp + slot * p.vsf_ss + h * p.vsf_sh
                        : p.k_sf + page * p.ksf_sp + slot * p.ksf_ss + h * p.ksf_sh;
    *reinterpret_cast<uint2*>(drow + 8 * jb) = make_uint2(packed[0], packed[1]);
    srow[jb] = static_cast<uint8_t>(sfb);
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(p.nnz) * p.num_kv_heads *
                        (p.head_dim_qk / 16 + p.head_dim_vo / 16);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  append_kernel<<<static_cast<int>(blocks), threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace nvfp4kv
