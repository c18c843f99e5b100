// quantize_append.cu -- bf16 -> NVFP4 quantise-into-page kernel, sm_103a.
//
// Per 16-element block of one token and kv head (the NVFP4 KV layout of page
// "Support NVFP4 KV cache decode on SM120": packed e2m1 + one E4M3 scale per
// 16 head-dim elements + one FP32 global scale per tensor):
//   s = E4M3_RNE_satfinite(amax / (6 g)),
//   code_i = e2m1_RNE_satfinite(x_i / (s g)) with ties to the even code and
//   the sign of x_i kept on zero codes, packed low nibble = even element.
// Every rounding decision is the exact-real one, in float32 only (float64 is
// a slow pipe on this part):
//  * an approximate t = amax / g / 6 (two correctly rounded divisions, a few
//    ulps from the exact ratio) is rounded to E4M3 by the hardware RN
//    conversion; the E4M3 grid is 2^-4 relative or coarser, so the exact
//    answer is that code or a neighbour, decided by comparing amax with
//    6 * midpoint * g exactly;
//  * element codes compare |x| with the seven e2m1 midpoints times s g.
// An exact comparison of a with m * g (m, g, a positive floats): m * g = P + E
// exactly with P = RN(m g) and E = fma(m, g, -P); a - P is exact when a and P
// are within a factor of two and otherwise much larger than |E|, so the sign
// of (a - P) - E is the sign of a - m g, and zero means a tie.
// One thread per block; the bf16 loads are issued before the page lookup; a
// token whose request, position or page id is out of range is skipped and
// flagged.  Global scales lie in [2^-64, 2^64] (checked on the host), so no
// product underflows or overflows.
#include <cstdint>

#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace nvfp4kv {
namespace {

__device__ __forceinline__ float e4m3_code_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xF, m = code & 7;
  if (e == 0) return static_cast<float>(m) * (1.0f / 512.0f);
  return __uint_as_float(((e - 7 + 127) << 23) | (m << 20));
}

// sign(a - m * g), exactly (see the file comment)
__device__ __forceinline__ int cmp_prod(float a, float m, float g) {
  const float P = __fmul_rn(m, g);
  const float E = fmaf(m, g, -P);
  const float d = __fsub_rn(a, P);
  return (d > E) - (d < E);
}

// E4M3 code of amax / (6 g): round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t scale_code(float amax, float g) {
  if (amax == 0.f) return 0u;
  const float t = __fdiv_rn(__fdiv_rn(amax, g), 6.0f);
  unsigned short pair;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(pair) : "f"(0.0f), "f"(t));
  uint32_t c = pair & 0xFFu;
  if (c > 0u) {  // below the midpoint with the code under c?
    const float mid = 0.5f * (e4m3_code_value(c - 1) + e4m3_code_value(c));
    const int sgn = cmp_prod(amax, 6.0f * mid, g);
    if (sgn < 0 || (sgn == 0 && (c & 1u))) return c - 1;
  }
  if (c < 0x7Eu) {  // above the midpoint with the code over c?
    const float mid = 0.5f * (e4m3_code_value(c) + e4m3_code_value(c + 1));
    const int sgn = cmp_prod(amax, 6.0f * mid, g);
    if (sgn > 0 || (sgn == 0 && (c & 1u))) return c + 1;
  }
  return c;
}

__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
  const int bpk = p.head_dim_qk / 16, bpv = p.head_dim_vo / 16;
  const int per = bpk + bpv;
  const int64_t total = static_cast<int64_t>(p.nnz) * p.num_kv_heads * per;
  const float mids[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       idx < total; idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int blk = static_cast<int>(idx % per);
    const int64_t th = idx / per;
    const int h = static_cast<int>(th % p.num_kv_heads);
    const int t = static_cast<int>(th / p.num_kv_heads);
    const bool isv = blk >= bpk;
    const int jb = isv ? blk - bpk : blk;

    // the block's bf16 values (independent of the page lookup below)
    const uint16_t* src = isv ? p.v + t * p.v_stride_tok + h * p.v_stride_head
                              : p.k + t * p.k_stride_tok + h * p.k_stride_head;
    src += 16 * jb;
    const uint4 lo = *reinterpret_cast<const uint4*>(src);
    const uint4 hi = *reinterpret_cast<const uint4*>(src + 8);

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

    const float g = isv ? p.v_global_scale : p.k_global_scale;
    const uint32_t sfb = scale_code(amax, g);
    const float s = e4m3_code_value(sfb);
    // thresholds T_k = mid_k * s * g: Tf_k = T_k rounded down to float32 and
    // whether that was exact.  |x| > T_k <=> |x| > Tf_k for a float |x|; a
    // tie needs T_k exact (|x| == Tf_k < T_k is simply below the threshold)
    float tf[7];
    bool ex[7];
#pragma unroll
    for (int k = 0; k < 7; ++k) {
      const float ms = mids[k] * s;  // exact: at most 7 significant bits
      const float P = __fmul_rn(ms, g);
      const float E = fmaf(ms, g, -P);
      tf[k] = E < 0.f ? __uint_as_float(__float_as_uint(P) - 1u) : P;
      ex[k] = E == 0.f;
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
