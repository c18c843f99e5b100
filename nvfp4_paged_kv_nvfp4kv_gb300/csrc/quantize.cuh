// quantize.cuh -- exact NVFP4 quantisation of one 16-element bf16 block
// (shared by the quantise-append kernel and the fused append + attention).
//
// Recipe: s = E4M3_RNE_satfinite(amax / (6 g)), code_i =
// e2m1_RNE_satfinite(x_i / (s g)), ties to the even code, zero codes keep the
// sign of x_i, low nibble = even element.  Every rounding decision is the
// exact-real one, in float32 only:
//  * an approximate t = amax * RN(1 / RN(6 g)) (a few ulps from the exact
//    ratio; the reciprocal does not depend on the data) is rounded to E4M3 by
//    the hardware RN conversion; the E4M3 grid is 2^-4 relative or coarser,
//    so the exact answer is that code or a neighbour, decided by comparing
//    amax with 6 * midpoint * g exactly (t overflows to inf only far above
//    the saturation point and underflows to 0 only far below the first
//    midpoint);
//  * element codes compare |x| with the seven e2m1 midpoints times s g.
// An exact comparison of a with m * g (m, g, a positive floats): m * g = P + E
// exactly with P = RN(m g) and E = fma(m, g, -P); a - P is exact when a and P
// are within a factor of two and otherwise much larger than |E|, so the sign
// of (a - P) - E is the sign of a - m g, and zero means a tie.  Global scales
// lie in [2^-64, 2^64], so no product underflows or overflows.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

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
// inv6g: RN(1 / RN(6 g)).
__device__ __forceinline__ uint32_t scale_code(float amax, float g, float inv6g) {
  if (amax == 0.f) return 0u;
  const float t = __fmul_rn(amax, inv6g);
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

// Quantise the 16 bf16 values in (lo, hi) with global scale g: returns the
// E4M3 scale byte and writes the 8 packed bytes.
__device__ __forceinline__ uint32_t quantize_block16(uint4 lo, uint4 hi, float g,
                                                     uint2* packed_out) {
  const float mids[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
  const uint32_t wv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  float x[16];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    x[2 * k] = __uint_as_float(wv[k] << 16);
    x[2 * k + 1] = __uint_as_float(wv[k] & 0xFFFF0000u);
  }
  const float inv6g = __frcp_rn(__fmul_rn(6.0f, g));
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(x[k]));
  const uint32_t sfb = scale_code(amax, g, inv6g);
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
  *packed_out = make_uint2(packed[0], packed[1]);
  return sfb;
}

}  // namespace
}  // namespace nvfp4kv
