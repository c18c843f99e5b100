// device_common.cuh -- small device helpers (inline PTX written from the PTX
// ISA) used by the attention kernels.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "internal.h"

namespace nvfp4kv {
namespace dev {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// cp.async: 16-byte global->shared copy bypassing L1 (.cg), and 4/8-byte
// copies (.ca; .cg only exists for 16 bytes).
__device__ __forceinline__ void cp_async_16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(smem)),
               "l"(gmem));
}
template <int N>
__device__ __forceinline__ void cp_async_small(void* smem, const void* gmem) {
  static_assert(N == 4 || N == 8 || N == 16, "cp.async size");
  if constexpr (N == 16) {
    cp_async_16(smem, gmem);
  } else {
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;\n" ::"r"(smem_addr(smem)),
                 "l"(gmem), "n"(N));
  }
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::);
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Loads from a 32-bit shared-memory address plus a compile-time byte offset
// (volatile: they stay after the waits and barriers that precede them).
template <int OFF = 0>
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1+%2];\n" : "=r"(v) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF = 0>
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1+%2];\n" : "=r"(v) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF = 0>
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1+%2];\n" : "=r"(v) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF = 0>
__device__ __forceinline__ uint2 lds_v2(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2+%3];\n" : "=r"(v.x), "=r"(v.y) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF = 0>
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4+%5];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a), "n"(OFF));
  return v;
}
// 16-byte cp.async to a 32-bit shared address: shared s + SOFF <- global
// g + GOFF
template <int SOFF = 0, int GOFF = SOFF>
__device__ __forceinline__ void cp_async_16s(uint32_t s, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0+%2], [%1+%3], 16;\n" ::"r"(s), "l"(g), "n"(SOFF),
               "n"(GOFF));
}

// ---- mbarrier ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(count));
}
// make the initialised barriers visible to the async proxy (tcgen05.commit)
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Four packed bytes (8 e2m1 codes) -> four f16x2: h[j] holds byte j, its low
// nibble (the even element) in the low half.
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n"
      " .reg .b8 b0, b1, b2, b3;\n"
      " mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      " cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      " cvt.rn.f16x2.e2m1x2 %3, b3;\n"
      "}\n"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Byte J of w (2 e2m1 codes) -> f16x2, its low nibble in the low half.
template <int J>
__device__ __forceinline__ uint32_t e2m1x2_byte_to_f16x2(uint32_t w) {
  static_assert(J >= 0 && J < 4, "byte index");
  uint32_t h;
  if constexpr (J == 0) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n}\n" : "=r"(h) : "r"(w));
  } else if constexpr (J == 1) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b1;\n}\n" : "=r"(h) : "r"(w));
  } else if constexpr (J == 2) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b2;\n}\n" : "=r"(h) : "r"(w));
  } else {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b3;\n}\n" : "=r"(h) : "r"(w));
  }
  return h;
}

// Two E4M3 bytes (low byte -> low half) -> f16x2.  Every E4M3 value is exact
// in f16 (range 2^-9 .. 448, 4 significant bits).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  unsigned short in = static_cast<unsigned short>(two_bytes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(in));
  return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// {lo: a.lo, hi: b.lo} and {lo: a.hi, hi: b.hi}
__device__ __forceinline__ uint32_t pack_lo(uint32_t a, uint32_t b) {
  return __byte_perm(a, b, 0x5410);
}
__device__ __forceinline__ uint32_t pack_hi(uint32_t a, uint32_t b) {
  return __byte_perm(a, b, 0x7632);
}
// broadcast a half: {x.lo, x.lo} / {x.hi, x.hi}
__device__ __forceinline__ uint32_t bcast_lo(uint32_t x) {
  return __byte_perm(x, x, 0x1010);
}
__device__ __forceinline__ uint32_t bcast_hi(uint32_t x) {
  return __byte_perm(x, x, 0x3232);
}

// Transpose of an 8 x 8 matrix of 16-bit values held one row pair per lane
// (lane 4r + c holds elements (r, 2c) and (r, 2c+1)).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(r) : "r"(x));
  return r;
}

// Two f32 -> f16x2 (round to nearest even), lo from a.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

// D += A * B, m16n8k16, f16 inputs, f32 accumulators.
//   A (row-major 16x16): a[0]={A[g][2t],A[g][2t+1]}, a[1]=rows g+8,
//                        a[2]=cols 2t+8.., a[3]=rows g+8, cols 2t+8..
//   B (col-major 16x8):  b[0]={B[2t][g],B[2t+1][g]}, b[1]=rows 2t+8..
//   D (16x8):            d[0]=D[g][2t], d[1]=D[g][2t+1], d[2]/d[3]=row g+8
// with g = lane/4, t = lane%4.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4],
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32).
__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;\n" : "=h"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

}  // namespace dev

// The CTA's work unit.  With a live last_page_len the unit's kv_len is the
// request's current length: its planned whole pages plus the current length
// of the last page (a value outside [1, page_size], or a length below the
// request's query rows, sets flag 0x8 and is clamped).
__device__ __forceinline__ WorkUnit load_unit(const AttendParams& p, int idx, bool report) {
  WorkUnit u = p.units[idx];
  if (p.live_last_page_len != nullptr) {
    const int P = p.page_size;
    const int full = (u.kv_len - 1) - (u.kv_len - 1) % P;  // tokens in whole pages
    int lpl = __ldg(p.live_last_page_len + u.b);
    int len = full + lpl;
    if (lpl < 1 || lpl > P || len < u.qo_len) {
      if (report) atomicOr(p.flags, 0x8u);
      lpl = max(1, min(P, lpl));
      len = max(u.qo_len, full + lpl);
    }
    u.kv_len = len;
  }
  return u;
}
// The unit of this CTA (one unit per CTA)
__device__ __forceinline__ WorkUnit load_unit(const AttendParams& p) {
  return load_unit(p, blockIdx.x, threadIdx.x == 0);
}

// Two f32 values as two packed output elements (bf16 or f16, lo from a).
__device__ __forceinline__ uint32_t pack_out2(float a, float b, bool f16) {
  return f16 ? dev::f32x2_to_f16x2(a, b)
             : ((uint32_t)dev::f32_to_bf16_bits(a) | ((uint32_t)dev::f32_to_bf16_bits(b) << 16));
}
__device__ __forceinline__ uint16_t pack_out1(float a, bool f16) {
  return f16 ? (uint16_t)(dev::f32x2_to_f16x2(a, 0.f) & 0xFFFFu) : dev::f32_to_bf16_bits(a);
}
}  // namespace nvfp4kv
