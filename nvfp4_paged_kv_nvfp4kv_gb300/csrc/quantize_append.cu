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
#include "quantize.cuh"

namespace nvfp4kv {
namespace {

__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
  const int bpk = p.head_dim_qk / 16, bpv = p.head_dim_vo / 16;
  const int per = bpk + bpv;
  const int64_t total = static_cast<int64_t>(p.nnz) * p.num_kv_heads * per;
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
      const int64_t L = np > 0 ? static_cast<int64_t>(np - 1) * p.page_size + p.last_page_len[b] : 0;
      ok = pos < L;
      if (ok) {
        page = p.kv_indices[beg + pos / p.page_size];
        ok = page >= 0 && page < p.num_pages;
      }
    }
    if (!ok) {
      if (p.flags && blk == 0 && h == 0) atomicOr(p.flags, 0x2u);
      continue;
    }
    const int slot = pos % p.page_size;

    const float g = isv ? p.v_global_scale : p.k_global_scale;
    uint2 packed;
    const uint32_t sfb = quantize_block16(lo, hi, g, &packed);
    uint8_t* drow = isv ? p.v_data + page * p.v_sp + slot * p.v_ss + h * p.v_sh
                        : p.k_data + page * p.k_sp + slot * p.k_ss + h * p.k_sh;
    uint8_t* srow = isv ? p.v_sf + page * p.vsf_sp + slot * p.vsf_ss + h * p.vsf_sh
                        : p.k_sf + page * p.ksf_sp + slot * p.ksf_ss + h * p.ksf_sh;
    *reinterpret_cast<uint2*>(drow + 8 * jb) = packed;
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
