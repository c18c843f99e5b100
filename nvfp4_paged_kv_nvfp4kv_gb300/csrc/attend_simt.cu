// attend_simt.cu -- CUDA-core variant of the paged NVFP4 attention kernel
// (float32 FMAs, no tensor cores), sm_103a.  Same work units, page pipeline,
// masking, softmax and outputs as the tensor-core kernel (attend_tc.cu); it
// exists to measure what the tensor-core contraction buys.
//
// Per page (16 tokens) and warp:
//  * QK: lane l takes token l % 16 and half l / 16 of the head dim; the
//    codes of one 16-element block are dotted with Q in float32 and the
//    block's E4M3 scale multiplies the block sum; the two halves add by one
//    shuffle.
//  * softmax: max / sum over the 16 lanes of a row (xor 1, 2, 4, 8).
//  * PV: lane l owns Dv/32 consecutive value dims; p * scale of each token is
//    read from a per-warp scratch row, and multiplies the token's codes.
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "epilogue.cuh"
#include "stage.cuh"

namespace nvfp4kv {
namespace {

using namespace dev;

constexpr int kSimtRows = 8;

template <int DK, int DV, int WARPS, int STAGES>
struct SimtTraits : PageStage<DK, DV> {
  using S = PageStage<DK, DV>;
  static constexpr int RB = kSimtRows;
  static constexpr int PIPE_BYTES = WARPS * STAGES * S::STAGE_BYTES;
  static constexpr int COMB_BYTES = WARPS * RB * (DV + 2) * 4;
  static constexpr int MAIN_BYTES = PIPE_BYTES > COMB_BYTES ? PIPE_BYTES : COMB_BYTES;
  static constexpr int Q_BYTES = RB * DK * 4;           // float32 Q rows
  static constexpr int P_BYTES = WARPS * RB * 16 * 4;   // per-warp p * scale rows
  static constexpr int SMEM = MAIN_BYTES + Q_BYTES + P_BYTES + RB * 16;
  static constexpr int VD = DV / 32;                    // value dims per lane
  static_assert(DK % 64 == 0 && DV % 64 == 0, "head dims");
};

template <int DK, int DV, int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32) attend_simt_kernel(const AttendParams p) {
  using T = SimtTraits<DK, DV, WARPS, STAGES>;
  using S = typename T::S;
  constexpr int RB = T::RB;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* pipe = smem;
  float* sQ = reinterpret_cast<float*>(smem + T::MAIN_BYTES);
  float* sP = reinterpret_cast<float*>(smem + T::MAIN_BYTES + T::Q_BYTES);
  int* sRowLim = reinterpret_cast<int*>(smem + T::MAIN_BYTES + T::Q_BYTES + T::P_BYTES);

  const WorkUnit u = load_unit(p);
  const int G = p.group;
  const int R = G * u.qo_len;
  const int row0 = blockIdx.y * RB;
  if (row0 >= R) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int idx = tid; idx < RB * DK; idx += WARPS * 32) {
    const int rr = idx / DK, d = idx % DK, r = row0 + rr;
    float v = 0.f;
    if (r < R) {
      const int i = r / G, gh = r % G;
      v = bf16_bits_to_f32(p.q[(int64_t)(u.qo_begin + i) * p.q_stride_tok +
                               (int64_t)(u.h_kv * G + gh) * p.q_stride_head + d]);
    }
    sQ[idx] = v;
  }
  if (tid < RB) {
    const int r = row0 + tid;
    sRowLim[tid] = r >= R ? -1
                          : (p.causal ? (u.kv_len - u.qo_len + r / G) : (u.kv_len - 1));
  }
  __syncthreads();
  int lim[RB];
  int min_lim = INT32_MAX;
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    lim[r] = sRowLim[r];
    if (lim[r] >= 0) min_lim = min(min_lim, lim[r]);
  }

  float m_run[RB], l_run[RB], o[RB][T::VD];
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    m_run[r] = -INFINITY;
    l_run[r] = 0.f;
#pragma unroll
    for (int k = 0; k < T::VD; ++k) o[r][k] = 0.f;
  }

  uint8_t* wpipe = pipe + warp * STAGES * S::STAGE_BYTES;
  float* wP = sP + warp * RB * 16;
  // tiles of 16 tokens: one page each at page size 16, sixteen 1-token pages
  // at page size 1 (lane r then copies through the id of row r)
  const bool rows = p.page_size == 1;
  const int ntiles = rows ? (u.num_pages + 15) / 16 : u.num_pages;
  const int npw = ntiles > warp ? (ntiles - warp + WARPS - 1) / WARPS : 0;
  const int32_t* pidx = p.kv_indices + u.page_begin;
  auto load_page = [&](int i) {
    int32_t pid;
    if (rows) {
      const int pg = 16 * (warp + i * WARPS) + (lane & 15);
      pid = pg < u.num_pages ? pidx[pg] : 0;
    } else {
      pid = pidx[warp + i * WARPS];
    }
    if (pid < 0 || pid >= p.cache.num_pages) {
      atomicOr(p.flags, 0x1u);
      pid = 0;
    }
    uint8_t* st = wpipe + (i % STAGES) * S::STAGE_BYTES;
    if (rows)
      issue_tile_rows<S>(st, p.cache, pid, u.h_kv, lane);
    else
      issue_page<S>(st, p.cache, pid, u.h_kv, lane);
  };
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < npw) load_page(s);
    cp_async_commit();
  }

  const int tok = lane & 15, half = lane >> 4;
  for (int i = 0; i < npw; ++i) {
    if (i + STAGES - 1 < npw) load_page(i + STAGES - 1);
    cp_async_commit();
    cp_async_wait<STAGES - 1>();
    __syncwarp();
    const uint8_t* st = wpipe + (i % STAGES) * S::STAGE_BYTES;
    const int tok0 = u.tok_begin + (warp + i * WARPS) * 16;

    // ---- scores of token `tok`, this lane's half of the head dim ---------
    float sc[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) sc[r] = 0.f;
#pragma unroll
    for (int c = 0; c < DK / 64; ++c) {       // 16-byte chunks of the half
      const int ch = half * (DK / 64) + c;    // chunk index in the row
      const uint4 v = *reinterpret_cast<const uint4*>(st + tok * S::KROW +
                                                      S::k_pos(tok, ch) * 16);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      const uint32_t sfp = *reinterpret_cast<const uint16_t*>(
          st + S::OFF_KSF + tok * S::KSFROW + 2 * ch);
      const uint32_t sf2 = e4m3x2_to_f16x2(sfp);
      const float2 sfs = __half22float2(*reinterpret_cast<const __half2*>(&sf2));
#pragma unroll
      for (int bl = 0; bl < 2; ++bl) {        // two 16-element blocks
        float part[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) part[r] = 0.f;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t h[4];
          e2m1x8_to_f16x8(w[2 * bl + q], h);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 cv = __half22float2(*reinterpret_cast<const __half2*>(&h[j]));
            const int d = 32 * ch + 16 * bl + 8 * q + 2 * j;
#pragma unroll
            for (int r = 0; r < RB; ++r) {
              const float2 qv = *reinterpret_cast<const float2*>(sQ + r * DK + d);
              part[r] = fmaf(qv.x, cv.x, fmaf(qv.y, cv.y, part[r]));
            }
          }
        }
        const float s_blk = bl ? sfs.y : sfs.x;
#pragma unroll
        for (int r = 0; r < RB; ++r) sc[r] = fmaf(s_blk, part[r], sc[r]);
      }
    }
    const bool need_mask = tok0 + 15 > min_lim;
    float pv[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      float x = (sc[r] + __shfl_xor_sync(0xffffffffu, sc[r], 16)) * p.qk_scale_log2;
      if (need_mask && tok0 + tok > lim[r]) x = -INFINITY;
      float mx = x;
#pragma unroll
      for (int o2 = 1; o2 < 16; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
      const float m_new = fmaxf(m_run[r], mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float corr = ex2(m_run[r] - m_use);
      m_run[r] = m_new;
      pv[r] = ex2(x - m_use);
      l_run[r] = l_run[r] * corr + (half == 0 ? pv[r] : 0.f);
      if (corr != 1.f) {  // warp-uniform: m is the same in every lane
#pragma unroll
        for (int k = 0; k < T::VD; ++k) o[r][k] *= corr;
      }
    }
    // p * (V block scale of the token for this lane's dims): lanes 0..15
    // write token `tok`'s factor; the lane's dims lie in one block
    {
      const int valid = u.kv_len - tok0;
      const int blk = (lane * T::VD) / 16;
      // every lane needs the scales of all 16 tokens for its block: the
      // scale is applied by the reader, p is written once per (row, token)
      if (half == 0) {
#pragma unroll
        for (int r = 0; r < RB; ++r) wP[r * 16 + tok] = pv[r];
      }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        uint32_t code2;
        if constexpr (T::VD == 2) {
          code2 = st[S::OFF_V + j * S::VROW + lane];
        } else if constexpr (T::VD == 4) {
          code2 = *reinterpret_cast<const uint16_t*>(st + S::OFF_V + j * S::VROW + 2 * lane);
        } else {
          code2 = *reinterpret_cast<const uint32_t*>(st + S::OFF_V + j * S::VROW + 4 * lane);
        }
        float s = __half2float(__ushort_as_half(static_cast<unsigned short>(
            e4m3x2_to_f16x2(st[S::OFF_VSF + j * S::VSFROW + blk]) & 0xFFFFu)));
        if (j >= valid) s = 0.f;  // slots past kv_len may hold any bytes
        uint32_t h[4];
        e2m1x8_to_f16x8(code2, h);
        float vv[T::VD];
#pragma unroll
        for (int k = 0; k < T::VD / 2; ++k) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[k]));
          vv[2 * k] = f.x * s;
          vv[2 * k + 1] = f.y * s;
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          const float pj = wP[r * 16 + j];
#pragma unroll
          for (int k = 0; k < T::VD; ++k) o[r][k] = fmaf(pj, vv[k], o[r][k]);
        }
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();

  // ---- combine the warps ------------------------------------------------
#pragma unroll
  for (int r = 0; r < RB; ++r)
#pragma unroll
    for (int o2 = 1; o2 < 16; o2 <<= 1) l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], o2);
  __syncthreads();
  float* sO = reinterpret_cast<float*>(pipe);
  float* sM = sO + WARPS * RB * DV;
  float* sL = sM + WARPS * RB;
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      sM[warp * RB + r] = m_run[r];
      sL[warp * RB + r] = l_run[r];
    }
  }
#pragma unroll
  for (int r = 0; r < RB; ++r)
#pragma unroll
    for (int k = 0; k < T::VD; ++k) sO[(warp * RB + r) * DV + lane * T::VD + k] = o[r][k];
  __syncthreads();
  finish_unit<RB, DV, WARPS>(p, u, row0, R, sM, sL, sO,
                            reinterpret_cast<float*>(sRowLim));
}

template <int DK, int DV>
bool make_simt(AttendConfig* cfg) {
  constexpr int WARPS = 4, STAGES = DK >= 512 ? 3 : 4;
  using T = SimtTraits<DK, DV, WARPS, STAGES>;
  cfg->kind = kKernelCudaCore;
  cfg->dk = DK;
  cfg->dv = DV;
  cfg->rows = T::RB;
  cfg->warps = WARPS;
  cfg->smem_bytes = T::SMEM;
  cfg->func = reinterpret_cast<const void*>(attend_simt_kernel<DK, DV, WARPS, STAGES>);
  return true;
}

}  // namespace

bool attend_config_simt(int dk, int dv, int /*rows*/, AttendConfig* cfg) {
#define NVFP4KV_SIMT_CASE(DK_, DV_) \
  if (dk == DK_ && dv == DV_) return make_simt<DK_, DV_>(cfg);
  NVFP4KV_SIMT_CASE(64, 64)
  NVFP4KV_SIMT_CASE(128, 128)
  NVFP4KV_SIMT_CASE(256, 256)
  NVFP4KV_SIMT_CASE(256, 128)
  NVFP4KV_SIMT_CASE(512, 256)
#undef NVFP4KV_SIMT_CASE
  return false;
}

}  // namespace nvfp4kv
