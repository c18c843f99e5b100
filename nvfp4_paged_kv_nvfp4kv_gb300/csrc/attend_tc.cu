// attend_tc.cu -- paged NVFP4 decode / extend attention on the tensor cores
// (mma.sync m16n8k16, f16 operands, f32 accumulators), sm_103a.
//
// What it computes (page "Support NVFP4 KV cache decode on SM120": packed
// e2m1 K/V with per-16 E4M3 scale caches, unpacked and scaled before the
// QK and PV products; page "fix(attention): correct SM120 NVFP4
// qk_correction layout, row-sum reduction, and lse": row reductions over
// exactly the lanes that own a row, lse written as natural-log sum-exp):
//   s_j = sm_scale * sum_d q_d * k_hat_{j,d},  online softmax over the
//   visible keys, o = sum_j p_j v_hat_j / sum_j p_j, lse = ln sum_j exp s_j.
//
// Design (one work unit = (request, kv head, chunk of pages) x a block of up
// to 16 query rows; the G heads of the group times the query positions):
//  * Each warp owns every WARPS-th page of the chunk and streams it through
//    its own STAGES-deep cp.async ring in shared memory (16-byte copies of the
//    packed K/V rows and the scale rows; any byte strides, NHD or HND).
//  * QK^T: S = Q . K_hat^T with M = query rows, N = 8 tokens, K = 16 dims.
//    The B operand wants two adjacent dims of one token per register, which
//    is exactly one packed byte: cvt.rn.f16x2.e2m1x2 then one f16x2 multiply
//    by the block scale (code * E4M3 scale is exact in f16).  The contraction
//    dims are permuted so each lane reads 16 contiguous bytes of a token row;
//    Q is permuted identically when its fragments are built.
//  * Global scales stay out of the f16 operands: g_K is folded into the f32
//    score scale, g_V into the epilogue.  Q is multiplied by a power of two
//    per row (exact) so its bf16 values land in f16's normal range.
//  * PV: O^T = V_hat^T . P^T with M = 16 value dims, N = 8 query rows,
//    K = 16 tokens; the S accumulator layout is already the P^T B-fragment
//    layout, so P never leaves registers.  The A operand needs pairs of
//    tokens per dim: two converted bytes are interleaved with one byte_perm
//    each, and multiplied by the pair of per-token scales.
//  * With a single block of at most 8 query rows (the usual decode shape) the
//    score product is taken transposed, S^T = K_hat . Q^T with M = 16 tokens
//    and N = 8 rows, so that every tensor-core slot holds a real token; the
//    two f16 P^T fragments are turned into the PV B operand with
//    movmatrix.trans, and the row maximum is raised lazily (only when a score
//    exceeds the running maximum by more than 2^8, decided by one warp vote
//    per page).
//  * Online softmax in the log2 domain; the max and sum reductions run over
//    the lanes that hold one row.  Warps combine through shared memory; the
//    unit writes bf16 out + lse, or an f32 partial state + lse for the merge
//    when the plan split the request.
//
// FP4 query and probabilities (kernel 4; page "fix(attention): correct SM120
// NVFP4 qk_correction layout, row-sum reduction, and lse", description: the
// SageAttention3-style NVFP4 attention quantises Q and P to FP4 and its row
// sum carries the factor of the FP4 P quantisation, which lse drops), one
// block of <= 8 rows, two launches of this kernel:
//  * MODE 1 quantises each 16-dim block of Q to NVFP4 (global scale 1, the
//    cache's exact recipe), takes the scores like MODE 0 and stores each
//    unit's row maxima (its page copies skip V; no PV);
//  * MODE 2 reads the maxima of all units of the request, takes p = 2^(x -
//    m) (m the row's maximum over all its keys), and per row and 16-token
//    tile quantises 2688 p to NVFP4: E4M3 scale RN(max / 6), e2m1 codes by
//    exact comparisons with midpoint x scale; code x scale is exact in f16,
//    so the mma.sync PV product takes exactly the block-scaled FP4 operand.
//    The row sum is that of the unquantised p times 2688, the maximum
//    m - log2(2688), so the common epilogue writes o = sum P_hat v_hat /
//    (2688 sum p) and lse = ln sum exp(s).

#include <cfloat>
#include <cstdint>
#include <type_traits>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "append_fused.cuh"
#include "internal.h"
#include "quantize.cuh"
#include "epilogue.cuh"
#include "stage.cuh"

namespace nvfp4kv {
namespace {

using namespace dev;

// Q fragments of the small shapes live in registers (1) or are re-read from
// shared memory at every k-step (0).
#ifndef NVFP4KV_TC_QREGS
#define NVFP4KV_TC_QREGS 1
#endif

template <int DK, int DV, int NT, int WARPS, int STAGES>
struct TcTraits : PageStage<DK, DV> {
  using S = PageStage<DK, DV>;
  static constexpr int RB = 8 * NT;                  // query rows per CTA
  static constexpr int CB = (DK / 8 < 16) ? DK / 8 : 16;  // K bytes per lane chunk
  static constexpr int NCH = (DK / 8) / CB;          // K chunks per lane
  static constexpr int KSTEPS = DK / 16;
  static constexpr int KS_PER_CH = CB / 2;
  static constexpr int VC = DV / 16;                 // V bytes per lane per token
  static constexpr int MT = DV / 16;                 // PV m-tiles
  static constexpr int PIPE_BYTES = WARPS * STAGES * S::STAGE_BYTES;
  static constexpr int COMB_BYTES = WARPS * RB * (DV + 2) * 4;
  static constexpr int MAIN_BYTES = PIPE_BYTES > COMB_BYTES ? PIPE_BYTES : COMB_BYTES;
  static constexpr int QROW = DK + 8;                // f16 elements, padded
  static constexpr int Q_BYTES = RB * QROW * 2;
  static constexpr int SMEM = MAIN_BYTES + Q_BYTES + RB * 16;
  static constexpr bool Q_IN_REGS = NVFP4KV_TC_QREGS && KSTEPS * 2 * NT <= 32;
  static_assert(S::VC == VC, "V lane chunk");
};

// Resident CTAs per SM asked of the register allocator for the small decode
// shapes (D <= 128, 8 rows); the larger shapes keep what they need.
#ifndef NVFP4KV_TC_MINB
#define NVFP4KV_TC_MINB 4
#endif
template <int DK, int DV, int NT>
constexpr int tc_min_blocks() {
  return (DK <= 128 && DV <= 128 && NT == 1) ? NVFP4KV_TC_MINB : 1;
}

// One row block: the running maximum is raised only when a score exceeds it
// by more than this (log2 domain), so p <= 2^kRaiseLog2 fits f16.
constexpr float kRaiseLog2 = 8.f;

// FP4 query and probabilities (MODE 1: the row-maximum pass, MODE 2: the
// attention pass).  p is scaled by the E4M3 maximum times the e2m1 maximum
// before its NVFP4 quantisation, so a block holding the row's maximum gets
// the scale 448.
constexpr float kPScale = 448.f * 6.f;
constexpr float kLog2PScale = 11.392317422778760f;  // log2(2688)

// e2m1 code (0..7) of x / sc, x >= 0, round to nearest, ties to the even
// code, saturating at 6: x is compared with the midpoints between adjacent
// values times the scale (th[k] = {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5}[k] *
// sc, exact products), and a tie goes up only where the upper code is even.
__device__ __forceinline__ uint32_t e2m1_code_of(float x, const float (&th)[7]) {
  return (uint32_t)(x > th[0]) + (uint32_t)(x >= th[1]) + (uint32_t)(x > th[2]) +
         (uint32_t)(x >= th[3]) + (uint32_t)(x > th[4]) + (uint32_t)(x >= th[5]) +
         (uint32_t)(x > th[6]);
}

template <int DK, int DV, int NT, int WARPS, int STAGES, int MODE>
__global__ void __launch_bounds__(WARPS * 32, (tc_min_blocks<DK, DV, NT>()))
    attend_tc_kernel(const AttendParams p) {
  using T = TcTraits<DK, DV, NT, WARPS, STAGES>;
  static_assert(MODE == 0 || NT == 1, "FP4 query and probabilities: one row block");
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* pipe = smem;
  uint16_t* sQ = reinterpret_cast<uint16_t*>(smem + T::MAIN_BYTES);
  float* sRowF = reinterpret_cast<float*>(smem + T::MAIN_BYTES + T::Q_BYTES);
  int* sRowLim = reinterpret_cast<int*>(sRowF + T::RB);

  const WorkUnit u = load_unit(p);
  const int G = p.group;
  const int R = G * u.qo_len;
  const int row0 = blockIdx.y * T::RB;
  if (row0 >= R) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  // ---- Q rows of this CTA: one 16-byte load per thread per chunk of 8
  // elements, issued now and consumed after the pipeline has started ------
  constexpr int QCH = T::RB * DK / 8;                      // 8-element chunks
  constexpr int QPT = (QCH + WARPS * 32 - 1) / (WARPS * 32);
  uint4 qv[QPT];
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int ci = tid + k * WARPS * 32;
    const int rr = ci / (DK / 8), r = row0 + rr;
    qv[k] = make_uint4(0u, 0u, 0u, 0u);
    if (ci < QCH && r < R) {
      const int i = r / G, gh = r % G;
      qv[k] = *reinterpret_cast<const uint4*>(p.q + (int64_t)(u.qo_begin + i) * p.q_stride_tok +
                                              (int64_t)(u.h_kv * G + gh) * p.q_stride_head +
                                              (ci % (DK / 8)) * 8);
    }
  }
  if (tid < T::RB) reinterpret_cast<int*>(sRowF)[tid] = 0;  // per-row amax bits

  // ---- fused append: quantise the step's new tokens of this kv head that
  // fall in this unit's pages and store them before any copy reads them.
  // When none of them lies in the pages the prologue copies, the work runs
  // after the prologue's copies are issued (its latency hides behind theirs).
  int new_lo = 0, new_hi = 0;
  if (p.new_k != nullptr) {
    new_lo = max(u.kv_len - u.qo_len, u.tok_begin);
    new_hi = min(u.kv_len, u.tok_begin + p.page_size * u.num_pages);
  }
  auto append_new = [&]() {
    append_unit_tokens<DK, DV>(p, u, new_lo, new_hi, tid, WARPS * 32);
  };
  // the prologue copies relative pages [0, WARPS * (STAGES - 1))
  const bool append_early =
      new_lo < new_hi && (new_lo - u.tok_begin) / 16 < WARPS * (STAGES - 1);
  if (append_early) {
    append_new();
    __syncthreads();
  }

  // ---- start the page pipeline: the first pages' copies are in flight
  // while Q is prepared ---------------------------------------------------
  uint8_t* wpipe = pipe + warp * STAGES * T::STAGE_BYTES;
  // tiles of 16 tokens: one page each at page size 16, sixteen 1-token pages
  // at page size 1
  const bool rows = p.page_size == 1;
  const int ntiles = rows ? (u.num_pages + 15) / 16 : u.num_pages;
  const int npw = ntiles > warp ? (ntiles - warp + WARPS - 1) / WARPS : 0;
  const int32_t* pidx = p.kv_indices + u.page_begin;

  // page ids are read one iteration before their copies are issued, so the
  // address computation never waits on a global load (page size 1: lane r
  // reads the id of row r; a row past the unit's pages reads page 0)
  auto page_id = [&](int i) -> int32_t {
    if (i >= npw) return 0;
    if (!rows) return pidx[warp + i * WARPS];
    const int pg = 16 * (warp + i * WARPS) + (lane & 15);
    return pg < u.num_pages ? pidx[pg] : 0;
  };
  auto load_page = [&](int i, int32_t pid) {
    if (pid < 0 || pid >= p.cache.num_pages) {
      atomicOr(p.flags, 0x1u);
      pid = 0;
    }
    uint8_t* st = wpipe + (i % STAGES) * T::STAGE_BYTES;
    // the row-maximum pass (MODE 1) reads no V
    if (rows)
      issue_tile_rows<typename T::S, MODE != 1>(st, p.cache, pid, u.h_kv, lane);
    else
      issue_page<typename T::S, MODE != 1>(st, p.cache, pid, u.h_kv, lane);
  };

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < npw) load_page(s, page_id(s));
    cp_async_commit();
  }
  int32_t next_pid = page_id(STAGES - 1);

  __syncthreads();  // the amax slots are zeroed; late appended tokens stored
  if constexpr (MODE == 0) {
    // ---- Q: per-row power-of-two prescale into f16, row limits ----------
    // amax of each row (non-negative floats order like their bit patterns)
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
      const int ci = tid + k * WARPS * 32;
      if (ci >= QCH) continue;
      const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
      float am = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        am = fmaxf(am, fmaxf(fabsf(bf16_bits_to_f32(w[j] & 0xFFFFu)),
                             fabsf(bf16_bits_to_f32(w[j] >> 16))));
      atomicMax(reinterpret_cast<int*>(sRowF) + ci / (DK / 8), __float_as_int(am));
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
      const int ci = tid + k * WARPS * 32;
      if (ci >= QCH) continue;
      const int rr = ci / (DK / 8);
      const float amax = __int_as_float(reinterpret_cast<const int*>(sRowF)[rr]);
      // e such that amax * 2^e lies in [2^14, 2^15)
      int e = 0;
      if (amax > 0.f) e = 14 - (int)((__float_as_uint(amax) >> 23) & 0xFF) + 127;
      e = max(-120, min(120, e));
      const float up = __uint_as_float((uint32_t)(127 + e) << 23);
      const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
      uint32_t h[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        h[j] = f32x2_to_f16x2(bf16_bits_to_f32(w[j] & 0xFFFFu) * up,
                              bf16_bits_to_f32(w[j] >> 16) * up);
      *reinterpret_cast<uint4*>(sQ + rr * T::QROW + (ci % (DK / 8)) * 8) =
          make_uint4(h[0], h[1], h[2], h[3]);
      if (ci % (DK / 8) == 0) {
        const int r = row0 + rr;
        sRowLim[rr] = r >= R ? -1 : (p.causal ? (u.kv_len - u.qo_len + r / G) : (u.kv_len - 1));
        // the row factor replaces the amax slot once every thread has read it
        qv[k].x = __float_as_uint(r >= R ? 0.f
                                         : p.qk_scale_log2 *
                                               __uint_as_float((uint32_t)(127 - e) << 23));
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
      const int ci = tid + k * WARPS * 32;
      if (ci < QCH && ci % (DK / 8) == 0) sRowF[ci / (DK / 8)] = __uint_as_float(qv[k].x);
    }
    __syncthreads();
  } else {
    // ---- Q quantised to NVFP4 (global scale 1) with the cache's exact
    // recipe, used as its f16 values (code x E4M3 scale is exact in f16).
    // The two 8-dim chunks of a 16-dim block sit in lanes 2m and 2m + 1,
    // which trade halves so that each quantises the whole block.
    static_assert((DK / 8) % 2 == 0 && (WARPS * 32) % 2 == 0, "block pairs");
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
      const int ci = tid + k * WARPS * 32;
      const uint4 mine = qv[k];
      uint4 other;
      other.x = __shfl_xor_sync(0xffffffffu, mine.x, 1);
      other.y = __shfl_xor_sync(0xffffffffu, mine.y, 1);
      other.z = __shfl_xor_sync(0xffffffffu, mine.z, 1);
      other.w = __shfl_xor_sync(0xffffffffu, mine.w, 1);
      const bool odd = ci & 1;
      uint2 packed;
      const uint32_t sfb = quantize_block16(odd ? other : mine, odd ? mine : other, 1.0f, &packed);
      const uint32_t sc = bcast_lo(e4m3x2_to_f16x2(sfb));
      uint32_t h[4];
      e2m1x8_to_f16x8(odd ? packed.y : packed.x, h);
      if (ci >= QCH) continue;
      const int rr = ci / (DK / 8);
#pragma unroll
      for (int j = 0; j < 4; ++j) h[j] = hmul2(h[j], sc);
      *reinterpret_cast<uint4*>(sQ + rr * T::QROW + (ci % (DK / 8)) * 8) =
          make_uint4(h[0], h[1], h[2], h[3]);
      if (ci % (DK / 8) == 0) {
        const int r = row0 + rr;
        sRowLim[rr] = r >= R ? -1 : (p.causal ? (u.kv_len - u.qo_len + r / G) : (u.kv_len - 1));
        sRowF[rr] = r >= R ? 0.f : p.qk_scale_log2;
      }
    }
    __syncthreads();
  }

  // per-lane row data: rows g (half 0) and g + 8 (half 1)
  float rowf[NT];
  int rowlim[NT];
  int min_lim = INT32_MAX;
#pragma unroll
  for (int hf = 0; hf < NT; ++hf) {
    rowf[hf] = sRowF[8 * hf + g];
    rowlim[hf] = sRowLim[8 * hf + g];
  }
  for (int rr = 0; rr < T::RB; ++rr)
    if (sRowLim[rr] >= 0) min_lim = min(min_lim, sRowLim[rr]);
  // one row block (NT == 1): this lane's query rows 2t and 2t+1, score
  // factor f, -m_use, raise threshold (-inf until the row has a maximum,
  // +inf for padding rows), causal limit, running max and partial sum
  float f2[2], nm2[2], thr2[2], mrow[2], lrow[2];
  int lim2[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    f2[k] = sRowF[(2 * t + k) % T::RB];
    lim2[k] = sRowLim[(2 * t + k) % T::RB];
    nm2[k] = 0.f;
    thr2[k] = lim2[k] >= 0 ? -INFINITY : INFINITY;
    mrow[k] = -INFINITY;
    lrow[k] = 0.f;
  }

  // Q fragments: k-step kk of chunk c = kk / KS_PER_CH, step m within it,
  // covers the 4 consecutive dims starting at 2*(4c+t)*CB + 4m.
  auto q_frag = [&](int kk, uint32_t (&a)[4]) {
    const int c = kk / T::KS_PER_CH, m = kk % T::KS_PER_CH;
    const int d0 = 2 * (4 * c + t) * T::CB + 4 * m;
    const uint2 lo = *reinterpret_cast<const uint2*>(sQ + g * T::QROW + d0);
    a[0] = lo.x;
    a[2] = lo.y;
    if constexpr (NT == 2) {
      const uint2 hi = *reinterpret_cast<const uint2*>(sQ + (g + 8) * T::QROW + d0);
      a[1] = hi.x;
      a[3] = hi.y;
    } else {
      a[1] = 0u;
      a[3] = 0u;
    }
  };
  uint32_t qreg[T::Q_IN_REGS ? T::KSTEPS : 1][4];
  if constexpr (T::Q_IN_REGS) {
#pragma unroll
    for (int kk = 0; kk < T::KSTEPS; ++kk) q_frag(kk, qreg[kk]);
  }

  // FP4 query and probabilities: MODE 1 keeps this lane's maxima of its rows'
  // scores; MODE 2 reads each row's maximum over every unit of its request
  // (written by MODE 1 in the previous launch)
  float mfix[2] = {-INFINITY, -INFINITY};
  if constexpr (MODE == 2) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int r = row0 + 2 * t + k;
      if (lim2[k] >= 0) {
        const float* rm = p.row_max + ((int64_t)(u.qo_begin + r / G) * p.num_qo_heads +
                                       u.h_kv * G + r % G) * p.row_max_splits;
        for (int sp = 0; sp < u.num_splits; ++sp) mfix[k] = fmaxf(mfix[k], rm[sp]);
      }
    }
  }

  // ---- per-warp state --------------------------------------------------
  float m_run[NT], l_run[NT];
  float oacc[T::MT][NT][4];
#pragma unroll
  for (int hf = 0; hf < NT; ++hf) {
    m_run[hf] = -INFINITY;
    l_run[hf] = 0.f;
  }
#pragma unroll
  for (int mt = 0; mt < T::MT; ++mt)
#pragma unroll
    for (int nq = 0; nq < NT; ++nq)
#pragma unroll
      for (int k = 0; k < 4; ++k) oacc[mt][nq][k] = 0.f;


  // new tokens on later pages: each warp stores those of its own pages just
  // before its loop; only this warp's later copies read them (the stores are
  // fenced and the warp synchronised before any of them is issued)
  if (new_lo < new_hi && !append_early) {
    append_unit_tokens<DK, DV>(p, u, new_lo, new_hi, lane, 32, warp, WARPS);
    __syncwarp();
  }

  for (int i = 0; i < npw; ++i) {
    if (i + STAGES - 1 < npw) load_page(i + STAGES - 1, next_pid);
    next_pid = page_id(i + STAGES);
    cp_async_commit();
    cp_async_wait<STAGES - 1>();
    __syncwarp();
    const uint8_t* st = wpipe + (i % STAGES) * T::STAGE_BYTES;
    const int tok0 = u.tok_begin + (warp + i * WARPS) * 16;
    // V rows and scales of this page, loaded before the score product
    const uint8_t* vrow = st + T::OFF_V + g * T::VC;
    const int tk[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
    constexpr int VW = T::VC / 4 > 0 ? T::VC / 4 : 1;  // 32-bit words per lane
    uint32_t vw[4][VW];
#pragma unroll
    for (int k = 0; k < (MODE == 1 ? 0 : 4); ++k) {
      const uint8_t* src = vrow + tk[k] * T::VROW;
      if constexpr (T::VC == 16) {
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        vw[k][0] = v.x; vw[k][1] = v.y; vw[k][2] = v.z; vw[k][3] = v.w;
      } else if constexpr (T::VC == 8) {
        const uint2 v = *reinterpret_cast<const uint2*>(src);
        vw[k][0] = v.x; vw[k][1] = v.y;
      } else {
        vw[k][0] = *reinterpret_cast<const uint32_t*>(src);
      }
    }
    // per-token scale pairs for each scale block the lane's bytes touch
    // Slots past kv_len on the request's last page hold whatever the pool
    // held (possibly a NaN scale byte); their p is 0, but 0 * NaN would
    // still poison the product, so their V scales are forced to 0.
    const int valid = u.kv_len - tok0;  // tokens of this page that exist
    constexpr int NBL = (T::VC * 2 + 15) / 16;
    uint32_t sA[NBL], sB[NBL];
#pragma unroll
    for (int bl = 0; bl < (MODE == 1 ? 0 : NBL); ++bl) {
      const int blk = (g * T::VC * 2) / 16 + bl;
      const uint8_t* sfs = st + T::OFF_VSF + blk;
      uint32_t s0 = sfs[tk[0] * T::VSFROW], s1 = sfs[tk[1] * T::VSFROW];
      uint32_t s2 = sfs[tk[2] * T::VSFROW], s3 = sfs[tk[3] * T::VSFROW];
      if (valid < 16) {
        if (tk[0] >= valid) s0 = 0;
        if (tk[1] >= valid) s1 = 0;
        if (tk[2] >= valid) s2 = 0;
        if (tk[3] >= valid) s3 = 0;
      }
      sA[bl] = e4m3x2_to_f16x2(s0 | (s1 << 8));
      sB[bl] = e4m3x2_to_f16x2(s2 | (s3 << 8));
    }

    uint32_t pfrag[NT][2];
    // K row `row` (a token of the page), 16-byte chunk ch of this lane
    auto krow = [&](int row, int ch, uint32_t (&w)[T::CB / 4], uint32_t& sc0, uint32_t& sc1) {
      if constexpr (T::CB == 16) {
        const int pos = T::S::k_pos(row, ch);
        const uint4 v = *reinterpret_cast<const uint4*>(st + row * T::KROW + pos * 16);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
        const uint32_t sfp = *reinterpret_cast<const uint16_t*>(
            st + T::OFF_KSF + row * T::KSFROW + 2 * ch);
        const uint32_t s2 = e4m3x2_to_f16x2(sfp);
        sc0 = bcast_lo(s2);
        sc1 = bcast_hi(s2);
      } else {
        const uint2 v = *reinterpret_cast<const uint2*>(st + row * T::KROW + ch * 8);
        w[0] = v.x; w[1] = v.y;
        const uint32_t sfb = st[T::OFF_KSF + row * T::KSFROW + ch];
        sc0 = bcast_lo(e4m3x2_to_f16x2(sfb));
        sc1 = sc0;
      }
    };
    if constexpr (NT == 1) {
      // ---- S^T = K_hat Q^T: tokens g, g+8 (M = 16) x query rows (N = 8) --
      // A = K_hat (the two token rows this lane reads), B = the Q rows'
      // fragments; two accumulators (alternate k-steps) halve the chain
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < T::NCH; ++c) {
        const int ch = 4 * c + t;
        uint32_t wg[T::CB / 4], w8[T::CB / 4], sg0, sg1, s80, s81;
        krow(g, ch, wg, sg0, sg1);
        krow(8 + g, ch, w8, s80, s81);
#pragma unroll
        for (int q = 0; q < T::CB / 4; ++q) {
          uint32_t hg[4], h8[4];
          e2m1x8_to_f16x8(wg[q], hg);
          e2m1x8_to_f16x8(w8[q], h8);
          const bool hi = T::CB == 16 && q >= 2;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            hg[j] = hmul2(hg[j], hi ? sg1 : sg0);
            h8[j] = hmul2(h8[j], hi ? s81 : s80);
          }
          const int kk = c * T::KS_PER_CH + 2 * q;
          uint32_t b0[4], b1[4];
          if constexpr (T::Q_IN_REGS) {
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              b0[x] = qreg[kk][x];
              b1[x] = qreg[kk + 1][x];
            }
          } else {
            q_frag(kk, b0);
            q_frag(kk + 1, b1);
          }
          const uint32_t a0[4] = {hg[0], h8[0], hg[1], h8[1]};
          const uint32_t a1[4] = {hg[2], h8[2], hg[3], h8[3]};
          mma_16816(sa, a0, b0[0], b0[2]);
          mma_16816(sb, a1, b1[0], b1[2]);
        }
      }
      // ---- softmax with a lazily raised maximum (log2 domain) -----------
      // x[0..3] = tokens g, g, g+8, g+8 x rows 2t, 2t+1, 2t, 2t+1
      float x[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) x[k] = fmaf(sa[k] + sb[k], f2[k & 1], nm2[k & 1]);
      if (tok0 + 15 > min_lim) {
        const int ta = tok0 + g, tb = tok0 + g + 8;
        if (ta > lim2[0]) x[0] = -INFINITY;
        if (ta > lim2[1]) x[1] = -INFINITY;
        if (tb > lim2[0]) x[2] = -INFINITY;
        if (tb > lim2[1]) x[3] = -INFINITY;
      }
      if constexpr (MODE == 1) {
        // the row-maximum pass: this lane's maxima of rows 2t, 2t+1
        mfix[0] = fmaxf(mfix[0], fmaxf(x[0], x[2]));
        mfix[1] = fmaxf(mfix[1], fmaxf(x[1], x[3]));
      } else if constexpr (MODE == 2) {
        // p against the row's maximum over all its keys, scaled by 448 * 6;
        // per row, the tile's 16 values (2 in each of the 8 lanes of the same
        // t) share an E4M3 scale RN(max / 6) and each becomes an e2m1 value
        // times it (masked keys have p = 0)
        float pp[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          pp[k] = mfix[k & 1] == -INFINITY ? 0.f : ex2(x[k] - mfix[k & 1]);
        lrow[0] += pp[0] + pp[2];
        lrow[1] += pp[1] + pp[3];
        float bm[2] = {fmaxf(pp[0], pp[2]) * kPScale, fmaxf(pp[1], pp[3]) * kPScale};
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          bm[0] = fmaxf(bm[0], __shfl_xor_sync(0xffffffffu, bm[0], o));
          bm[1] = fmaxf(bm[1], __shfl_xor_sync(0xffffffffu, bm[1], o));
        }
        unsigned short sc8;  // E4M3 scales: row 2t low byte, row 2t + 1 high
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n"
            : "=h"(sc8) : "f"(__fdiv_rn(bm[1], 6.f)), "f"(__fdiv_rn(bm[0], 6.f)));
        const uint32_t sch = e4m3x2_to_f16x2(sc8);
        constexpr float kMid[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.f};
        uint32_t code[4];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const float scf =
              __half2float(__ushort_as_half((unsigned short)(k ? sch >> 16 : sch & 0xFFFFu)));
          float th[7];
#pragma unroll
          for (int m = 0; m < 7; ++m) th[m] = kMid[m] * scf;
          code[k] = scf > 0.f ? e2m1_code_of(pp[k] * kPScale, th) : 0u;
          code[k + 2] = scf > 0.f ? e2m1_code_of(pp[k + 2] * kPScale, th) : 0u;
        }
        // e2m1 value x E4M3 scale is exact in f16 (at most 2688)
        pfrag[0][0] = movmatrix_trans(hmul2(e2m1x2_byte_to_f16x2<0>(code[0] | code[1] << 4), sch));
        pfrag[0][1] = movmatrix_trans(hmul2(e2m1x2_byte_to_f16x2<0>(code[2] | code[3] << 4), sch));
      } else {
        const bool trig = (x[0] > thr2[0]) | (x[2] > thr2[0]) | (x[1] > thr2[1]) | (x[3] > thr2[1]);
        if (__any_sync(0xffffffffu, trig)) {
          // raise each row's maximum to this page's exact maximum (a row's
          // values sit in the 8 lanes of the same t)
          float mx[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], o));
            mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], o));
          }
          float corr[2] = {1.f, 1.f};
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            if (mx[k] != -INFINITY && (mrow[k] == -INFINITY || mx[k] > 0.f)) {
              if (mrow[k] != -INFINITY) corr[k] = ex2(-mx[k]);  // 2^(m_old - m_new)
              mrow[k] = (mrow[k] == -INFINITY ? 0.f : mrow[k]) + mx[k];
              nm2[k] = -mrow[k];
              thr2[k] = kRaiseLog2;
              x[k] -= mx[k];
              x[k + 2] -= mx[k];
            }
            lrow[k] *= corr[k];
          }
          if (corr[0] != 1.f || corr[1] != 1.f) {
#pragma unroll
            for (int mt = 0; mt < T::MT; ++mt) {
              oacc[mt][0][0] *= corr[0];
              oacc[mt][0][1] *= corr[1];
              oacc[mt][0][2] *= corr[0];
              oacc[mt][0][3] *= corr[1];
            }
          }
        }
        const float p0 = ex2(x[0]), p1 = ex2(x[1]), p2 = ex2(x[2]), p3 = ex2(x[3]);
        lrow[0] += p0 + p2;
        lrow[1] += p1 + p3;
        // P^T fragments for the PV product: transpose the two 8 x 8 blocks
        // (tokens 0-7 and 8-15 x the 8 rows)
        pfrag[0][0] = movmatrix_trans(f32x2_to_f16x2(p0, p1));
        pfrag[0][1] = movmatrix_trans(f32x2_to_f16x2(p2, p3));
      }
    } else {
      // ---- S = Q K^T for tokens tok0 .. tok0+15 (two n-tiles) -------------
      // two accumulators per n-tile (alternate k-steps) halve the dependent
      // mma chain; they are added after the last k-step
      float sacc[2][4], sacc2[2][4];
  #pragma unroll
      for (int nt = 0; nt < 2; ++nt)
  #pragma unroll
        for (int k = 0; k < 4; ++k) {
          sacc[nt][k] = 0.f;
          sacc2[nt][k] = 0.f;
        }
  #pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int row = 8 * nt + g;
  #pragma unroll
        for (int c = 0; c < T::NCH; ++c) {
          const int ch = 4 * c + t;
          uint32_t w[T::CB / 4];
          uint32_t sc0, sc1;
          if constexpr (T::CB == 16) {
            const int pos = T::S::k_pos(row, ch);
            const uint4 v = *reinterpret_cast<const uint4*>(st + row * T::KROW + pos * 16);
            w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
            const uint32_t sfp = *reinterpret_cast<const uint16_t*>(
                st + T::OFF_KSF + row * T::KSFROW + 2 * ch);
            const uint32_t s2 = e4m3x2_to_f16x2(sfp);
            sc0 = bcast_lo(s2);
            sc1 = bcast_hi(s2);
          } else {
            const uint2 v = *reinterpret_cast<const uint2*>(st + row * T::KROW + ch * 8);
            w[0] = v.x; w[1] = v.y;
            const uint32_t sfb = st[T::OFF_KSF + row * T::KSFROW + ch];
            sc0 = bcast_lo(e4m3x2_to_f16x2(sfb));
            sc1 = sc0;
          }
  #pragma unroll
          for (int q = 0; q < T::CB / 4; ++q) {
            uint32_t h[4];
            e2m1x8_to_f16x8(w[q], h);
            const uint32_t sc = (T::CB == 16 && q >= 2) ? sc1 : sc0;
  #pragma unroll
            for (int j = 0; j < 4; ++j) h[j] = hmul2(h[j], sc);
            const int kk = c * T::KS_PER_CH + 2 * q;
            uint32_t a0[4], a1[4];
            if constexpr (T::Q_IN_REGS) {
  #pragma unroll
              for (int x = 0; x < 4; ++x) {
                a0[x] = qreg[kk][x];
                a1[x] = qreg[kk + 1][x];
              }
            } else {
              q_frag(kk, a0);
              q_frag(kk + 1, a1);
            }
            mma_16816(sacc[nt], a0, h[0], h[1]);
            mma_16816(sacc2[nt], a1, h[2], h[3]);
          }
        }
      }
  #pragma unroll
      for (int nt = 0; nt < 2; ++nt)
  #pragma unroll
        for (int k = 0; k < 4; ++k) sacc[nt][k] += sacc2[nt][k];

      // ---- online softmax (log2 domain), rows g and g+8 -------------------
      const bool need_mask = tok0 + 15 > min_lim;
      float corr[NT];
  #pragma unroll
      for (int hf = 0; hf < NT; ++hf) {
        float x[4] = {sacc[0][2 * hf] * rowf[hf], sacc[0][2 * hf + 1] * rowf[hf],
                      sacc[1][2 * hf] * rowf[hf], sacc[1][2 * hf + 1] * rowf[hf]};
        if (need_mask) {
          const int j0 = tok0 + 2 * t;
          if (j0 > rowlim[hf]) x[0] = -INFINITY;
          if (j0 + 1 > rowlim[hf]) x[1] = -INFINITY;
          if (j0 + 8 > rowlim[hf]) x[2] = -INFINITY;
          if (j0 + 9 > rowlim[hf]) x[3] = -INFINITY;
        }
        float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run[hf], mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        corr[hf] = ex2(m_run[hf] - m_use);
        m_run[hf] = m_new;
        const float p0 = ex2(x[0] - m_use), p1 = ex2(x[1] - m_use);
        const float p2 = ex2(x[2] - m_use), p3 = ex2(x[3] - m_use);
        l_run[hf] = l_run[hf] * corr[hf] + ((p0 + p1) + (p2 + p3));
        pfrag[hf][0] = f32x2_to_f16x2(p0, p1);
        pfrag[hf][1] = f32x2_to_f16x2(p2, p3);
      }
      // rescale O^T columns (query rows 8nq+2t, 8nq+2t+1); skipped when no
      // row maximum of the warp moved (corr == 1 exactly for every row)
      bool moved = false;
  #pragma unroll
      for (int hf = 0; hf < NT; ++hf) moved |= corr[hf] != 1.f;
      if (__any_sync(0xffffffffu, moved)) {
  #pragma unroll
      for (int nq = 0; nq < NT; ++nq) {
        const float cA = __shfl_sync(0xffffffffu, corr[nq], (2 * t) * 4);
        const float cB = __shfl_sync(0xffffffffu, corr[nq], (2 * t + 1) * 4);
  #pragma unroll
        for (int mt = 0; mt < T::MT; ++mt) {
          oacc[mt][nq][0] *= cA;
          oacc[mt][nq][1] *= cB;
          oacc[mt][nq][2] *= cA;
          oacc[mt][nq][3] *= cB;
        }
      }
      }
    }

    // ---- O^T += V_hat^T P^T ---------------------------------------------
    // tokens 2t, 2t+1, 2t+8, 2t+9; lane group g owns bytes [g*VC, g*VC+VC)
    if constexpr (MODE != 1) {
      // Interleave the nibbles of two tokens' bytes before converting: for
      // words W0 (token 2t) and W1 (token 2t+1), X holds in each byte the
      // even-dim code of W0 (low nibble) and of W1 (high nibble), Y the
      // odd-dim codes, so cvt(X byte j) = {v[2t][d], v[2t+1][d]} is A row g
      // and cvt(Y byte j) is A row g+8 of m-tile 4wq+j.
      constexpr uint32_t kLoNib = 0x0F0F0F0Fu;
#pragma unroll
      for (int wq = 0; wq < VW; ++wq) {
        uint32_t x[2], y[2];
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          const uint32_t w0 = vw[2 * pr][wq], w1 = vw[2 * pr + 1][wq];
          x[pr] = (w0 & kLoNib) | ((w1 << 4) & ~kLoNib);
          y[pr] = ((w0 >> 4) & kLoNib) | (w1 & ~kLoNib);
        }
        auto mtile = [&](auto jc) {
          constexpr int j = decltype(jc)::value;
          const int mt = 4 * wq + j;
          if (mt >= T::VC) return;
          const int bl = (mt * 2) / 16;
          uint32_t a[4];
          a[0] = hmul2(e2m1x2_byte_to_f16x2<j>(x[0]), sA[bl]);
          a[1] = hmul2(e2m1x2_byte_to_f16x2<j>(y[0]), sA[bl]);
          a[2] = hmul2(e2m1x2_byte_to_f16x2<j>(x[1]), sB[bl]);
          a[3] = hmul2(e2m1x2_byte_to_f16x2<j>(y[1]), sB[bl]);
#pragma unroll
          for (int nq = 0; nq < NT; ++nq)
            mma_16816(oacc[mt][nq], a, pfrag[nq][0], pfrag[nq][1]);
        };
        mtile(std::integral_constant<int, 0>{});
        mtile(std::integral_constant<int, 1>{});
        mtile(std::integral_constant<int, 2>{});
        mtile(std::integral_constant<int, 3>{});
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();

  if constexpr (MODE == 1) {
    // ---- the row-maximum pass: the unit's maxima (over the 8 lanes of each
    // t, then over the warps) stored for the attention pass --------------
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
      for (int o = 4; o < 32; o <<= 1)
        mfix[k] = fmaxf(mfix[k], __shfl_xor_sync(0xffffffffu, mfix[k], o));
    __syncthreads();  // every warp is done with its pipeline buffers
    float* sMx = reinterpret_cast<float*>(pipe);  // [WARPS][RB]
    if (g == 0) {
      sMx[warp * T::RB + 2 * t] = mfix[0];
      sMx[warp * T::RB + 2 * t + 1] = mfix[1];
    }
    __syncthreads();
    if (tid < T::RB && row0 + tid < R) {
      const int r = row0 + tid;
      float m = -INFINITY;
      for (int w = 0; w < WARPS; ++w) m = fmaxf(m, sMx[w * T::RB + tid]);
      p.row_max[((int64_t)(u.qo_begin + r / G) * p.num_qo_heads + u.h_kv * G + r % G) *
                    p.row_max_splits + u.split] = m;
    }
    return;
  }
  // ---- combine the warps ------------------------------------------------
  if constexpr (NT == 1) {  // rows 2t, 2t+1: sum over the 8 lanes of the same t
#pragma unroll
    for (int k = 0; k < 2; ++k) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) lrow[k] += __shfl_xor_sync(0xffffffffu, lrow[k], o);
    }
  } else {
#pragma unroll
    for (int hf = 0; hf < NT; ++hf) {
      l_run[hf] += __shfl_xor_sync(0xffffffffu, l_run[hf], 1);
      l_run[hf] += __shfl_xor_sync(0xffffffffu, l_run[hf], 2);
    }
  }
  __syncthreads();  // every warp is done with its pipeline buffers
  float* sO = reinterpret_cast<float*>(pipe);           // [WARPS][RB][DV]
  float* sM = sO + WARPS * T::RB * DV;                  // [WARPS][RB]
  float* sL = sM + WARPS * T::RB;                       // [WARPS][RB]
  if constexpr (NT == 1) {
    if (g == 0) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if constexpr (MODE == 2) {
          // the row sum carries the scale of p and the maximum drops it, so
          // the combine divides o by 2688 * sum p and lse = m + log2(sum p);
          // a warp that saw no key of the row contributes nothing
          sM[warp * T::RB + 2 * t + k] = lrow[k] > 0.f ? mfix[k] - kLog2PScale : -INFINITY;
          sL[warp * T::RB + 2 * t + k] = lrow[k] * kPScale;
        } else {
          sM[warp * T::RB + 2 * t + k] = mrow[k];
          sL[warp * T::RB + 2 * t + k] = lrow[k];
        }
      }
    }
  } else if (t == 0) {
#pragma unroll
    for (int hf = 0; hf < NT; ++hf) {
      sM[warp * T::RB + 8 * hf + g] = m_run[hf];
      sL[warp * T::RB + 8 * hf + g] = l_run[hf];
    }
  }
#pragma unroll
  for (int mt = 0; mt < T::MT; ++mt) {
    const int vb = g * T::VC + mt;  // byte of the V row -> dims 2vb, 2vb+1
#pragma unroll
    for (int nq = 0; nq < NT; ++nq) {
      float* o0 = sO + (warp * T::RB + 8 * nq + 2 * t) * DV + 2 * vb;
      float* o1 = o0 + DV;
      *reinterpret_cast<float2*>(o0) = make_float2(oacc[mt][nq][0], oacc[mt][nq][2]);
      *reinterpret_cast<float2*>(o1) = make_float2(oacc[mt][nq][1], oacc[mt][nq][3]);
    }
  }
  __syncthreads();

  finish_unit<T::RB, DV, WARPS>(p, u, row0, R, sM, sL, sO, sRowF);
}

// Launch shape (compile-time; the defaults are the tuned values).
#ifndef NVFP4KV_TC_WARPS
#define NVFP4KV_TC_WARPS 4
#endif
#ifndef NVFP4KV_TC_STAGES
#define NVFP4KV_TC_STAGES 4
#endif

template <int DK, int DV, int NT, int MODE = 0>
bool make_tc(AttendConfig* cfg) {
  // 512-wide K rows: 8 warps per CTA (one CTA per SM by shared memory, and
  // twice the warps streaming pages): 30.9 against 42.3 us on the 512/256
  // decode workload
  constexpr int WARPS = DK >= 512 ? 8 : NVFP4KV_TC_WARPS;
  constexpr int STAGES = DK >= 512 ? 3 : NVFP4KV_TC_STAGES;
  using T = TcTraits<DK, DV, NT, WARPS, STAGES>;
  cfg->kind = MODE == 0 ? kKernelTensorCore : kKernelFp4QP;
  cfg->dk = DK;
  cfg->dv = DV;
  cfg->rows = T::RB;
  cfg->warps = WARPS;
  cfg->smem_bytes = T::SMEM;
  cfg->func =
      reinterpret_cast<const void*>(attend_tc_kernel<DK, DV, NT, WARPS, STAGES, MODE>);
  return true;
}

}  // namespace

bool attend_config_tc(int dk, int dv, int rows, AttendConfig* cfg) {
  const int nt = rows <= 8 ? 1 : 2;
#define NVFP4KV_TC_CASE(DK_, DV_)                                                   \
  if (dk == DK_ && dv == DV_) return nt == 1 ? make_tc<DK_, DV_, 1>(cfg) : make_tc<DK_, DV_, 2>(cfg);
  NVFP4KV_TC_CASE(64, 64)
  NVFP4KV_TC_CASE(128, 128)
  NVFP4KV_TC_CASE(256, 256)
  NVFP4KV_TC_CASE(256, 128)
  NVFP4KV_TC_CASE(512, 256)
#undef NVFP4KV_TC_CASE
  return false;
}

// The FP4 query and probabilities kernels (one row block of <= 8 rows): pass
// 1 writes the units' row maxima, pass 2 attends with them.
bool attend_config_tc_fp4qp(int dk, int dv, int rows, int pass, AttendConfig* cfg) {
  if (rows > 8 || (pass != 1 && pass != 2)) return false;
  if (dk == 64 && dv == 64) return pass == 1 ? make_tc<64, 64, 1, 1>(cfg) : make_tc<64, 64, 1, 2>(cfg);
  if (dk == 128 && dv == 128)
    return pass == 1 ? make_tc<128, 128, 1, 1>(cfg) : make_tc<128, 128, 1, 2>(cfg);
  return false;
}

}  // namespace nvfp4kv
