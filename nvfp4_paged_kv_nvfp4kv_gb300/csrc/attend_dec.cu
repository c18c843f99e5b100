// attend_dec.cu -- paged NVFP4 decode attention for one block of at most 8
// query rows per (request, kv head) and head dims of at most 128, over caches
// whose (page, head) regions are contiguous (HND), sm_103a.
//
// It computes what attend_tc.cu computes (page "Support NVFP4 KV cache decode
// on SM120": packed e2m1 K/V with per-16 E4M3 scale caches, unpacked and
// scaled before the QK and PV products; page "fix(attention): correct SM120
// NVFP4 qk_correction layout, row-sum reduction, and lse": row reductions over
// exactly the lanes that own a row, lse written as natural-log sum-exp), with
// the same arithmetic, but streams the pages differently:
//  * Each warp owns every WARPS-th page of the work unit.  Its page ids sit in
//    one register (lane k holds the id of its page 32 b + k), read 32 pages
//    ahead and checked against the pool once; a page's id comes from a shuffle.
//  * Every lane copies 16-byte pieces of a page (packed K rows, packed V rows,
//    the two scale regions) with cp.async into a ring of STAGES stages per
//    warp, one commit group per page.
//  * A CTA holds four such units (16 warps).  The warp schedulers favour the
//    oldest warps, so separate CTAs of one SM finish their equal shares at
//    very different times; the four units of a CTA instead meet at a
//    CTA-wide barrier after every round of STAGES pages and stay level.
//  * Tokens of a page are taken in the order m -> m ^ ((m >> 1) & 1) for the
//    rows of the score product, the columns of P and the rows of V alike (a
//    contraction does not depend on the order of its terms), so the lanes'
//    reads of the unpadded V rows hit distinct banks.
//  * The step's new tokens (nvfp4kv_decode_append_run) are quantised by the
//    warp that owns their page when it reaches that page (the recipe of
//    quantize_append): the bytes go to the cache for later steps and straight
//    into the landed stage, so no copy has to wait for the cache store.  Each
//    page belongs to one CTA, so no other CTA reads the stored bytes.
//  * S^T = K_hat . Q^T (M = 16 tokens, N = 8 query rows) with mma.sync
//    m16n8k16, the running maximum raised lazily (only when a score exceeds
//    it by more than 2^8), and O^T += V_hat^T . P^T with P kept in registers,
//    as in attend_tc.cu.
#include <cfloat>
#include <cstdint>
#include <type_traits>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "epilogue.cuh"
#include "internal.h"
#include "quantize.cuh"

namespace nvfp4kv {
namespace {

using namespace dev;

constexpr float kDecRaiseLog2 = 8.f;
constexpr uint32_t kPaceHintNs = 2000;  // suspend hint of one pacing poll
constexpr int kPacePolls = 5000;        // a pacing wait gives up after these polls

// One poll of an mbarrier phase that may suspend the thread until the phase
// completes or about `ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_wait_hint(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive_one(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}

template <int DK, int DV, int WARPS, int STAGES>
struct DecTraits {
  static constexpr int KROW = DK / 2, VROW = DV / 2, KSFROW = DK / 16, VSFROW = DV / 16;
  static constexpr int K_BYTES = 16 * KROW, V_BYTES = 16 * VROW;
  static constexpr int KSF_BYTES = 16 * KSFROW, VSF_BYTES = 16 * VSFROW;
  static constexpr int OFF_V = K_BYTES, OFF_KSF = OFF_V + V_BYTES, OFF_VSF = OFF_KSF + KSF_BYTES;
  static constexpr int STAGE_BYTES = OFF_VSF + VSF_BYTES;
  static constexpr int RB = 8;                         // query rows per CTA
  static constexpr int CB = (DK / 8 < 16) ? DK / 8 : 16;  // K bytes per lane chunk
  static constexpr int NCH = (DK / 8) / CB;
  static constexpr int KSTEPS = DK / 16;
  static constexpr int KS_PER_CH = CB / 2;
  static constexpr int VC = DV / 16;                   // V bytes per lane per token
  static constexpr int MT = DV / 16;                   // PV m-tiles
  static constexpr int PIPE_BYTES = WARPS * STAGES * STAGE_BYTES;
  static constexpr int COMB_BYTES = WARPS * RB * (DV + 2) * 4;
  static constexpr int MAIN_BYTES = PIPE_BYTES > COMB_BYTES ? PIPE_BYTES : COMB_BYTES;
  static constexpr int QROW = DK + 8;                  // f16 elements, padded
  static constexpr int Q_BYTES = RB * QROW * 2;
  static constexpr int OFF_Q = MAIN_BYTES;
  static constexpr int OFF_ROW = OFF_Q + Q_BYTES;      // RB floats + RB ints; later
  static constexpr int ROW_BYTES = 2 * RB * 4 + 16;    // the epilogue's 2 RB + 1 words
  // bf16 K and V rows of the fused append's new tokens (at most RB per unit)
  static constexpr int NEW_ROW = (DK + DV) * 2;
  static constexpr int OFF_PID = (OFF_ROW + ROW_BYTES + 15) / 16 * 16;  // page id per stage
  static constexpr int OFF_NEW = (OFF_PID + WARPS * STAGES * 4 + 15) / 16 * 16;
  static constexpr int SMEM = OFF_NEW + RB * NEW_ROW;
  static constexpr int SMEM_Q = (SMEM + 127) / 128 * 128;  // one quad's share of the CTA
  static_assert(DK <= 128 && DV <= 128 && DK % 64 == 0 && DV % 64 == 0, "head dims");
  static_assert(K_BYTES % 16 == 0 && V_BYTES % 16 == 0 && KSF_BYTES % 16 == 0 &&
                    VSF_BYTES % 16 == 0 && STAGE_BYTES % 16 == 0, "bulk copy sizes");
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// token of mma row / P column m of a page
__device__ __forceinline__ int tok_of(int m) { return m ^ ((m >> 1) & 1); }

// QUADS groups of WARPS warps per CTA, one work unit each (unit
// QUADS * blockIdx.x + quad).  The groups share nothing but the CTA: each
// synchronises on its own named barrier.  Their pages go in rounds of STAGES
// per warp, and no warp starts a round before every warp of the CTA has
// finished the round before the previous one (two mbarriers, one per round
// parity), so the units of an SM advance together instead of in the order
// the warp schedulers favour.  The pacing carries no data: a pacing wait
// that runs out sets NVFP4KV_FLAG_PACE_TIMEOUT and the warp goes on.
template <int DK, int DV, int WARPS, int STAGES, int QUADS>
__global__ void __launch_bounds__(WARPS * 32 * QUADS, 1) attend_dec_kernel(const AttendParams p) {
  using T = DecTraits<DK, DV, WARPS, STAGES>;
  extern __shared__ __align__(128) uint8_t smem_all[];
  const int quad = threadIdx.x / (WARPS * 32);
  const int unit = blockIdx.x * QUADS + quad;
  int* s_rounds = reinterpret_cast<int*>(smem_all + QUADS * T::SMEM_Q);
  uint64_t* s_pace = reinterpret_cast<uint64_t*>(smem_all + QUADS * T::SMEM_Q + 8);
  if (threadIdx.x == 0) {
    *s_rounds = 0;
    const int live = min(QUADS, p.num_units - (int)blockIdx.x * QUADS);
    mbar_init(&s_pace[0], live * WARPS);  // one arrival per warp of a unit
    mbar_init(&s_pace[1], live * WARPS);
  }
  __syncthreads();  // (CTA-wide 1 of 2)
  if (unit >= p.num_units) {
    __syncthreads();  // (CTA-wide 2 of 2); no unit for this group
    return;
  }
  auto qsync = [quad] {
    asm volatile("bar.sync %0, %1;\n" ::"r"(1 + quad), "n"(WARPS * 32) : "memory");
  };
  uint8_t* smem = smem_all + quad * T::SMEM_Q;
  uint8_t* pipe = smem;
  uint16_t* sQ = reinterpret_cast<uint16_t*>(smem + T::OFF_Q);
  float* sRowF = reinterpret_cast<float*>(smem + T::OFF_ROW);
  int* sRowLim = reinterpret_cast<int*>(sRowF + T::RB);
  int32_t* sPid = reinterpret_cast<int32_t*>(smem + T::OFF_PID);
  uint8_t* sNew = smem + T::OFF_NEW;

  const int tid = threadIdx.x % (WARPS * 32), lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  const WorkUnit u = load_unit(p, unit, tid == 0);
  const int G = p.group;
  const int R = G * u.qo_len;   // <= 8: one row block
  const int npw = u.num_pages > warp ? (u.num_pages - warp + WARPS - 1) / WARPS : 0;
  const int32_t* pidx = p.kv_indices + u.page_begin + warp;

  // ids of this warp's pages 32 blk .. 32 blk + 31 (lane k: page 32 blk + k),
  // checked against the pool (a bad id becomes -1: page 0 is read, flagged)
  auto load_ids = [&](int blk) -> int32_t {
    const int j = 32 * blk + lane;
    int32_t id = 0;
    if (j < npw) {
      id = __ldg(pidx + j * WARPS);
      if (id < 0 || id >= p.cache.num_pages) {
        atomicOr(p.flags, 0x1u);
        id = -1;
      }
    }
    return id;
  };
  int32_t ids_cur = load_ids(0);
  int32_t ids_nxt = npw > 32 ? load_ids(1) : 0;

  // ---- fused append: this kv head's new tokens in the unit's pages --------
  // [new_lo, new_hi): positions of the step's new tokens in this unit.  The
  // warp that streams a token's page prefetches its bf16 K and V rows into
  // sNew (cp.async, with its first page) and, when the page has landed,
  // quantises them (the recipe of quantize_append) into the cache for later
  // steps and into the stage (its copy may have read the page before the
  // cache store).  A page belongs to one warp, so no other warp or CTA reads
  // the stored bytes in this launch.
  const int first_new = u.kv_len - u.qo_len;
  int new_lo = 0, new_hi = 0;
  if (p.new_k != nullptr) {
    new_lo = max(first_new, u.tok_begin);
    new_hi = min(u.kv_len, u.tok_begin + 16 * u.num_pages);
  }
  {
    constexpr int NCK = T::NEW_ROW / 16;  // 16-byte chunks of one new token
    for (int idx = lane; idx < (new_hi - new_lo) * NCK; idx += 32) {
      const int tok = new_lo + idx / NCK, ch = idx % NCK;
      if (((tok - u.tok_begin) / 16) % WARPS != warp) continue;
      const int i = tok - first_new;
      const uint16_t* src =
          ch < DK / 8 ? p.new_k + (int64_t)(u.qo_begin + i) * p.nk_stride_tok +
                            (int64_t)u.h_kv * p.nk_stride_head + 8 * ch
                      : p.new_v + (int64_t)(u.qo_begin + i) * p.nv_stride_tok +
                            (int64_t)u.h_kv * p.nv_stride_head + 8 * (ch - DK / 8);
      cp_async_16(sNew + (tok - new_lo) * T::NEW_ROW + 16 * ch, src);
    }
  }
  // ---- Q rows: one 16-byte load per thread per 8 elements ----------------
  constexpr int QCH = T::RB * DK / 8;
  constexpr int QPT = (QCH + WARPS * 32 - 1) / (WARPS * 32);
  uint4 qv[QPT];
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int ci = tid + k * WARPS * 32;
    const int rr = ci / (DK / 8);
    qv[k] = make_uint4(0u, 0u, 0u, 0u);
    if (ci < QCH && rr < R) {
      const int i = rr / G, gh = rr % G;
      qv[k] = *reinterpret_cast<const uint4*>(p.q + (int64_t)(u.qo_begin + i) * p.q_stride_tok +
                                              (int64_t)(u.h_kv * G + gh) * p.q_stride_head +
                                              (ci % (DK / 8)) * 8);
    }
  }
  if (tid < T::RB) reinterpret_cast<int*>(sRowF)[tid] = 0;  // per-row amax bits

  qsync();  // amax slots zeroed

  // ---- the page pipeline: lane 0 copies, everyone waits on the stage -----
  uint8_t* wpipe = pipe + warp * STAGES * T::STAGE_BYTES;
  const CacheView& c = p.cache;
  const uint8_t* kb = c.k_data + (int64_t)u.h_kv * c.k_sh;
  const uint8_t* vb = c.v_data + (int64_t)u.h_kv * c.v_sh;
  const uint8_t* ksb = c.k_sf + (int64_t)u.h_kv * c.ksf_sh;
  const uint8_t* vsb = c.v_sf + (int64_t)u.h_kv * c.vsf_sh;
  const uint32_t ksp = (uint32_t)c.k_sp, vsp = (uint32_t)c.v_sp;
  const uint32_t kssp = (uint32_t)c.ksf_sp, vssp = (uint32_t)c.vsf_sp;
  // per-lane 16-byte chunks of the cp.async path: K and V rows (KC chunks
  // each, lane-strided), then the two scale regions (lanes 0 .. SC-1 for K,
  // SC .. 2 SC - 1 for V)
  constexpr int KC = T::K_BYTES / 512, SC = T::KSF_BYTES / 16;
  static_assert(T::K_BYTES == T::V_BYTES && T::KSF_BYTES == T::VSF_BYTES && 2 * SC <= 32,
                "cp.async layout");
  const uint8_t* kl = kb + lane * 16;
  const uint8_t* vl = vb + lane * 16;
  const uint8_t* sl = lane < SC ? ksb + lane * 16 : vsb + (lane - SC) * 16;
  const uint32_t slp = lane < SC ? kssp : vssp;
  const int soff = lane < SC ? T::OFF_KSF + lane * 16 : T::OFF_VSF + (lane - SC) * 16;
  // shared addresses: this warp's stages, and this lane's copy targets in one
  const uint32_t wpipe_s = smem_addr(wpipe);
  const uint32_t lane_cp = wpipe_s + lane * 16, lane_sc = wpipe_s + soff;
  // page j into stage js (= j % STAGES)
  auto issue = [&](int j, int32_t pid, int js) {
    uint8_t* st = wpipe + js * T::STAGE_BYTES;
    if (lane == 0) sPid[warp * STAGES + js] = pid;
    const uint32_t pg = (uint32_t)max(pid, 0);
    {
      (void)st;
      const uint32_t so = js * T::STAGE_BYTES;
      const uint8_t* ks = kl + (uint64_t)pg * ksp;
      const uint8_t* vs = vl + (uint64_t)pg * vsp;
      static_assert(KC == 1 || KC == 2, "chunks per lane");
      cp_async_16s<0>(lane_cp + so, ks);
      if constexpr (KC == 2) cp_async_16s<512>(lane_cp + so, ks);
      // V rows: the stage's V region starts OFF_V bytes in
      cp_async_16s<T::OFF_V, 0>(lane_cp + so, vs);
      if constexpr (KC == 2) cp_async_16s<T::OFF_V + 512, 512>(lane_cp + so, vs);
      if (lane < 2 * SC) cp_async_16s<0>(lane_sc + so, sl + (uint64_t)pg * slp);
      cp_async_commit();
    }
  };
#pragma unroll
  for (int j = 0; j < STAGES - 1; ++j) {
    const int32_t pid = __shfl_sync(0xffffffffu, ids_cur, j);
    if (j < npw) issue(j, pid, j);
    else cp_async_commit();
  }
  // ---- Q: per-row power-of-two prescale into f16, row limits ------------
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
  qsync();
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int ci = tid + k * WARPS * 32;
    if (ci >= QCH) continue;
    const int rr = ci / (DK / 8);
    const float amax = __int_as_float(reinterpret_cast<const int*>(sRowF)[rr]);
    int e = 0;  // amax * 2^e in [2^14, 2^15)
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
      sRowLim[rr] = rr >= R ? -1 : (p.causal ? (u.kv_len - u.qo_len + rr / G) : (u.kv_len - 1));
      qv[k].x = __float_as_uint(rr >= R ? 0.f
                                        : p.qk_scale_log2 *
                                              __uint_as_float((uint32_t)(127 - e) << 23));
    }
  }
  qsync();
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int ci = tid + k * WARPS * 32;
    if (ci < QCH && ci % (DK / 8) == 0) sRowF[ci / (DK / 8)] = __uint_as_float(qv[k].x);
  }
  qsync();

  // this lane's query rows 2t and 2t+1: score factor f, -m_use (the
  // running max, log2 domain, once the row has one: bit k of has_max) and
  // partial sum.  A row's raise threshold is 2^8 once it has a maximum, -inf
  // before (any score raises), +inf for a padding row (never); thr_lane is
  // the smaller of the lane's two.  The causal limits stay in sRowLim.
  float f2[2], nm2[2], lrow[2];
  uint32_t has_max = 0;
  int min_lim = INT32_MAX;
  for (int rr = 0; rr < T::RB; ++rr)
    if (sRowLim[rr] >= 0) min_lim = min(min_lim, sRowLim[rr]);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    f2[k] = sRowF[2 * t + k];
    nm2[k] = 0.f;
    lrow[k] = 0.f;
  }
  auto lane_threshold = [&]() {
    float th = INFINITY;
#pragma unroll
    for (int k = 0; k < 2; ++k)
      th = fminf(th, (has_max >> k) & 1u ? kDecRaiseLog2
                                         : (sRowLim[2 * t + k] >= 0 ? -INFINITY : INFINITY));
    return th;
  };
  float thr_lane = lane_threshold();
  // Q fragments (the B operand of S^T): k-step kk covers the 4 dims at
  // 2 (4c + t) CB + 4m for chunk c = kk / KS_PER_CH, step m
  uint32_t qreg[T::KSTEPS][2];
#pragma unroll
  for (int kk = 0; kk < T::KSTEPS; ++kk) {
    const int cc = kk / T::KS_PER_CH, m = kk % T::KS_PER_CH;
    const uint2 lo = *reinterpret_cast<const uint2*>(sQ + g * T::QROW + 2 * (4 * cc + t) * T::CB + 4 * m);
    qreg[kk][0] = lo.x;
    qreg[kk][1] = lo.y;
  }
  float oacc[T::MT][4];
#pragma unroll
  for (int mt = 0; mt < T::MT; ++mt)
#pragma unroll
    for (int k = 0; k < 4; ++k) oacc[mt][k] = 0.f;

  auto patch_new = [&](uint8_t* st, int tok0, int is) {
    const int lo = max(new_lo, tok0), hi = min(new_hi, tok0 + 16);
    if (lo >= hi) return;
    __syncwarp();
    const int32_t pid = sPid[warp * STAGES + is];
    constexpr int NB = DK / 16 + DV / 16;
    const CacheView& cv = p.cache;
    for (int idx = lane; idx < (hi - lo) * NB; idx += 32) {
      const int tok = lo + idx / NB, blk = idx % NB, slot = tok - tok0;
      const bool isv = blk >= DK / 16;
      const int jb = isv ? blk - DK / 16 : blk;
      const uint8_t* src = sNew + (tok - new_lo) * T::NEW_ROW + (isv ? DK * 2 : 0) + 32 * jb;
      uint2 packed;
      const uint32_t sfb = quantize_block16(*reinterpret_cast<const uint4*>(src),
                                            *reinterpret_cast<const uint4*>(src + 16),
                                            isv ? p.v_global_scale : p.k_global_scale, &packed);
      uint8_t* srow = st + (isv ? T::OFF_V + slot * T::VROW : slot * T::KROW);
      *reinterpret_cast<uint2*>(srow + 8 * jb) = packed;
      st[(isv ? T::OFF_VSF + slot * T::VSFROW : T::OFF_KSF + slot * T::KSFROW) + jb] =
          static_cast<uint8_t>(sfb);
      if (pid < 0) {
        atomicOr(p.flags, 0x2u);
        continue;
      }
      uint8_t* drow = const_cast<uint8_t*>(
          isv ? cv.v_data + pid * cv.v_sp + slot * cv.v_ss + u.h_kv * cv.v_sh
              : cv.k_data + pid * cv.k_sp + slot * cv.k_ss + u.h_kv * cv.k_sh);
      uint8_t* dsf = const_cast<uint8_t*>(
          isv ? cv.v_sf + pid * cv.vsf_sp + slot * cv.vsf_ss + u.h_kv * cv.vsf_sh
              : cv.k_sf + pid * cv.ksf_sp + slot * cv.ksf_ss + u.h_kv * cv.ksf_sh);
      *reinterpret_cast<uint2*>(drow + 8 * jb) = packed;
      dsf[jb] = static_cast<uint8_t>(sfb);
    }
    __syncwarp();  // the stage holds the new tokens before anyone reads it
  };

  // rows of the page this lane reads: tokens of mma rows g, g+8 (K) and of
  // P columns 2t, 2t+1, 2t+8, 2t+9 (V)
  // (tok_of(m + 8) = tok_of(m) + 8 and tok_of(2t + 1) = tok_of(2t) ^ 1, so
  // the second row of each pair is an immediate 8 rows further on)
  static_assert(T::NCH == 1, "one K chunk per lane");
  const int kr0 = tok_of(g), vt0 = tok_of(2 * t), vt1 = vt0 ^ 1;
  // shared addresses in stage 0 (stage s is s * STAGE_BYTES further on): K
  // row kr0 at the lane's chunk t, its scale pair, V rows vt0 / vt1 at byte
  // g VC, their scales at block g VC / 8
  const uint32_t o_k = wpipe_s + kr0 * T::KROW + t * T::CB;
  const uint32_t o_ks = wpipe_s + T::OFF_KSF + kr0 * T::KSFROW + t * (T::CB / 8);
  const uint32_t o_v0 = wpipe_s + T::OFF_V + vt0 * T::VROW + g * T::VC;
  const uint32_t o_v1 = wpipe_s + T::OFF_V + vt1 * T::VROW + g * T::VC;
  const uint32_t o_vs0 = wpipe_s + T::OFF_VSF + vt0 * T::VSFROW + (g * T::VC) / 8;
  const uint32_t o_vs1 = wpipe_s + T::OFF_VSF + vt1 * T::VSFROW + (g * T::VC) / 8;
  // Pages whose tokens reach the smallest row limit need the causal /
  // length mask, and pages holding this step's new tokens need the patch:
  // both sit at the end of the unit, so the loop runs a lean body over the
  // pages before the first such page and the full body over the rest.
  int tail_tok = min_lim;  // a page is special once tok0 + 15 > tail_tok
  if (new_lo < new_hi) tail_tok = min(tail_tok, new_lo - 1);
  int n_lean = 0;          // this warp's pages before the first special one
  {
    const int ok = tail_tok - 15 - u.tok_begin;  // pages pi with 16 pi <= ok
    const int unit_ok = ok >= 0 ? ok / 16 + 1 : 0;
    n_lean = unit_ok > warp ? min(npw, (unit_ok - warp + WARPS - 1) / WARPS) : 0;
  }
  // page i, held in stage is (= i % STAGES: a constant where the caller
  // unrolls, so the stage offsets become immediates)
  auto page = [&](int i, auto special, int is) {
    constexpr bool SP = decltype(special)::value;
    const int j = i + STAGES - 1;
    if (j < npw) {
      if ((j & 31) == 0) {
        ids_cur = ids_nxt;
        ids_nxt = load_ids(j / 32 + 1);
      }
      issue(j, __shfl_sync(0xffffffffu, ids_cur, j & 31), (is + STAGES - 1) % STAGES);
    } else {
      cp_async_commit();  // keep one group per page for the wait count
    }
    cp_async_wait<STAGES - 1>();
    __syncwarp();
    const uint32_t so = is * T::STAGE_BYTES;
    const int tok0 = u.tok_begin + (warp + i * WARPS) * 16;
    if constexpr (SP) {
      if (new_lo < new_hi) patch_new(wpipe + so, tok0, is);
    }
    const uint32_t sb = so;

    // V rows vt0, vt1, vt0 + 8, vt1 + 8 and their scales
    constexpr int VW = T::VC / 4 > 0 ? T::VC / 4 : 1;
    constexpr int V8 = 8 * T::VROW, VS8 = 8 * T::VSFROW;
    uint32_t vw[4][VW];
    if constexpr (T::VC == 8) {
      const uint2 a = lds_v2<0>(sb + o_v0), b = lds_v2<0>(sb + o_v1);
      const uint2 c2 = lds_v2<V8>(sb + o_v0), d = lds_v2<V8>(sb + o_v1);
      vw[0][0] = a.x; vw[0][1] = a.y; vw[1][0] = b.x; vw[1][1] = b.y;
      vw[2][0] = c2.x; vw[2][1] = c2.y; vw[3][0] = d.x; vw[3][1] = d.y;
    } else {
      vw[0][0] = lds_u32<0>(sb + o_v0);
      vw[1][0] = lds_u32<0>(sb + o_v1);
      vw[2][0] = lds_u32<V8>(sb + o_v0);
      vw[3][0] = lds_u32<V8>(sb + o_v1);
    }
    uint32_t s0 = lds_u8<0>(sb + o_vs0), s1 = lds_u8<0>(sb + o_vs1);
    uint32_t s2 = lds_u8<VS8>(sb + o_vs0), s3 = lds_u8<VS8>(sb + o_vs1);
    const int valid = u.kv_len - tok0;  // tokens of this page that exist
    if (SP && valid < 16) {
      // slots past kv_len may hold a NaN scale byte: their V scale is 0
      if (vt0 >= valid) s0 = 0;
      if (vt1 >= valid) s1 = 0;
      if (vt0 + 8 >= valid) s2 = 0;
      if (vt1 + 8 >= valid) s3 = 0;
    }
    const uint32_t sA = e4m3x2_to_f16x2(__byte_perm(s0, s1, 0x1140));
    const uint32_t sB = e4m3x2_to_f16x2(__byte_perm(s2, s3, 0x1140));

    // ---- S^T = K_hat Q^T: mma rows g, g+8 = tokens kr0, kr0 + 8 ---------
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb4[4] = {0.f, 0.f, 0.f, 0.f};
    constexpr int K8 = 8 * T::KROW, KS8 = 8 * T::KSFROW;
    {
      constexpr int cc = 0;
      uint32_t wg[T::CB / 4], w8[T::CB / 4], sg0, sg1, s80, s81;
      if constexpr (T::CB == 16) {
        const uint4 a = lds_v4<0>(sb + o_k), b = lds_v4<K8>(sb + o_k);
        wg[0] = a.x; wg[1] = a.y; wg[2] = a.z; wg[3] = a.w;
        w8[0] = b.x; w8[1] = b.y; w8[2] = b.z; w8[3] = b.w;
        const uint32_t ga = e4m3x2_to_f16x2(lds_u16<0>(sb + o_ks));
        const uint32_t gb = e4m3x2_to_f16x2(lds_u16<KS8>(sb + o_ks));
        sg0 = bcast_lo(ga); sg1 = bcast_hi(ga);
        s80 = bcast_lo(gb); s81 = bcast_hi(gb);
      } else {
        const uint2 a = lds_v2<0>(sb + o_k), b = lds_v2<K8>(sb + o_k);
        wg[0] = a.x; wg[1] = a.y;
        w8[0] = b.x; w8[1] = b.y;
        sg0 = sg1 = bcast_lo(e4m3x2_to_f16x2(lds_u8<0>(sb + o_ks)));
        s80 = s81 = bcast_lo(e4m3x2_to_f16x2(lds_u8<KS8>(sb + o_ks)));
      }
#pragma unroll
      for (int q = 0; q < T::CB / 4; ++q) {
        uint32_t hg[4], h8[4];
        e2m1x8_to_f16x8(wg[q], hg);
        e2m1x8_to_f16x8(w8[q], h8);
        const bool hi = T::CB == 16 && q >= 2;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          hg[e] = hmul2(hg[e], hi ? sg1 : sg0);
          h8[e] = hmul2(h8[e], hi ? s81 : s80);
        }
        const int kk = cc * T::KS_PER_CH + 2 * q;
        const uint32_t a0[4] = {hg[0], h8[0], hg[1], h8[1]};
        const uint32_t a1[4] = {hg[2], h8[2], hg[3], h8[3]};
        mma_16816(sa, a0, qreg[kk][0], qreg[kk][1]);
        mma_16816(sb4, a1, qreg[kk + 1][0], qreg[kk + 1][1]);
      }
    }

    // ---- softmax with a lazily raised maximum (log2 domain) -------------
    // x[0..3] = tokens kr0, kr0, kr1, kr1 x rows 2t, 2t+1, 2t, 2t+1
    float x[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) x[k] = fmaf(sa[k] + sb4[k], f2[k & 1], nm2[k & 1]);
    if (SP && tok0 + 15 > min_lim) {
      const int ta = tok0 + kr0, tb = ta + 8;
      const int l0 = sRowLim[2 * t], l1 = sRowLim[2 * t + 1];
      if (ta > l0) x[0] = -INFINITY;
      if (ta > l1) x[1] = -INFINITY;
      if (tb > l0) x[2] = -INFINITY;
      if (tb > l1) x[3] = -INFINITY;
    }
    // raise test against the lane's smaller threshold (a superset of the
    // rows that need it: the raise itself works per row)
    const bool trig = fmax3(x[0], x[1], fmaxf(x[2], x[3])) > thr_lane;
    if (__builtin_expect(__any_sync(0xffffffffu, trig), 0)) {
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
        const bool has = (has_max >> k) & 1u;
        if (mx[k] != -INFINITY && (!has || mx[k] > 0.f)) {
          if (has) corr[k] = ex2(-mx[k]);  // 2^(m_old - m_new)
          nm2[k] -= mx[k];                 // m_new = m_old + mx (0 + mx for a first max)
          has_max |= 1u << k;
          x[k] -= mx[k];
          x[k + 2] -= mx[k];
        }
        lrow[k] *= corr[k];
      }
      thr_lane = lane_threshold();
      if (corr[0] != 1.f || corr[1] != 1.f) {
#pragma unroll
        for (int mt = 0; mt < T::MT; ++mt) {
          oacc[mt][0] *= corr[0];
          oacc[mt][1] *= corr[1];
          oacc[mt][2] *= corr[0];
          oacc[mt][3] *= corr[1];
        }
      }
    }
    const float p0 = ex2(x[0]), p1 = ex2(x[1]), p2 = ex2(x[2]), p3 = ex2(x[3]);
    lrow[0] += p0 + p2;
    lrow[1] += p1 + p3;
    // P^T fragments for the PV product (the two 8 x 8 blocks transposed)
    const uint32_t pf0 = movmatrix_trans(f32x2_to_f16x2(p0, p1));
    const uint32_t pf1 = movmatrix_trans(f32x2_to_f16x2(p2, p3));

    // ---- O^T += V_hat^T P^T: P columns 2t, 2t+1, 2t+8, 2t+9 -------------
    {
      constexpr uint32_t kLoNib = 0x0F0F0F0Fu;
#pragma unroll
      for (int wq = 0; wq < VW; ++wq) {
        uint32_t xs[2], ys[2];
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          const uint32_t w0 = vw[2 * pr][wq], w1 = vw[2 * pr + 1][wq];
          xs[pr] = (w0 & kLoNib) | ((w1 << 4) & ~kLoNib);
          ys[pr] = ((w0 >> 4) & kLoNib) | (w1 & ~kLoNib);
        }
        auto mtile = [&](auto jc) {
          constexpr int jj = decltype(jc)::value;
          const int mt = 4 * wq + jj;
          if (mt >= T::VC) return;
          uint32_t a[4];
          a[0] = hmul2(e2m1x2_byte_to_f16x2<jj>(xs[0]), sA);
          a[1] = hmul2(e2m1x2_byte_to_f16x2<jj>(ys[0]), sA);
          a[2] = hmul2(e2m1x2_byte_to_f16x2<jj>(xs[1]), sB);
          a[3] = hmul2(e2m1x2_byte_to_f16x2<jj>(ys[1]), sB);
          mma_16816(oacc[mt], a, pf0, pf1);
        };
        mtile(std::integral_constant<int, 0>{});
        mtile(std::integral_constant<int, 1>{});
        mtile(std::integral_constant<int, 2>{});
        mtile(std::integral_constant<int, 3>{});
      }
    }
    __syncwarp();  // every lane has read the stage before lane 0 refills it
  };
  // Rounds of STAGES pages: every warp of the CTA takes part in the same
  // number of rounds (the CTA's largest) and works in as many as it has
  // pages for.  A round of lean pages is unrolled (the stage offsets are
  // then immediates); a round that reaches the tail pages, or the end, runs
  // the full body page by page.
  const int my_rounds = (npw + STAGES - 1) / STAGES;
  if (lane == 0) atomicMax(s_rounds, my_rounds);
  __syncthreads();  // (CTA-wide 2 of 2)
  const int rounds = *s_rounds;
  for (int r = 0; r < rounds; ++r) {
    const int i = r * STAGES;
    if (i + STAGES <= n_lean) {
#pragma unroll
      for (int k = 0; k < STAGES; ++k) page(i + k, std::false_type{}, k);
    } else {
#pragma unroll 1
      for (int k = 0; k < STAGES && i + k < npw; ++k) page(i + k, std::true_type{}, k);
    }
    // pacing: round r done; wait until every warp has done round r - 1
    if (lane == 0) {
      mbar_arrive_one(&s_pace[r & 1]);
      if (r >= 1) {
        bool done = false;
        for (int k = 0; k < kPacePolls && !done; ++k)
          done = mbar_wait_hint(&s_pace[(r - 1) & 1], ((r - 1) >> 1) & 1, kPaceHintNs);
        if (!done) atomicOr(p.flags, 0x10u);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();

  // ---- combine the warps ------------------------------------------------
#pragma unroll
  for (int k = 0; k < 2; ++k) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) lrow[k] += __shfl_xor_sync(0xffffffffu, lrow[k], o);
  }
  qsync();  // every warp is done with its pipeline buffers
  float* sO = reinterpret_cast<float*>(pipe);   // [WARPS][RB][DV]
  float* sM = sO + WARPS * T::RB * DV;          // [WARPS][RB]
  float* sL = sM + WARPS * T::RB;               // [WARPS][RB]
  if (g == 0) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      sM[warp * T::RB + 2 * t + k] = (has_max >> k) & 1u ? -nm2[k] : -INFINITY;
      sL[warp * T::RB + 2 * t + k] = lrow[k];
    }
  }
#pragma unroll
  for (int mt = 0; mt < T::MT; ++mt) {
    const int vbyte = g * T::VC + mt;  // byte of the V row -> dims 2vbyte, 2vbyte+1
    float* o0 = sO + (warp * T::RB + 2 * t) * DV + 2 * vbyte;
    float* o1 = o0 + DV;
    *reinterpret_cast<float2*>(o0) = make_float2(oacc[mt][0], oacc[mt][2]);
    *reinterpret_cast<float2*>(o1) = make_float2(oacc[mt][1], oacc[mt][3]);
  }
  qsync();

  finish_unit<T::RB, DV, WARPS>(p, u, 0, R, sM, sL, sO, sRowF, tid, qsync);
}

template <int DK, int DV, int QUADS>
bool make_dec(AttendConfig* cfg) {
  constexpr int WARPS = 4, STAGES = 4;
  using T = DecTraits<DK, DV, WARPS, STAGES>;
  cfg->kind = kKernelTensorCore;
  cfg->dk = DK;
  cfg->dv = DV;
  cfg->rows = T::RB;
  cfg->warps = WARPS * QUADS;
  cfg->units_per_cta = QUADS;
  cfg->smem_bytes = QUADS * T::SMEM_Q + 32;
  cfg->func = reinterpret_cast<const void*>(attend_dec_kernel<DK, DV, WARPS, STAGES, QUADS>);
  return true;
}

}  // namespace

// The decode kernel for (dk, dv) when a CTA has at most 8 query rows and the
// cache's (page, head) regions are contiguous, with `quads` units per CTA (4,
// or 1 for a grid of at most one unit per SM, where nothing competes and the
// smaller CTA starts sooner); false when not built.
bool attend_config_dec(int dk, int dv, int rows, int quads, AttendConfig* cfg) {
  if (rows > 8 || (quads != 1 && quads != 4)) return false;
  if (dk == 64 && dv == 64) return quads == 4 ? make_dec<64, 64, 4>(cfg) : make_dec<64, 64, 1>(cfg);
  if (dk == 128 && dv == 128)
    return quads == 4 ? make_dec<128, 128, 4>(cfg) : make_dec<128, 128, 1>(cfg);
  return false;
}

}  // namespace nvfp4kv
