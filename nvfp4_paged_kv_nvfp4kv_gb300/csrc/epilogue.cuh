// epilogue.cuh -- end of an attention work unit: combine the warps' online-
// softmax states of the CTA's query rows and store them; when the plan split
// the request, store an f32 partial state and let the last CTA of the
// (request, kv head, row block) fold all partials (log-sum-exp merge).
//
// The last CTA is found with a counter per (request, kv head, row block):
// every CTA publishes its partials (__threadfence) and then increments the
// counter; the CTA that sees num_splits - 1 is last, reads the partials
// through L2 (ld.global.cg) and resets the counter to 0 for the next run.
// No CTA waits for another.
#pragma once

#include <cstdint>

#include "device_common.cuh"
#include "internal.h"

namespace nvfp4kv {

// The split group's last CTA folds its partials.  Run by NTHREADS threads
// (tid in [0, NTHREADS)) that synchronise with `sync`; sFin: scratch of at
// least RB floats + 1 int.  Every thread must have stored its partials.
// Each thread folds whole (row, 4 dims) items: batches of MB partial states
// (their lse and o loaded together) with a running maximum, so the fold
// costs ceil(S / MB) dependent L2 round trips.
template <int RB, int DV, int NTHREADS, int MB = 8, class Sync>
__device__ __forceinline__ void merge_if_last(const AttendParams& p, const WorkUnit& u,
                                              int row0, int R, float* sFin, int tid,
                                              Sync sync) {
  using namespace dev;
  constexpr float kLog2e = 1.44269504088896340736f;
  constexpr float kLn2 = 0.69314718055994530942f;
  const int G = p.group, Hq = p.num_qo_heads;
  int* s_last = reinterpret_cast<int*>(sFin + 2 * RB);
  __threadfence();
  sync();
  if (tid == 0) {
    int* ctr = p.counters + (int64_t)u.pair * gridDim.y + blockIdx.y;
    const int old = atomicAdd(ctr, 1);
    *s_last = (old == u.num_splits - 1);
    if (*s_last) *ctr = 0;  // every other CTA of the group has arrived
  }
  sync();
  if (!*s_last) return;
  __threadfence();
  const int S = u.num_splits;
  constexpr int DQ = DV / 4;
  for (int idx = tid; idx < RB * DQ; idx += NTHREADS) {
    const int rr = idx / DQ, d4 = idx % DQ, r = row0 + rr;
    if (r >= R) continue;
    const int i = r / G, head = u.h_kv * G + r % G;
    const int64_t base = (int64_t)u.partial_base + ((int64_t)i * Hq + head) * S;
    float M = -INFINITY, L = 0.f;  // running max (log2 units) and sum
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < S; s0 += MB) {
      float lw[MB];
      float4 v[MB];
#pragma unroll
      for (int j = 0; j < MB; ++j) {
        lw[j] = -INFINITY;
        v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s0 + j < S) {
          lw[j] = __ldcg(p.partial_lse + base + s0 + j) * kLog2e;
          v[j] = __ldcg(reinterpret_cast<const float4*>(p.partial_o + (base + s0 + j) * DV) + d4);
        }
      }
      float mb = lw[0];
#pragma unroll
      for (int j = 1; j < MB; ++j) mb = fmaxf(mb, lw[j]);
      if (mb == -INFINITY) continue;
      const float mn = fmaxf(M, mb);
      const float cf = M == -INFINITY ? 0.f : ex2(M - mn);
      L *= cf;
      acc.x *= cf; acc.y *= cf; acc.z *= cf; acc.w *= cf;
#pragma unroll
      for (int j = 0; j < MB; ++j) {
        const float w = ex2(lw[j] - mn);  // 0 for lw = -inf
        L += w;
        acc.x += w * v[j].x; acc.y += w * v[j].y; acc.z += w * v[j].z; acc.w += w * v[j].w;
      }
      M = mn;
    }
    const bool any = M != -INFINITY && L > 0.f;
    const float inv = any ? 1.f / L : 0.f;
    const int64_t qrow = u.qo_begin + i;
    uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + (qrow * Hq + head) * DV + 4 * d4);
    dst[0] = pack_out2(acc.x * inv, acc.y * inv, p.out_f16);
    dst[1] = pack_out2(acc.z * inv, acc.w * inv, p.out_f16);
    if (d4 == 0 && p.lse) p.lse[qrow * Hq + head] = any ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
}

// sM/sL: [WARPS][RB] running max (log2 domain) and sum of each warp;
// sO: [WARPS][RB][DV] each warp's un-normalised output rows;
// sFin: scratch of at least 2*RB floats + 1 int.  Run by the unit's
// WARPS * 32 threads (tid in [0, WARPS * 32)), which synchronise with `sync`.
template <int RB, int DV, int WARPS, class Sync>
__device__ __forceinline__ void finish_unit(const AttendParams& p, const WorkUnit& u,
                                            int row0, int R, const float* sM,
                                            const float* sL, const float* sO,
                                            float* sFin, int tid, Sync sync) {
  using namespace dev;
  constexpr float kLn2 = 0.69314718055994530942f;
  const int G = p.group, Hq = p.num_qo_heads;
  const bool partial = p.split && u.num_splits > 1;

  for (int idx = tid; idx < RB * (DV / 2); idx += WARPS * 32) {
    const int rr = idx / (DV / 2), d = 2 * (idx % (DV / 2));
    const int r = row0 + rr;
    if (r >= R) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, sM[w * RB + rr]);
    float L = 0.f, o0 = 0.f, o1 = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < WARPS; ++w) {
        const float mw = sM[w * RB + rr];
        const float sc = (mw == -INFINITY) ? 0.f : ex2(mw - M);
        L += sL[w * RB + rr] * sc;
        const float2 ow = *reinterpret_cast<const float2*>(sO + (w * RB + rr) * DV + d);
        o0 += ow.x * sc;
        o1 += ow.y * sc;
      }
      const float inv = p.v_scale / L;
      o0 *= inv;
      o1 *= inv;
    }
    const float lse_v = (M == -INFINITY) ? -INFINITY : (M + log2f(L)) * kLn2;
    const int i = r / G, head = u.h_kv * G + r % G;
    const int64_t qrow = u.qo_begin + i;
    if (!partial) {
      *reinterpret_cast<uint32_t*>(p.out + (qrow * Hq + head) * DV + d) =
          pack_out2(o0, o1, p.out_f16);
      if (d == 0 && p.lse) p.lse[qrow * Hq + head] = lse_v;
    } else {
      const int64_t pi = (int64_t)u.partial_base +
                         ((int64_t)i * Hq + head) * u.num_splits + u.split;
      *reinterpret_cast<float2*>(p.partial_o + pi * DV + d) = make_float2(o0, o1);
      if (d == 0) p.partial_lse[pi] = lse_v;
    }
  }
  if (!partial) return;

  merge_if_last<RB, DV, WARPS * 32, 20>(p, u, row0, R, sFin, tid, sync);
}

// The same for a CTA that is one unit (all its threads, __syncthreads).
template <int RB, int DV, int WARPS>
__device__ __forceinline__ void finish_unit(const AttendParams& p, const WorkUnit& u,
                                            int row0, int R, const float* sM,
                                            const float* sL, const float* sO,
                                            float* sFin) {
  finish_unit<RB, DV, WARPS>(p, u, row0, R, sM, sL, sO, sFin, (int)threadIdx.x,
                             [] { __syncthreads(); });
}

}  // namespace nvfp4kv
