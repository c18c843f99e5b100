// attend_tcgen05.cu -- paged NVFP4 decode / extend attention on the fifth-
// generation tensor cores (tcgen05.mma, accumulators in tensor memory),
// sm_103a.
//
// It computes what attend_tc.cu computes (page "Support NVFP4 KV cache
// decode on SM120": packed e2m1 K/V with per-16 E4M3 scale caches, unpacked
// and scaled before the QK and PV products; page "fix(attention): correct
// SM120 NVFP4 qk_correction layout, row-sum reduction, and lse": lse is the
// natural-log sum-exp of the scaled scores, written for every row):
//   s_j = sm_scale * sum_d q_d * k_hat_{j,d},  o = sum_j p_j v_hat_j / sum_j p_j.
//
// One CTA = one work unit (request, kv head, chunk of pages) x a block of N
// query rows (N = 16, 32 or 64; the G heads of the group times the query
// positions, padded).  Tiles of 128 tokens (8 pages) pass through four warp
// roles:
//  * loader (warp 9): 16-byte cp.async copies of the tile's packed rows and
//    scale rows into a ring of RS stages (any byte strides); a row's four
//    16-byte chunks are rotated by (row / 2) % 4 so that the dequant threads'
//    row reads hit distinct banks.  Completion: cp.async.mbarrier.arrive.
//  * dequant (warps 4-7, thread = token): e2m1 -> f16 (cvt.rn.f16x2.e2m1x2)
//    times the E4M3 block scale (exact in f16).  K_hat goes to tensor memory
//    (lane = token, two dims per 32-bit column): the A operand of the score
//    product.  V_hat goes to shared memory in the 128-byte-swizzled operand
//    layout.
//  * MMA (warp 8, one thread): S^T = K_hat . Q^T (M = 128 tokens, N rows,
//    K = Dk; A from tensor memory, B = Q in shared memory) into one of two
//    tensor-memory tiles; O^T += V_hat^T . P^T (M = 128 value dims, N rows,
//    K = 128 tokens; both operands MN-major in shared memory) accumulated in
//    tensor memory over the unit.  tcgen05.commit signals each product.
//  * softmax (warps 0-3, thread = token): reads its S^T row (tcgen05.ld),
//    p = 2^(x - m) written as the f16 P^T operand, per-row partial sums kept
//    per thread and added up once at the end.
// Putting the tile's tokens on the M side fills the 128-row MMA even for a
// handful of query rows.  The running row maximum m is raised only when a
// score exceeds it by more than 2^8 (or the row has none yet): then the
// exact tile maximum is taken and O and the partial sums are rescaled;
// otherwise p <= 2^8 fits f16 and no cross-thread reduction is needed.
// Every wait is bounded; a wait that runs out sets flag 0x4 and the CTA
// winds down (waiting, bounded, for its own copies and products first).
#include <cstdint>

#include <cuda_runtime.h>

#include "append_fused.cuh"
#include "device_common.cuh"
#include "epilogue.cuh"
#include "internal.h"

namespace nvfp4kv {
namespace {

using namespace dev;

constexpr int kTileTok = 128;
constexpr int kTilePages = kTileTok / kPageSize;
constexpr int kThreads = 320;  // softmax 0-3, dequant 4-7, MMA 8, loader 9
constexpr float kRaise = 8.f;  // log2 of the largest p before m is raised
constexpr uint32_t kSpin = 1u << 22;

// ---- tensor memory, tcgen05 and barrier helpers (inline PTX) -------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
// 32 lanes x 16 columns: thread i <-> lane (address lane + i)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
// Wait for outstanding tcgen05.ld and make their results the registers'
// current values for the code that follows.
template <int NR>
__device__ __forceinline__ void tmem_wait_ld(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int k = 0; k < NR; ++k) asm volatile("" : "+r"(r[k]));
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (16-byte units), descriptor version 1, swizzle mode.
constexpr uint32_t kSwz128 = 2, kSwz64 = 4, kSwz32 = 6;
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swz) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swz << 61);
}
// Instruction descriptor, kind::f16: f16 A and B, f32 D, operand majors
// (0 = K-major, 1 = MN-major), N >> 3, M >> 4.
constexpr uint32_t idesc_f16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D[tmem] (+)= A[tmem] . B[smem]
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// D[tmem] (+)= A[smem] . B[smem]
__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// one arrival on `bar` once every tcgen05 operation this thread issued is done
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}
// one arrival on `bar` once this thread's earlier cp.async copies landed
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ bool named_or(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ bool named_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
// Bounded wait; gives up early once another thread of the CTA gave up.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         uint32_t* flags) {
  for (uint32_t it = 0; it < kSpin; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
  }
  *abort = 1;
  atomicOr(flags, 0x4u);
  return false;
}
// Bounded wait that ignores the abort flag (the wind-down of copies and
// products in flight).
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity, uint32_t* flags) {
  for (uint32_t it = 0; it < kSpin; ++it)
    if (mbar_try_wait(bar, parity)) return;
  atomicOr(flags, 0x4u);
}
// order-preserving float <-> int keys (for integer max reductions)
__device__ __forceinline__ int fkey(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float funkey(int k) {
  return __int_as_float(k >= 0 ? k : k ^ 0x7FFFFFFF);
}

template <int N>
struct Tg5 {
  static constexpr int DK = 128, DV = 128;
  static constexpr int RS = 4;                          // packed stages
  static constexpr int PAGE = 1024 + 128 + 1024 + 128;  // K, K scales, V, V scales
  static constexpr int RAW = kTilePages * PAGE;
  static constexpr int VH = kTileTok * DV * 2;          // one V_hat tile (f16)
  static constexpr int PB = kTileTok * N * 2;           // one P^T tile (f16)
  static constexpr int ROWB = N * 2;                    // P bytes per token
  static constexpr uint32_t PSWZ = N == 16 ? kSwz32 : N == 32 ? kSwz64 : kSwz128;
  static constexpr int PSWB = N == 16 ? 1 : N == 32 ? 2 : 3;  // swizzle bits
  static constexpr int QB = N * DK * 2;
  static constexpr int OFF_V = 0;
  static constexpr int OFF_P = OFF_V + 2 * VH;
  static constexpr int OFF_Q = OFF_P + 2 * PB;
  static constexpr int OFF_RAW = OFF_Q + QB;
  static constexpr int OFF_MISC = OFF_RAW + RS * RAW;
  static constexpr int MISC = 8192;
  static constexpr int SMEM = OFF_MISC + MISC + 1024;  // + alignment slack
  // tensor memory columns: K_hat x2 (64 each), S^T x2 (N each), O^T (N)
  static constexpr int KCOL = 0, SCOL = 128, OCOL = 128 + 2 * N;
  static constexpr int TCOLS = (OCOL + N) <= 256 ? 256 : 512;
  static constexpr uint32_t IDESC_QK = idesc_f16(128, N, 0, 0);
  static constexpr uint32_t IDESC_PV = idesc_f16(128, N, 1, 1);
  static_assert(OFF_P % 1024 == 0 && OFF_Q % 1024 == 0 && OFF_RAW % 1024 == 0, "align");
  static_assert(RAW % 16 == 0 && OFF_MISC % 16 == 0, "align");
  static_assert(OCOL + N <= TCOLS, "tensor memory");
};

// swizzled byte offset inside a 1024-byte-aligned operand region (the
// operand layouts' 16-byte-chunk xor with address bits 7..)
template <int B>
__device__ __forceinline__ uint32_t swz(uint32_t off) {
  return off ^ (((off >> 7) & ((1u << B) - 1)) << 4);
}

template <int N>
__global__ void __launch_bounds__(kThreads, 1) attend_tcgen05_kernel(const AttendParams p) {
  using T = Tg5<N>;
  constexpr int DK = T::DK, DV = T::DV, RS = T::RS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sV = smem + T::OFF_V;
  uint8_t* sP = smem + T::OFF_P;
  uint8_t* sQ = smem + T::OFF_Q;
  uint8_t* sRaw = smem + T::OFF_RAW;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::OFF_MISC);
  uint64_t* raw_full = bars;               // [RS] loader -> dequant
  uint64_t* raw_empty = bars + RS;         // [RS] dequant -> loader
  uint64_t* kv_full = bars + 2 * RS;       // [2] dequant -> MMA
  uint64_t* kv_empty = bars + 2 * RS + 2;  // [2] MMA -> dequant
  uint64_t* s_full = bars + 2 * RS + 4;    // [2] MMA -> softmax
  uint64_t* p_full = bars + 2 * RS + 6;    // [2] softmax -> MMA
  uint64_t* pv_done = bars + 2 * RS + 8;   // [2] MMA -> softmax
  uint64_t* q_full = bars + 2 * RS + 10;   // softmax -> MMA
  uint64_t* fin = bars + 2 * RS + 11;      // MMA wind-down
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * RS + 12);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_minlim = reinterpret_cast<int*>(s_tmem + 2);
  float4* s_rowp = reinterpret_cast<float4*>(s_tmem + 4);  // [N] {f, -m_use, thr, lim}
  float* s_m = reinterpret_cast<float*>(s_rowp + N);        // [N] running max (log2)
  int* s_max = reinterpret_cast<int*>(s_m + N);             // [N] reduction keys
  float* s_delta = reinterpret_cast<float*>(s_max + N);     // [N]
  float* s_corr = s_delta + N;                              // [N]
  int* s_qamax = reinterpret_cast<int*>(s_corr + N);        // [N]
  float* s_l = reinterpret_cast<float*>(s_qamax + N);       // [4][N]
  float* s_fin = s_l + 4 * N;                               // [2N + 1]

  const WorkUnit u = p.units[blockIdx.x];
  const int G = p.group;
  const int R = G * u.qo_len;
  const int row0 = blockIdx.y * N;
  if (row0 >= R) return;  // uniform: before any barrier or tensor memory use
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = (u.num_pages + kTilePages - 1) / kTilePages;
  const int tok_end = min(u.kv_len, u.tok_begin + kPageSize * u.num_pages);

  if (tid == 0) {
    for (int s = 0; s < RS; ++s) {
      mbar_init(&raw_full[s], 32);
      mbar_init(&raw_empty[s], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&kv_full[b], 4);
      mbar_init(&kv_empty[b], 1);
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(q_full, 4);
    mbar_init(fin, 1);
    mbar_init_fence();
    *s_abort = 0;
    *s_minlim = INT32_MAX;
  }
  if (tid < N) s_qamax[tid] = 0;
  if (warp == 8) {
    tmem_alloc(s_tmem, T::TCOLS);
    tmem_relinquish();
  }
  // fused append: the step's new tokens of this unit's pages, stored before
  // any copy reads them
  if (p.new_k != nullptr) {
    const int lo = max(u.kv_len - u.qo_len, u.tok_begin), hi = tok_end;
    if (lo < hi) append_unit_tokens<DK, DV>(p, u, lo, hi, tid, kThreads);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 9) {
    // ================= loader =================
    const CacheView& c = p.cache;
    const int32_t* pidx = p.kv_indices + u.page_begin;
    const int r_lo = lane >> 2, ch = lane & 3;  // row (mod 8) and chunk of this lane
    int issued = 0;
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % RS;
      if (i >= RS) {
        const bool ok = __all_sync(0xffffffffu,
                                   wait_bar(&raw_empty[s], ((i / RS) - 1) & 1, s_abort, p.flags));
        if (!ok) break;
      }
      const int np_t = min(kTilePages, u.num_pages - i * kTilePages);
      int32_t pid = 0;
      if (lane < np_t) {
        pid = pidx[i * kTilePages + lane];
        if (pid < 0 || pid >= c.num_pages) {
          atomicOr(p.flags, 0x1u);
          pid = 0;
        }
      }
      uint8_t* st = sRaw + s * T::RAW;
#pragma unroll
      for (int q = 0; q < kTilePages; ++q) {
        const int32_t pq = __shfl_sync(0xffffffffu, pid, q);
        if (q >= np_t) break;
        uint8_t* pg = st + q * T::PAGE;
        const uint8_t* kb = c.k_data + pq * c.k_sp + u.h_kv * c.k_sh;
        const uint8_t* vb = c.v_data + pq * c.v_sp + u.h_kv * c.v_sh;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int slot = r_lo + 8 * half;  // 0..15
          const int row = 16 * q + slot;     // token of the tile
          const int pos = (ch ^ ((row >> 1) & 3)) << 4;
          cp_async_16(pg + slot * 64 + pos, kb + slot * c.k_ss + ch * 16);
          cp_async_16(pg + 1152 + slot * 64 + pos, vb + slot * c.v_ss + ch * 16);
        }
        if (lane < 16) {
          cp_async_small<8>(pg + 1024 + lane * 8,
                            c.k_sf + pq * c.ksf_sp + u.h_kv * c.ksf_sh + lane * c.ksf_ss);
        } else {
          const int sl = lane - 16;
          cp_async_small<8>(pg + 2176 + sl * 8,
                            c.v_sf + pq * c.vsf_sp + u.h_kv * c.vsf_sh + sl * c.vsf_ss);
        }
      }
      cp_async_arrive(&raw_full[s]);
      issued = i + 1;
    }
    // wind-down: every copy issued has landed before the CTA may exit
    for (int i = max(0, issued - RS); i < issued; ++i)
      drain_bar(&raw_full[i % RS], (i / RS) & 1, p.flags);
  } else if (warp >= 4 && warp < 8) {
    // ================= dequant (thread = token) =================
    const int j = tid - 128;  // token of the tile; tensor-memory lane
    const int slot = j & 15, rot = (j >> 1) & 3;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % RS, b = i & 1;
      bool ok = wait_bar(&raw_full[s], (i / RS) & 1, s_abort, p.flags);
      if (ok && i >= 2) ok = wait_bar(&kv_empty[b], ((i >> 1) - 1) & 1, s_abort, p.flags);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const bool valid = u.tok_begin + i * kTileTok + j < tok_end;
      const uint8_t* pg = sRaw + s * T::RAW + (j >> 4) * T::PAGE;
      // ---- K_hat row -> tensor memory columns [64 b, 64 b + 64) ----------
      {
        const uint2 sf = *reinterpret_cast<const uint2*>(pg + 1024 + slot * 8);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint4 w = *reinterpret_cast<const uint4*>(pg + slot * 64 + ((cc ^ rot) << 4));
          const uint32_t s2 = e4m3x2_to_f16x2(((cc < 2 ? sf.x : sf.y) >> (16 * (cc & 1))));
          const uint32_t slo = bcast_lo(s2), shi = bcast_hi(s2);
          uint32_t kr[16];
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t h[4];
            e2m1x8_to_f16x8(ww[q], h);
#pragma unroll
            for (int e = 0; e < 4; ++e) kr[4 * q + e] = hmul2(h[e], q < 2 ? slo : shi);
          }
          tmem_st16(tmem + lane_base + T::KCOL + 64 * b + 16 * cc, kr);
        }
      }
      // ---- V_hat row -> shared memory (MN-major operand layout) ---------
      {
        uint2 sf = *reinterpret_cast<const uint2*>(pg + 2176 + slot * 8);
        if (!valid) sf = make_uint2(0u, 0u);  // no stale byte can poison 0 * NaN
        uint8_t* vt = sV + b * T::VH;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint4 w =
              *reinterpret_cast<const uint4*>(pg + 1152 + slot * 64 + ((cc ^ rot) << 4));
          const uint32_t s2 = e4m3x2_to_f16x2(((cc < 2 ? sf.x : sf.y) >> (16 * (cc & 1))));
          const uint32_t slo = bcast_lo(s2), shi = bcast_hi(s2);
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t h[4];
            e2m1x8_to_f16x8(ww[q], h);
            const uint32_t sc = q < 2 ? slo : shi;
            // dims 32cc + 8q .. +7: 64-dim block cc/2, 16-byte chunk 4(cc&1)+q
            const uint32_t off = (uint32_t)(cc >> 1) * (kTileTok * 128) + (j >> 3) * 1024 +
                                 (j & 7) * 128 + (4 * (cc & 1) + q) * 16;
            *reinterpret_cast<uint4*>(vt + swz<3>(off)) =
                make_uint4(hmul2(h[0], sc), hmul2(h[1], sc), hmul2(h[2], sc), hmul2(h[3], sc));
          }
        }
      }
      tmem_wait_st();
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&kv_full[b]);
        mbar_arrive(&raw_empty[s]);
      }
    }
  } else if (warp == 8) {
    // ================= MMA issue (one thread) =================
    if (lane == 0) {
      const uint32_t q_base = smem_addr(sQ), v_base = smem_addr(sV), p_base = smem_addr(sP);
      auto qk = [&](int i) -> bool {
        const int b = i & 1;
        if (!wait_bar(&kv_full[b], (i >> 1) & 1, s_abort, p.flags)) return false;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < DK / 16; ++k) {
          const uint64_t bd =
              smem_desc(q_base + (k >> 2) * (N * 128) + (k & 3) * 32, 16, 1024, kSwz128);
          umma_ts(tmem + T::SCOL + N * b, tmem + T::KCOL + 64 * b + 8 * k, bd, T::IDESC_QK,
                  k > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[b]);
        return true;
      };
      bool ok = wait_bar(q_full, 0, s_abort, p.flags);
      tc_fence_after();
      if (ok && ntiles > 0) ok = qk(0);
      for (int i = 0; ok && i < ntiles; ++i) {
        if (i + 1 < ntiles && !qk(i + 1)) break;
        const int b = i & 1;
        if (!wait_bar(&p_full[b], (i >> 1) & 1, s_abort, p.flags)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kTileTok / 16; ++k) {
          const uint64_t ad =
              smem_desc(v_base + b * T::VH + k * 2048, kTileTok * 128, 1024, kSwz128);
          const uint64_t bd = smem_desc(p_base + b * T::PB + k * 16 * T::ROWB, T::PB,
                                        8 * T::ROWB, T::PSWZ);
          umma_ss(tmem + T::OCOL, ad, bd, T::IDESC_PV, (i > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&pv_done[b]);
        umma_commit(&kv_empty[b]);
      }
      // wind-down: every product issued has completed
      umma_commit(fin);
      drain_bar(fin, 0, p.flags);
    }
    __syncwarp();
  } else {
    // ================= softmax + epilogue (warps 0-3) =================
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    // ---- Q block: bf16 -> f16 times a power of two per row, swizzled ------
    constexpr int QCH = N * DK / 8;  // 16-byte chunks of f16
    uint4 qv[QCH / 128];
#pragma unroll
    for (int k = 0; k < QCH / 128; ++k) {
      const int ci = tid + 128 * k, r = ci / (DK / 8), c8 = ci % (DK / 8), gr = row0 + r;
      qv[k] = make_uint4(0u, 0u, 0u, 0u);
      if (gr < R)
        qv[k] = *reinterpret_cast<const uint4*>(
            p.q + (int64_t)(u.qo_begin + gr / G) * p.q_stride_tok +
            (int64_t)(u.h_kv * G + gr % G) * p.q_stride_head + c8 * 8);
      const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
      float am = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        am = fmaxf(am, fmaxf(fabsf(bf16_bits_to_f32(w[e] & 0xFFFFu)),
                             fabsf(bf16_bits_to_f32(w[e] >> 16))));
      atomicMax(&s_qamax[r], __float_as_int(am));
    }
    named_sync(1, 128);
    auto exp_of = [&](int r) {  // e with amax * 2^e in [2^14, 2^15)
      const float amax = __int_as_float(s_qamax[r]);
      int e = 0;
      if (amax > 0.f) e = 14 - (int)((__float_as_uint(amax) >> 23) & 0xFF) + 127;
      return max(-120, min(120, e));
    };
#pragma unroll
    for (int k = 0; k < QCH / 128; ++k) {
      const int ci = tid + 128 * k, r = ci / (DK / 8), c8 = ci % (DK / 8);
      const float up = __uint_as_float((uint32_t)(127 + exp_of(r)) << 23);
      const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
      uint32_t h[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        h[e] = f32x2_to_f16x2(bf16_bits_to_f32(w[e] & 0xFFFFu) * up,
                              bf16_bits_to_f32(w[e] >> 16) * up);
      const uint32_t off = (uint32_t)(c8 >> 3) * (N * 128) + (r >> 3) * 1024 + (r & 7) * 128 +
                           (c8 & 7) * 16;
      *reinterpret_cast<uint4*>(sQ + swz<3>(off)) = make_uint4(h[0], h[1], h[2], h[3]);
    }
    if (tid < N) {
      const int r = tid, gr = row0 + r;
      float4 rp;
      if (gr < R) {
        const int lim = p.causal ? (u.kv_len - u.qo_len + gr / G) : (u.kv_len - 1);
        rp = make_float4(p.qk_scale_log2 * __uint_as_float((uint32_t)(127 - exp_of(r)) << 23),
                         0.f, -INFINITY, __int_as_float(lim));
        atomicMin(s_minlim, lim);
      } else {  // padding row: every score -inf, never raises
        rp = make_float4(0.f, -INFINITY, INFINITY, __int_as_float(-1));
      }
      s_rowp[r] = rp;
      s_m[r] = -INFINITY;
    }
    fence_async_smem();
    named_sync(1, 128);
    __syncwarp();
    if (lane == 0) mbar_arrive(q_full);
    const int min_lim = *s_minlim;

    float lpart[N];
#pragma unroll
    for (int r = 0; r < N; ++r) lpart[r] = 0.f;
    bool alive = true;
    for (int i = 0; i < ntiles; ++i) {
      const int b = i & 1;
      // S(i) done also means PV(i-2) done: P buffer b is free again
      alive = named_and(1, 128, wait_bar(&s_full[b], (i >> 1) & 1, s_abort, p.flags));
      if (!alive) break;
      tc_fence_after();
      uint32_t sv[N];
#pragma unroll
      for (int c = 0; c < N / 16; ++c)
        tmem_ld16(tmem + lane_base + T::SCOL + N * b + 16 * c, sv + 16 * c);
      tmem_wait_ld<N>(sv);
      const int tile_tok0 = u.tok_begin + i * kTileTok;
      const int tok = tile_tok0 + tid;
      const bool tok_ok = tok < tok_end;
      const bool mask_rows = tile_tok0 + kTileTok - 1 > min_lim;
      float t[N];
      bool trig = false;
#pragma unroll
      for (int r = 0; r < N; ++r) {
        const float4 rp = s_rowp[r];
        float x = fmaf(__uint_as_float(sv[r]), rp.x, rp.y);
        if (!tok_ok || (mask_rows && tok > __float_as_int(rp.w))) x = -INFINITY;
        trig |= x > rp.z;
        t[r] = x;
      }
      if (named_or(1, 128, trig)) {
        // ---- raise the running maxima to the tile's exact row maxima ----
        if (tid < N) s_max[tid] = INT32_MIN;
        named_sync(1, 128);
#pragma unroll
        for (int r = 0; r < N; ++r) {
          const int k = __reduce_max_sync(0xffffffffu, fkey(t[r]));
          if (lane == 0) atomicMax(&s_max[r], k);
        }
        named_sync(1, 128);
        bool moved = false;
        if (tid < N) {
          const int r = tid;
          const float tm = funkey(s_max[r]);  // tile max, relative to the old m_use
          const float m_old = s_m[r];
          float delta = 0.f, corr = 1.f;
          if (tm != -INFINITY && (m_old == -INFINITY || tm > 0.f)) {
            const float m_use_old = (m_old == -INFINITY) ? 0.f : m_old;
            const float m_new = m_use_old + tm;
            delta = tm;
            if (m_old != -INFINITY) corr = ex2(m_old - m_new);
            s_m[r] = m_new;
            float4 rp = s_rowp[r];
            rp.y = -m_new;
            rp.z = kRaise;
            s_rowp[r] = rp;
            moved = corr != 1.f;
          }
          s_delta[r] = delta;
          s_corr[r] = corr;
        }
        const bool rescale = named_or(1, 128, moved) && i > 0;
#pragma unroll
        for (int r = 0; r < N; ++r) {
          t[r] -= s_delta[r];
          lpart[r] *= s_corr[r];
        }
        if (rescale) {  // O^T columns *= corr, once PV(i-1) is done
          alive = named_and(1, 128,
                            wait_bar(&pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, s_abort, p.flags));
          if (!alive) break;
          tc_fence_after();
          uint32_t ov[N];
#pragma unroll
          for (int c = 0; c < N / 16; ++c)
            tmem_ld16(tmem + lane_base + T::OCOL + 16 * c, ov + 16 * c);
          tmem_wait_ld<N>(ov);
#pragma unroll
          for (int r = 0; r < N; ++r)
            ov[r] = __float_as_uint(__uint_as_float(ov[r]) * s_corr[r]);
#pragma unroll
          for (int c = 0; c < N / 16; ++c)
            tmem_st16(tmem + lane_base + T::OCOL + 16 * c, ov + 16 * c);
          tmem_wait_st();
        }
      }
      // ---- p = 2^t, partial sums, P^T row of this token ----------------
      uint8_t* prow = sP + b * T::PB;
#pragma unroll
      for (int c = 0; c < N / 8; ++c) {
        uint32_t h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = ex2(t[8 * c + 2 * e]), p1 = ex2(t[8 * c + 2 * e + 1]);
          lpart[8 * c + 2 * e] += p0;
          lpart[8 * c + 2 * e + 1] += p1;
          h[e] = f32x2_to_f16x2(p0, p1);
        }
        const uint32_t off =
            (uint32_t)(tid >> 3) * (8 * T::ROWB) + (tid & 7) * T::ROWB + c * 16;
        *reinterpret_cast<uint4*>(prow + swz<T::PSWB>(off)) = make_uint4(h[0], h[1], h[2], h[3]);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[b]);
    }

    // ---- epilogue: O^T row of value dim `tid`, all rows of the block ------
    if (alive && ntiles > 0)
      alive = named_and(1, 128,
                        wait_bar(&pv_done[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, s_abort,
                                 p.flags));
    if (alive) {
      tc_fence_after();
#pragma unroll
      for (int r = 0; r < N; ++r) {
        float v = lpart[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) s_l[warp * N + r] = v;
      }
      uint32_t ov[N];
#pragma unroll
      for (int c = 0; c < N / 16; ++c) tmem_ld16(tmem + lane_base + T::OCOL + 16 * c, ov + 16 * c);
      tmem_wait_ld<N>(ov);
      named_sync(1, 128);
      constexpr float kLn2 = 0.69314718055994530942f;
      const bool partial = p.split && u.num_splits > 1;
      const int Hq = p.num_qo_heads;
#pragma unroll
      for (int r = 0; r < N; ++r) {
        const int gr = row0 + r;
        if (gr >= R) break;
        const float L = s_l[r] + s_l[N + r] + s_l[2 * N + r] + s_l[3 * N + r];
        const float m = s_m[r];
        const bool any = L > 0.f && m != -INFINITY;
        const float o = any ? __uint_as_float(ov[r]) * (p.v_scale / L) : 0.f;
        const float lse_v = any ? (m + log2f(L)) * kLn2 : -INFINITY;
        const int qi = gr / G, head = u.h_kv * G + gr % G;
        const int64_t qrow = u.qo_begin + qi;
        if (!partial) {
          p.out[(qrow * Hq + head) * DV + tid] = f32_to_bf16_bits(o);
          if (tid == 0 && p.lse) p.lse[qrow * Hq + head] = lse_v;
        } else {
          const int64_t pi = (int64_t)u.partial_base +
                             ((int64_t)qi * Hq + head) * u.num_splits + u.split;
          p.partial_o[pi * DV + tid] = o;
          if (tid == 0) p.partial_lse[pi] = lse_v;
        }
      }
      if (partial)
        merge_if_last<N, DV, 128>(p, u, row0, R, s_fin, tid, [] { named_sync(1, 128); });
    }
    tc_fence_before();
  }

  // ---- every role is done: release tensor memory -------------------------
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, T::TCOLS);
  }
}

template <int N>
bool make_tg5(AttendConfig* cfg) {
  cfg->kind = kKernelTcgen05;
  cfg->dk = 128;
  cfg->dv = 128;
  cfg->rows = N;
  cfg->warps = kThreads / 32;
  cfg->smem_bytes = Tg5<N>::SMEM;
  cfg->func = reinterpret_cast<const void*>(&attend_tcgen05_kernel<N>);
  return true;
}

}  // namespace

// tcgen05 kernel for (dk, dv) with up to `rows` query rows per CTA.
bool attend_config_tcgen05(int dk, int dv, int rows, AttendConfig* cfg) {
  if (dk != 128 || dv != 128) return false;
  if (rows <= 16) return make_tg5<16>(cfg);
  if (rows <= 32) return make_tg5<32>(cfg);
  return make_tg5<64>(cfg);
}

}  // namespace nvfp4kv
