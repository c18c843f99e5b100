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
// positions, padded).  Tiles of 128 tokens (8 pages) pass through three
// roles; warp w works on tensor-memory lanes 32 (w % 4) .. + 31:
//  * dequant (warps 8-11; thread = token, both halves of the head dims; 13
//    warps in all, so every thread may hold 128 registers): each
//    thread copies its own token's packed bytes and scale bytes RS - 1 tiles
//    ahead (cp.async groups, no cross-thread hand-off), then e2m1 -> f16
//    (cvt.rn.f16x2.e2m1x2) times the E4M3 block scale (exact in f16).  K_hat
//    goes to tensor memory (lane = token, two dims per 32-bit column): the A
//    operand of the score product.  V_hat goes to shared memory in the
//    128-byte-swizzled operand layout.  Three K_hat / V_hat buffers.
//  * softmax (warps 0-7; thread = token for S^T, = value dim for O^T, one
//    half of the query-row columns): tcgen05.ld of its S^T row, p = 2^(x - m)
//    written as the f16 P^T operand.
//  * product issue (warp 12, one thread): S^T = K_hat . Q^T (M = 128 tokens,
//    N rows, K = Dk; A from tensor memory, B = Q in shared memory) into one
//    of two tensor-memory tiles, and O^T += V_hat^T . P^T (M = 128 value
//    dims, N rows, K = 128 tokens; both operands MN-major in shared memory)
//    accumulated in tensor memory over the unit, with the row sums
//    l += 1^T . P^T beside it (A = a block of ones in tensor memory), each as
//    soon as its inputs are ready; tcgen05.commit signals them on mbarriers.  One thread can
//    issue a product about every 54 cycles, whatever N, so this layout suits
//    many query rows per kv head (extend); decode keeps the mma.sync kernel.
// Putting the tile's tokens on the M side fills the 128-row MMA even for a
// handful of query rows.  The running row maximum m is raised only when a
// score exceeds it by more than 2^8 (or the row has none yet): then the
// exact tile maximum is taken and O and the partial sums are rescaled;
// otherwise p <= 2^8 fits f16 and no cross-thread reduction is needed.
// Every wait is bounded; a wait that runs out sets flag 0x4 and the CTA
// winds down (its copies and products in flight complete first).
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
constexpr int kThreads = 416;  // softmax warps 0-7, dequant warps 8-11, issue warp 12
constexpr int kKB = 3;         // K_hat / V_hat buffers
constexpr float kRaise = 8.f;  // log2 of the largest p before m is raised
// Wait bounds (the defaults give up after about a second; a test build
// shortens them to about a millisecond).
#ifndef NVFP4KV_TG5_SLEEP_NS
#define NVFP4KV_TG5_SLEEP_NS 20000
#endif
#ifndef NVFP4KV_TG5_POLLS
#define NVFP4KV_TG5_POLLS 50000
#endif
#ifndef NVFP4KV_TG5_IDLE_POLLS
#define NVFP4KV_TG5_IDLE_POLLS (1u << 21)
#endif
// Test build only: the first dequant warp of CTA (0, 0) withholds its arrival
// for the first tile, so the product issuer's bounded wait runs out and the
// CTA takes the abort path (flag 0x4, every wait returns, the kernel ends).
#ifndef NVFP4KV_TG5_TEST_SKIP_ARRIVE
#define NVFP4KV_TG5_TEST_SKIP_ARRIVE 0
#endif
constexpr uint32_t kSleepNs = NVFP4KV_TG5_SLEEP_NS;  // suspend hint of one poll
constexpr uint32_t kPolls = NVFP4KV_TG5_POLLS;       // polls before a wait gives up
constexpr uint32_t kIdlePolls = NVFP4KV_TG5_IDLE_POLLS;  // idle rounds of the issuer

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
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
// NC consecutive columns (a multiple of 8) of this thread's lane
template <int NC>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t* r) {
  static_assert(NC % 8 == 0, "columns");
  if constexpr (NC % 16 == 0) {
#pragma unroll
    for (int c = 0; c < NC / 16; ++c) tmem_ld16(taddr + 16 * c, r + 16 * c);
  } else {
#pragma unroll
    for (int c = 0; c < NC / 8; ++c) tmem_ld8(taddr + 8 * c, r + 8 * c);
  }
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
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
template <int NC>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t* r) {
  static_assert(NC % 8 == 0, "columns");
  if constexpr (NC % 16 == 0) {
#pragma unroll
    for (int c = 0; c < NC / 16; ++c) tmem_st16(taddr + 16 * c, r + 16 * c);
  } else {
#pragma unroll
    for (int c = 0; c < NC / 8; ++c) tmem_st8(taddr + 8 * c, r + 8 * c);
  }
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
// non-blocking test of a phase
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
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
// One poll that may suspend the thread until the phase completes (or the
// hinted time, in ns, elapses): waiting warps sleep instead of spinning and
// leave the issue slots to the warps that work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kSleepNs)
      : "memory");
  return ok != 0;
}
// Bounded wait (at least kPolls polls, at most kPolls * kSleepNs ns); gives
// up early once another thread of the CTA gave up.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         uint32_t* flags) {
  for (uint32_t it = 0; it < kPolls; ++it) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (*abort) return false;
  }
  *abort = 1;
  atomicOr(flags, 0x4u);
  return false;
}
// Bounded wait that ignores the abort flag (the wind-down of copies and
// products in flight).
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity, uint32_t* flags) {
  for (uint32_t it = 0; it < kPolls; ++it)
    if (mbar_try_wait_sleep(bar, parity)) return;
  atomicOr(flags, 0x4u);
}
// max of three floats in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
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
  static constexpr int NH = N / 2;                    // columns per softmax thread
  static constexpr int RS = N == 64 ? 3 : 4;          // copy stages per dequant thread
  static constexpr int WST = 2304;                    // one dequant warp's stage
  static constexpr int STAGE = 8 * WST;               // 8 pages of K, V and scales
  static constexpr int VH = kTileTok * DV * 2;        // one V_hat tile (f16)
  static constexpr int PB = kTileTok * N * 2;         // one P^T tile (f16)
  static constexpr int ROWB = N * 2;                  // P bytes per token
  static constexpr uint32_t PSWZ = N == 16 ? kSwz32 : N == 32 ? kSwz64 : kSwz128;
  static constexpr int PSWB = N == 16 ? 1 : N == 32 ? 2 : 3;  // swizzle bits
  static constexpr int QB = N * DK * 2;
  static constexpr int OFF_V = 0;
  static constexpr int OFF_P = OFF_V + kKB * VH;
  static constexpr int OFF_Q = OFF_P + 2 * PB;
  static constexpr int OFF_RAW = OFF_Q + QB;
  static constexpr int OFF_MISC = OFF_RAW + RS * STAGE;
  static constexpr int MISC = 8192;
  static constexpr int SMEM = OFF_MISC + MISC + 1024;  // + alignment slack
  // tensor memory columns: K_hat x3 (64 each), S^T x2 (N each), O^T (N),
  // row sums (N; every lane holds them), a 128 x 16 block of f16 ones (8)
  static constexpr int KCOL = 0, SCOL = 64 * kKB, OCOL = SCOL + 2 * N, LCOL = OCOL + N;
  static constexpr int ONES = LCOL + N;
  static constexpr int TCOLS = (ONES + 8) <= 256 ? 256 : 512;
  static constexpr uint32_t IDESC_QK = idesc_f16(128, N, 0, 0);
  static constexpr uint32_t IDESC_PV = idesc_f16(128, N, 1, 1);
  static constexpr uint32_t IDESC_L = idesc_f16(128, N, 0, 1);
  static_assert(OFF_P % 1024 == 0 && OFF_Q % 1024 == 0 && OFF_RAW % 1024 == 0, "align");
  static_assert(STAGE % 1024 == 0 && OFF_MISC % 16 == 0, "align");
  static_assert(ONES + 8 <= TCOLS, "tensor memory");
  static_assert(SMEM <= 232448, "shared memory");
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
  constexpr int DK = T::DK, DV = T::DV, RS = T::RS, NH = T::NH;
  constexpr int CW = NH < 16 ? NH : 16;  // columns per softmax chunk
  constexpr int NCH = NH / CW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sV = smem + T::OFF_V;
  uint8_t* sP = smem + T::OFF_P;
  uint8_t* sQ = smem + T::OFF_Q;
  uint8_t* sRaw = smem + T::OFF_RAW;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::OFF_MISC);
  uint64_t* kv_full = bars;        // [3] dequant -> MMA issue
  uint64_t* kv_empty = bars + 3;   // [3] PV done -> dequant
  uint64_t* s_full = bars + 6;     // [2] QK done -> softmax
  uint64_t* p_full = bars + 8;     // [2] softmax -> MMA issue
  uint64_t* pv_done = bars + 10;   // [2] PV done -> softmax
  uint64_t* q_full = bars + 12;    // Q block ready -> MMA issue
  uint64_t* fin = bars + 13;       // wind-down of the products
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_minlim = reinterpret_cast<int*>(s_tmem + 2);
  // per query-row column: score factor, -m_use, raise threshold, causal limit
  float* s_f = reinterpret_cast<float*>(s_tmem + 4);
  float* s_nm = s_f + N;
  float* s_thr = s_nm + N;
  int* s_lim = reinterpret_cast<int*>(s_thr + N);
  float* s_m = reinterpret_cast<float*>(s_lim + N);     // running max (log2)
  int* s_max = reinterpret_cast<int*>(s_m + N);         // reduction keys, then shifts
  float* s_corr = reinterpret_cast<float*>(s_max + N);
  int* s_qamax = reinterpret_cast<int*>(s_corr + N);
  float* s_fin = reinterpret_cast<float*>(s_qamax + N);  // [2N + 1]

  const WorkUnit u = load_unit(p);
  const int G = p.group;
  const int R = G * u.qo_len;
  const int row0 = blockIdx.y * N;
  if (row0 >= R) return;  // uniform: before any barrier or tensor memory use
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3;                        // tensor-memory lane quarter
  const int j = 32 * q4 + lane;                   // token of the tile / value dim
  const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
  const int unit_tok = p.page_size * u.num_pages;  // tokens the unit's pages hold
  const int ntiles = (unit_tok + kTileTok - 1) / kTileTok;
  const int tok_end = min(u.kv_len, u.tok_begin + unit_tok);

  if (tid == 0) {
    for (int b = 0; b < kKB; ++b) {
      mbar_init(&kv_full[b], 4);
      mbar_init(&kv_empty[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 8);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(q_full, 8);
    mbar_init(fin, 1);
    mbar_init_fence();
    *s_abort = 0;
    *s_minlim = INT32_MAX;
  }
  if (tid < N) s_qamax[tid] = 0;
  if (warp == 0) {
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

  if (warp >= 8 && warp < 12) {
    // ================= dequant (thread = token, all head dims) ===========
    const CacheView& c = p.cache;
    // this thread's token j of tile t: page rel / page_size, slot rel % page_size
    // stage layout per (warp, half hd of the dims): K chunks [2][32][16], V
    // chunks [2][32][16], K scales [32][4], V scales [32][4]
    auto wst = [&](int hd) { return sRaw + (4 * hd + q4) * T::WST; };
    // page id of this thread's token in tile t (-1 past the unit), loaded one
    // tile before its copies are issued
    auto load_pid = [&](int t) -> int32_t {
      const int pg = (t * kTileTok + j) / p.page_size;
      return (t < ntiles && pg < u.num_pages) ? __ldg(p.kv_indices + u.page_begin + pg) : -1;
    };
    auto issue = [&](int t, int32_t pid) {
      const int rel = t * kTileTok + j;
      const int pg = rel / p.page_size, slot = rel % p.page_size;
      if (pg >= u.num_pages) return;
      if (pid < 0 || pid >= c.num_pages) {
        atomicOr(p.flags, 0x1u);
        pid = 0;
      }
      const uint8_t* kr = c.k_data + pid * c.k_sp + u.h_kv * c.k_sh + slot * c.k_ss;
      const uint8_t* vr = c.v_data + pid * c.v_sp + u.h_kv * c.v_sh + slot * c.v_ss;
      const uint8_t* ks = c.k_sf + pid * c.ksf_sp + u.h_kv * c.ksf_sh + slot * c.ksf_ss;
      const uint8_t* vs = c.v_sf + pid * c.vsf_sp + u.h_kv * c.vsf_sh + slot * c.vsf_ss;
#pragma unroll
      for (int hd = 0; hd < 2; ++hd) {
        uint8_t* st = wst(hd) + (t % RS) * T::STAGE;
        cp_async_16(st + lane * 16, kr + 32 * hd);
        cp_async_16(st + 512 + lane * 16, kr + 32 * hd + 16);
        cp_async_16(st + 1024 + lane * 16, vr + 32 * hd);
        cp_async_16(st + 1536 + lane * 16, vr + 32 * hd + 16);
        cp_async_small<4>(st + 2048 + lane * 4, ks + 4 * hd);
        cp_async_small<4>(st + 2176 + lane * 4, vs + 4 * hd);
      }
    };
#pragma unroll
    for (int t = 0; t < RS - 1; ++t) {
      if (t < ntiles) issue(t, load_pid(t));
      cp_async_commit();
    }
    int32_t pid_next = load_pid(RS - 1);
    for (int i = 0; i < ntiles; ++i) {
      const int32_t pid = pid_next;
      pid_next = load_pid(i + RS);
      if (i + RS - 1 < ntiles) issue(i + RS - 1, pid);
      cp_async_commit();
      cp_async_wait<RS - 1>();  // this thread's copies of tile i landed
      const int bi = i % kKB;
      if (i >= kKB) {
        // one lane polls; the others sleep in the shuffle
        bool ok = true;
        if (lane == 0) ok = wait_bar(&kv_empty[bi], ((i / kKB) - 1) & 1, s_abort, p.flags);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      tc_fence_after();
      const bool valid = u.tok_begin + i * kTileTok + j < tok_end;
#pragma unroll
      for (int hd = 0; hd < 2; ++hd) {
      const uint8_t* st = wst(hd) + (i % RS) * T::STAGE;
      // ---- K_hat: tensor memory columns 64 bi + 32 hd + [0, 32) -----------
      {
        const uint32_t sf = *reinterpret_cast<const uint32_t*>(st + 2048 + lane * 4);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const uint4 w = *reinterpret_cast<const uint4*>(st + cc * 512 + lane * 16);
          const uint32_t s2 = e4m3x2_to_f16x2(sf >> (16 * cc));
          const uint32_t slo = bcast_lo(s2), shi = bcast_hi(s2);
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
          uint32_t kr[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t h[4];
            e2m1x8_to_f16x8(ww[q], h);
#pragma unroll
            for (int e = 0; e < 4; ++e) kr[4 * q + e] = hmul2(h[e], q < 2 ? slo : shi);
          }
          tmem_st16(tmem + lane_base + T::KCOL + 64 * bi + 32 * hd + 16 * cc, kr);
        }
      }
      // ---- V_hat: shared memory, 64-dim block hd (MN-major operand) -------
      {
        // no stale scale byte of a slot past the end can poison 0 * NaN
        const uint32_t sf = valid ? *reinterpret_cast<const uint32_t*>(st + 2176 + lane * 4) : 0u;
        uint8_t* vt = sV + bi * T::VH + hd * (kTileTok * 128);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const uint4 w = *reinterpret_cast<const uint4*>(st + 1024 + cc * 512 + lane * 16);
          const uint32_t s2 = e4m3x2_to_f16x2(sf >> (16 * cc));
          const uint32_t slo = bcast_lo(s2), shi = bcast_hi(s2);
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t h[4];
            e2m1x8_to_f16x8(ww[q], h);
            const uint32_t sc = q < 2 ? slo : shi;
            const uint32_t off = (j >> 3) * 1024 + (j & 7) * 128 + (4 * cc + q) * 16;
            *reinterpret_cast<uint4*>(vt + swz<3>(off)) =
                make_uint4(hmul2(h[0], sc), hmul2(h[1], sc), hmul2(h[2], sc), hmul2(h[3], sc));
          }
        }
      }
      }  // hd
      tmem_wait_st();
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      const bool withhold = NVFP4KV_TG5_TEST_SKIP_ARRIVE && blockIdx.x == 0 &&
                            blockIdx.y == 0 && warp == 8 && i == 0;
      if (lane == 0 && !withhold) mbar_arrive(&kv_full[bi]);
    }
    cp_async_wait<0>();
  } else if (warp == 12) {
    // ================= product issue (one thread) =========================
    if (lane == 0) {
      // descriptors of the first k-step; later k-steps advance the start
      // address field (16-byte units) by constant offsets
      const uint64_t qd0 = smem_desc(smem_addr(sQ), 16, 1024, kSwz128);
      const uint64_t vd0 = smem_desc(smem_addr(sV), kTileTok * 128, 1024, kSwz128);
      const uint64_t pd0 = smem_desc(smem_addr(sP), T::PB, 8 * T::ROWB, T::PSWZ);
      auto issue_qk = [&](int k) {
        tc_fence_after();
        const int bi = k % kKB, sb = k & 1;
        const uint32_t d = tmem + T::SCOL + N * sb, a = tmem + T::KCOL + 64 * bi;
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk)
          umma_ts(d, a + 8 * kk, qd0 + (((kk >> 2) * (N * 128) + (kk & 3) * 32) >> 4),
                  T::IDESC_QK, kk > 0 ? 1u : 0u);
        umma_commit(&s_full[sb]);
      };
      auto issue_pv = [&](int i) {
        tc_fence_after();
        const int bi = i % kKB, sb = i & 1;
        const uint64_t vd = vd0 + ((bi * T::VH) >> 4), pd = pd0 + ((sb * T::PB) >> 4);
        // O^T += V_hat^T P^T and the row sums l += 1^T P^T (A = ones)
#pragma unroll
        for (int k = 0; k < kTileTok / 16; ++k) {
          const uint64_t pk = pd + ((k * 16 * T::ROWB) >> 4);
          const uint32_t acc = (i > 0 || k > 0) ? 1u : 0u;
          umma_ss(tmem + T::OCOL, vd + ((k * 2048) >> 4), pk, T::IDESC_PV, acc);
          umma_ts(tmem + T::LCOL, tmem + T::ONES, pk, T::IDESC_L, acc);
        }
        umma_commit(&pv_done[sb]);
        umma_commit(&kv_empty[bi]);
      };
      // Issue whichever product has its inputs: S(qk) once K_hat(qk) is in
      // and S buffer qk & 1 was consumed (PV(qk - 2) issued), O += PV(pv)
      // once P(pv) is written.
      bool ok = wait_bar(q_full, 0, s_abort, p.flags);
      int qk = 0, pv = 0;
      uint32_t idle = 0;
      while (ok && pv < ntiles) {
        bool prog = false;
        if (qk < ntiles && qk < pv + 2 && mbar_test_wait(&kv_full[qk % kKB], (qk / kKB) & 1)) {
          issue_qk(qk);
          ++qk;
          prog = true;
        }
        if (pv < qk && mbar_test_wait(&p_full[pv & 1], (pv >> 1) & 1)) {
          issue_pv(pv);
          ++pv;
          prog = true;
        }
        if (prog) {
          idle = 0;
          continue;
        }
        if (*s_abort) break;
        if (++idle > kIdlePolls) {
          *s_abort = 1;
          atomicOr(p.flags, 0x4u);
          break;
        }
        __nanosleep(32);
      }
      // wind-down: every product issued has completed
      umma_commit(fin);
      drain_bar(fin, 0, p.flags);
    }
    __syncwarp();
  } else {
    // ================= softmax + epilogue (warps 0-7) =====================
    const int c0 = (warp >> 2) * NH;  // this thread's first query-row column
    // ---- Q block: bf16 -> f16 times a power of two per row, swizzled ------
    constexpr int QCH = N * DK / 8;  // 16-byte chunks of f16
    constexpr int QPT = QCH / 256;
    uint4 qv[QPT];
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
      const int ci = tid + 256 * k, r = ci / (DK / 8), c8 = ci % (DK / 8), gr = row0 + r;
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
    named_sync(3, 256);
    auto exp_of = [&](int r) {  // e with amax * 2^e in [2^14, 2^15)
      const float amax = __int_as_float(s_qamax[r]);
      int e = 0;
      if (amax > 0.f) e = 14 - (int)((__float_as_uint(amax) >> 23) & 0xFF) + 127;
      return max(-120, min(120, e));
    };
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
      const int ci = tid + 256 * k, r = ci / (DK / 8), c8 = ci % (DK / 8);
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
      if (gr < R) {
        const int lim = p.causal ? (u.kv_len - u.qo_len + gr / G) : (u.kv_len - 1);
        s_f[r] = p.qk_scale_log2 * __uint_as_float((uint32_t)(127 - exp_of(r)) << 23);
        s_nm[r] = 0.f;
        s_thr[r] = -INFINITY;  // no maximum yet: any visible score raises
        s_lim[r] = lim;
        atomicMin(s_minlim, lim);
      } else {  // padding row: every score -inf, never raises
        s_f[r] = 0.f;
        s_nm[r] = -INFINITY;
        s_thr[r] = INFINITY;
        s_lim[r] = -1;
      }
      s_m[r] = -INFINITY;
    }
    if (warp < 4) {  // the ones block of the row-sum product, lanes 32 warp ..
      uint32_t ones[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) ones[e] = 0x3C003C00u;  // f16 1.0 pairs
      tmem_st8(tmem + lane_base + T::ONES, ones);
      tmem_wait_st();
    }
    fence_async_smem();
    tc_fence_before();
    named_sync(3, 256);
    __syncwarp();
    if (lane == 0) mbar_arrive(q_full);
    const int min_lim = *s_minlim;
    const int nvalid = min(N, R - row0);  // columns that are real query rows
    const bool active = c0 < nvalid;      // warp-uniform

    // x = log2-domain score relative to the running max, -inf where masked
    // (a token past the unit's end gets garbage here: it is kept out of the
    // raise test and its p is stored as 0)
    auto scores = [&](int ch, int sb, bool mask_rows, int tok, float (&x)[CW]) {
      uint32_t sv[CW];
      tmem_ld<CW>(tmem + lane_base + T::SCOL + N * sb + c0 + ch * CW, sv);
      tmem_wait_ld<CW>(sv);
      const int cb = c0 + ch * CW;
#pragma unroll
      for (int e4 = 0; e4 < CW; e4 += 4) {
        const float4 f = *reinterpret_cast<const float4*>(s_f + cb + e4);
        const float4 nm = *reinterpret_cast<const float4*>(s_nm + cb + e4);
        const float ff[4] = {f.x, f.y, f.z, f.w}, nn[4] = {nm.x, nm.y, nm.z, nm.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          x[e4 + e] = fmaf(__uint_as_float(sv[e4 + e]), ff[e], nn[e]);
        if (mask_rows) {
          const int4 lm = *reinterpret_cast<const int4*>(s_lim + cb + e4);
          const int ll[4] = {lm.x, lm.y, lm.z, lm.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (tok > ll[e]) x[e4 + e] = -INFINITY;
        }
      }
    };

    // The two column halves (warps 0-3 and 4-7) are independent groups: each
    // votes and reduces over its own 128 threads (barrier 1 + half).  A wait
    // that runs out sets the abort flag; the loop then runs to its end with
    // every later wait returning at once, so no thread leaves a barrier
    // sequence the others still follow.
    const int gbar = 1 + (warp >> 2), gtid = tid & 127;
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      bool ok = true;
      if (lane == 0) ok = wait_bar(bar, parity, s_abort, p.flags);
      return __shfl_sync(0xffffffffu, ok, 0);
    };
    // Some column of this half has no maximum yet (then each score is tested
    // against its column's threshold, else all against kRaise at once).
    bool unset = active;  // group-uniform: every real column starts unset
    for (int i = 0; i < ntiles; ++i) {
      const int sb = i & 1;
      // S(i) done also means PV(i-2) done: P buffer sb is free again.
      warp_wait(&s_full[sb], (i >> 1) & 1);
      tc_fence_after();
      const int tile_tok0 = u.tok_begin + i * kTileTok;
      const int tok = tile_tok0 + j;
      const bool tok_ok = tok < tok_end;
      const bool mask_rows = tile_tok0 + kTileTok - 1 > min_lim;
      float x[NH];
      bool trig = false;
      if (active) {
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
          float xc[CW];
          scores(ch, sb, mask_rows, tok, xc);
          if (unset) {
            const float4* th = reinterpret_cast<const float4*>(s_thr + c0 + ch * CW);
#pragma unroll
            for (int e4 = 0; e4 < CW / 4; ++e4) {
              const float4 t4 = th[e4];
              trig |= (xc[4 * e4] > t4.x) | (xc[4 * e4 + 1] > t4.y) |
                      (xc[4 * e4 + 2] > t4.z) | (xc[4 * e4 + 3] > t4.w);
            }
          }
#pragma unroll
          for (int e = 0; e < CW; ++e) x[ch * CW + e] = xc[e];
        }
        if (!unset) {  // every real column has a maximum: one test of the largest
          float m3[(NH + 2) / 3];
#pragma unroll
          for (int e = 0; e < NH / 3; ++e) m3[e] = fmax3(x[3 * e], x[3 * e + 1], x[3 * e + 2]);
          if constexpr (NH % 3 == 1) m3[NH / 3] = x[NH - 1];
          if constexpr (NH % 3 == 2) m3[NH / 3] = fmaxf(x[NH - 2], x[NH - 1]);
          float mx = m3[0];
#pragma unroll
          for (int e = 1; e < (NH + 2) / 3; e += 2)
            mx = e + 1 < (NH + 2) / 3 ? fmax3(mx, m3[e], m3[e + 1]) : fmaxf(mx, m3[e]);
          trig = mx > kRaise;
        }
        trig = trig && tok_ok;
      }
      if (named_or(gbar, 128, trig)) {
        // ---- raise this half's running maxima to the tile's row maxima ----
        if (gtid < NH) s_max[c0 + gtid] = INT32_MIN;
        named_sync(gbar, 128);
        if (active) {  // lane e keeps column e's warp maximum: one atomic per lane
          int kk = INT32_MIN;
#pragma unroll
          for (int e = 0; e < NH; ++e) {
            const int k = __reduce_max_sync(0xffffffffu, fkey(tok_ok ? x[e] : -INFINITY));
            kk = lane == e ? k : kk;
          }
          if (lane < NH) atomicMax(&s_max[c0 + lane], kk);
        }
        named_sync(gbar, 128);
        bool moved = false;
        if (gtid < NH) {
          const int r = c0 + gtid;
          const float tm = funkey(s_max[r]);  // tile max, relative to the old m_use
          const float m_old = s_m[r];
          float corr = 1.f, delta = 0.f;
          if (tm != -INFINITY && (m_old == -INFINITY || tm > 0.f)) {
            const float m_new = (m_old == -INFINITY ? 0.f : m_old) + tm;
            if (m_old != -INFINITY) corr = ex2(m_old - m_new);
            delta = tm;
            s_m[r] = m_new;
            s_nm[r] = -m_new;
            s_thr[r] = kRaise;
            moved = corr != 1.f;
          }
          s_corr[r] = corr;
          s_max[r] = __float_as_int(delta);
        }
        const bool rescale = named_or(gbar, 128, moved) && i > 0;
        unset = named_or(gbar, 128, gtid < NH && c0 + gtid < nvalid && s_m[c0 + gtid] == -INFINITY);
#pragma unroll
        for (int e = 0; e < NH; ++e) x[e] -= __int_as_float(s_max[c0 + e]);
        if (rescale && active) {  // O^T and row-sum columns *= corr, once PV(i-1) is done
          warp_wait(&pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1);
          tc_fence_after();
#pragma unroll
          for (int blk = 0; blk < 2; ++blk)
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
              uint32_t ov[CW];
              const uint32_t oa = tmem + lane_base + (blk ? T::LCOL : T::OCOL) + c0 + ch * CW;
              tmem_ld<CW>(oa, ov);
              tmem_wait_ld<CW>(ov);
#pragma unroll
              for (int e = 0; e < CW; ++e)
                ov[e] = __float_as_uint(__uint_as_float(ov[e]) * s_corr[c0 + ch * CW + e]);
              tmem_st<CW>(oa, ov);
            }
          tmem_wait_st();
        }
      }
      // ---- p = 2^x: the P^T row segment of this token --------------------
      if (active) {
        uint8_t* pt = sP + sb * T::PB;
        auto pstore = [&](int c8, const uint32_t (&h)[4]) {
          const uint32_t off =
              (uint32_t)(j >> 3) * (8 * T::ROWB) + (j & 7) * T::ROWB + (c0 / 8 + c8) * 16;
          *reinterpret_cast<uint4*>(pt + swz<T::PSWB>(off)) = make_uint4(h[0], h[1], h[2], h[3]);
        };
        if (tok_ok) {
#pragma unroll
          for (int c8 = 0; c8 < NH / 8; ++c8) {
            uint32_t h[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              h[e] = f32x2_to_f16x2(ex2(x[8 * c8 + 2 * e]), ex2(x[8 * c8 + 2 * e + 1]));
            pstore(c8, h);
          }
        } else {  // a token past the unit's end: p = 0
          const uint32_t z[4] = {0u, 0u, 0u, 0u};
#pragma unroll
          for (int c8 = 0; c8 < NH / 8; ++c8) pstore(c8, z);
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
    }

    // ---- epilogue: O^T row of value dim j, this thread's row columns ------
    if (ntiles > 0) warp_wait(&pv_done[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1);
    {
      tc_fence_after();
      constexpr float kLn2 = 0.69314718055994530942f;
      const bool partial = p.split && u.num_splits > 1;
      const int Hq = p.num_qo_heads;
      if (active) {
        // The row sum, the normaliser and the output row of a column are the
        // same in every lane: lane e (mod CW) derives them for column e of the
        // chunk, once, and the warp reads them back by shuffle.
        const int e_l = lane & (CW - 1);
        uint16_t* const out_u = p.out + (int64_t)u.qo_begin * Hq * DV;
        float* const part_u = partial ? p.partial_o + (int64_t)u.partial_base * DV : nullptr;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
          uint32_t ov[CW], lv[CW];
          tmem_ld<CW>(tmem + lane_base + T::OCOL + c0 + ch * CW, ov);
          tmem_ld<CW>(tmem + lane_base + T::LCOL + c0 + ch * CW, lv);
          tmem_wait_ld<CW>(ov);
          tmem_wait_ld<CW>(lv);
          float L = __uint_as_float(lv[0]);
#pragma unroll
          for (int e = 1; e < CW; ++e) L = e_l == e ? __uint_as_float(lv[e]) : L;
          const int col_l = c0 + ch * CW + e_l;
          float f_l = 0.f;
          int off_l = 0;  // output row of the column, from the unit's first row
          if (col_l < nvalid) {
            const float m = s_m[col_l];
            const bool any = L > 0.f && m != -INFINITY;
            f_l = any ? p.v_scale / L : 0.f;
            const float lse_v = any ? (m + log2f(L)) * kLn2 : -INFINITY;
            const int gr = row0 + col_l, qi = gr / G, head = u.h_kv * G + gr % G;
            off_l = partial ? (qi * Hq + head) * u.num_splits + u.split : qi * Hq + head;
            if (q4 == 0 && lane < CW) {
              if (!partial) {
                if (p.lse) p.lse[(int64_t)u.qo_begin * Hq + off_l] = lse_v;
              } else {
                p.partial_lse[(int64_t)u.partial_base + off_l] = lse_v;
              }
            }
          }
#pragma unroll
          for (int e = 0; e < CW; ++e) {
            const float f = __shfl_sync(0xffffffffu, f_l, e);
            const int off = __shfl_sync(0xffffffffu, off_l, e);
            if (c0 + ch * CW + e < nvalid) {
              const float o = f != 0.f ? __uint_as_float(ov[e]) * f : 0.f;
              if (!partial)
                out_u[(int64_t)off * DV + j] = pack_out1(o, p.out_f16);
              else
                part_u[(int64_t)off * DV + j] = o;
            }
          }
        }
      }
      if (partial)
        merge_if_last<N, DV, 256, 4>(p, u, row0, R, s_fin, tid, [] { named_sync(3, 256); });
    }
    tc_fence_before();
  }

  // ---- every role is done: release tensor memory -------------------------
  __syncthreads();
  if (warp == 0) {
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
