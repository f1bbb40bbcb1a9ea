// Device helpers shared by the kernels of libspec.so (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "spec.h"

namespace spec {

// ----------------------------------------------------------------------------------------
// Workspace (caller-allocated, zero-filled once; every call leaves its counters at zero):
// a 256-byte header (cross-block ticket of the GEMV call, error word at byte offset 4), the
// GEMV per-block partials, the accept per-slice sums, and the accept tickets in the last 4*B
// bytes of the buffer. The layout is built in abi.cu.
// ----------------------------------------------------------------------------------------
struct WsHeader {
  uint32_t gemv_ticket;
  uint32_t error;  // byte offset 4: error bits, set by bounded waits that gave up
  uint32_t pad[62];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

enum : uint32_t {
  ERR_GEMV_WAIT_FULL = 1u << 0,
  ERR_GEMV_WAIT_EMPTY = 1u << 1,
  ERR_GEMV_WAIT_RED = 1u << 2,
  ERR_GEMV_DRAIN = 1u << 3,
  ERR_TC_WAIT = 1u << 4,
};

// Per-block, per-row partial statistics of a GEMV tile (32 bytes).
struct GemvPartial {
  float m;        // largest finite-or--inf logit of the tile (-inf if none)
  float second;   // second largest (excluding the argmax element)
  int32_t idx;    // lowest index attaining m (global vocabulary id), -1 if none
  int32_t flags;  // bit 0: a NaN or +Inf was seen
  unsigned long long s;  // sum over the tile of rint(exp((z - m)/T) * 2^40)
  unsigned long long pad;
};
static_assert(sizeof(GemvPartial) == 32, "partial is 32 bytes");

constexpr int kMaxRows = 8;          // verify rows per GEMV call
constexpr int kAcceptSlice = 1024;   // vocabulary entries per accept block
constexpr int kAcceptThreads = 256;
constexpr float kQuantScale = 1099511627776.0f;  // 2^40: weights in [0,1] -> integer units

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ----------------------------------------------------------------------------------------
// PTX wrappers: shared-memory addresses, mbarriers, bulk (TMA) copies, timers.
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch. pdl_trigger lets the next kernel of the stream (launched with
// programmatic stream serialization) be scheduled before this one ends; pdl_wait blocks until
// every kernel this one depends on has completed and its writes are visible. A kernel calls
// pdl_wait before it touches anything an earlier kernel may write, and only reads data no
// kernel of the path writes (the weights) before it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// try_wait with a suspend-time hint: a waiting thread sleeps (up to ~hint ns, or until the
// phase completes) instead of spinning on issue slots other warps need.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase: gives up after ~limit_ns of wall time (the timer is read
// every 64 polls) and returns false; the caller records an error and stops waiting.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Packed fp32x2 arithmetic on 64-bit registers (two fp32 lanes: low word = x, high = y).
__device__ __forceinline__ void ffma2_acc(unsigned long long& acc, unsigned long long a,
                                          unsigned long long b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ unsigned long long pack2(uint32_t lo, uint32_t hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ float sum2(unsigned long long v) {
  uint32_t lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
  return __uint_as_float(lo) + __uint_as_float(hi);
}
__device__ __forceinline__ void lds128_b64(const void* p, unsigned long long& a,
                                           unsigned long long& b) {
  asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(smem_u32(p)));
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

// ----------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC'11): ten rounds of (x0,x1,x2,x3) -> (hi(M1*x2)^x1^k0, lo(M1*x2), hi(M0*x0)^x3^k1,
// lo(M0*x0)) with the Weyl key schedule between rounds. Only word 0 is used.
// ----------------------------------------------------------------------------------------
enum : uint32_t { PURPOSE_DRAFT = 1, PURPOSE_ACCEPT = 2, PURPOSE_RESIDUAL = 3, PURPOSE_BONUS = 4 };

__device__ __forceinline__ uint32_t philox_word0(uint64_t seed, int64_t pos, uint32_t purpose) {
  uint32_t x0 = static_cast<uint32_t>(static_cast<uint64_t>(pos));
  uint32_t x1 = static_cast<uint32_t>(static_cast<uint64_t>(pos) >> 32);
  uint32_t x2 = 0u, x3 = purpose;
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * x0, hi0 = __umulhi(0xD2511F53u, x0);
    const uint32_t lo1 = 0xCD9E8D57u * x2, hi1 = __umulhi(0xCD9E8D57u, x2);
    x0 = hi1 ^ x1 ^ k0;
    x1 = lo1;
    x2 = hi0 ^ x3 ^ k1;
    x3 = lo0;
  }
  return x0;
}

// 24-bit uniform integer (u = u24 * 2^-24) and its float value (exact in fp32).
__device__ __forceinline__ uint32_t uniform_u24(uint64_t seed, int64_t pos, uint32_t purpose) {
  return philox_word0(seed, pos, purpose) >> 8;
}
__device__ __forceinline__ float u24_to_float(uint32_t u24) {
  return static_cast<float>(u24) * 5.9604644775390625e-08f;  // 2^-24
}

// floor(u24 * total / 2^24) with a 128-bit intermediate: the integer target of an inverse-CDF
// draw over integer weights summing to `total` (always < total when total > 0).
__device__ __forceinline__ unsigned long long cdf_target(uint32_t u24, unsigned long long total) {
  const unsigned long long lo = static_cast<unsigned long long>(u24) * total;
  const unsigned long long hi = __umul64hi(static_cast<unsigned long long>(u24), total);
  return (hi << 40) | (lo >> 24);
}

// Quantise a weight in [0, 1] to integer units of 2^-40, rounded to nearest (ties to even),
// without a 64-bit conversion instruction (those run on the narrow FP64 path): x = w * 2^40 is
// exact in fp32; below 2^23 adding 2^23 rounds x to an integer held in the low significand
// bits; from 2^23 up x is already an integer, rebuilt from its significand and exponent. Zero,
// negative inputs, NaN and x >= 2^41 (none of which the callers produce) give 0.
__device__ __forceinline__ unsigned long long quantise(float w) {
  const float x = __fmul_rn(w, kQuantScale);
  const uint32_t small = __float_as_uint(__fadd_rn(x, 8388608.f)) - 0x4B000000u;
  const uint32_t b = __float_as_uint(x);
  const unsigned long long big = static_cast<unsigned long long>((b & 0x7FFFFFu) | 0x800000u)
                                 << (((b >> 23) - 150u) & 63u);
  // both forms are computed and one is selected: no divergent branch per element
  return (x < 8388608.f) ? ((x > 0.f) ? small : 0ull) : ((x < 2199023255552.f) ? big : 0ull);
}

// ----------------------------------------------------------------------------------------
// Argmax / second-max combine with ties to the lowest index.
// ----------------------------------------------------------------------------------------
struct Top2 {
  float best;
  float second;
  int32_t idx;  // kNoIndex when empty
};
constexpr int32_t kNoIndex = 0x7fffffff;

__device__ __forceinline__ Top2 top2_empty() { return Top2{-INFINITY, -INFINITY, kNoIndex}; }

__device__ __forceinline__ void top2_push(Top2& t, float v, int32_t i) {
  if (v > t.best || (v == t.best && i < t.idx)) {
    t.second = fmaxf(t.second, t.best);
    t.best = v;
    t.idx = i;
  } else {
    t.second = fmaxf(t.second, v);
  }
}

__device__ __forceinline__ Top2 top2_merge(const Top2& a, const Top2& b) {
  const bool a_wins = (a.best > b.best) || (a.best == b.best && a.idx < b.idx);
  if (a_wins) return Top2{a.best, fmaxf(a.second, b.best), a.idx};
  return Top2{b.best, fmaxf(b.second, a.best), b.idx};
}

__device__ __forceinline__ Top2 warp_top2(Top2 t) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Top2 u;
    u.best = __shfl_xor_sync(0xffffffffu, t.best, o);
    u.second = __shfl_xor_sync(0xffffffffu, t.second, o);
    u.idx = __shfl_xor_sync(0xffffffffu, t.idx, o);
    t = top2_merge(t, u);
  }
  return t;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace spec
