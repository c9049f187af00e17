// Device-side helpers of the selective scan kernels (sm_103a).
//
// Transcendentals use the PTX approximate instructions directly
// (ex2.approx, rcp.approx: the MUFU unit).  exp(x) is computed as
// ex2(x * log2(e)); A is pre-multiplied by log2(e) once per thread so the
// per-state discretization exp(dt * A) is one multiply and one MUFU.EX2.
//
// Pairs of fp32 values travel as float2 ("f2") in an aligned register pair and
// are combined with the packed f32x2 fma/mul/add of sm_100+ (the __ffma2_rn,
// __fmul2_rn and __fadd2_rn builtins), which issue two FP32 operations per
// instruction slot.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ss_types.h"

namespace ssk {

constexpr float kLog2e = 1.4426950408889634f;

// Index checks of the debug build.  span_ok(err, start, count, total) says whether elements
// [start, start + count) lie inside an array of `total` elements; a span outside is recorded in
// the status word (kDevBounds) and the caller then skips the accesses it guards.  Compiled
// with SS_DEBUG_BOUNDS only: in the normal build it is the constant true and the checks vanish.
__device__ __forceinline__ void record_bounds(int* err) {
  if (err) atomicOr(err, kDevBounds);
}
__device__ __forceinline__ bool span_ok(int* err, int64_t start, int64_t count, int64_t total) {
#ifdef SS_DEBUG_BOUNDS
  if (start >= 0 && count >= 0 && start <= total - count) return true;
  record_bounds(err);
  return false;
#else
  (void)err; (void)start; (void)count; (void)total;
  return true;
#endif
}

__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float rcp(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Per-thread asynchronous 16-byte copy global -> shared (L2 only), its group
// fences, and a 16-byte shared load.  All four are volatile asm statements, so
// the compiler keeps them in program order relative to each other (a ring
// slot is read only after the wait that covers its copy) while it may still
// schedule ordinary arithmetic around them.
__device__ __forceinline__ unsigned smem_addr(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void cp_async16(unsigned sa, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }
__device__ __forceinline__ uint4 lds16(unsigned sa) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(sa));
  return v;
}

// ---------------------------------------------------------------- packed pairs

typedef float2 f2;

__device__ __forceinline__ f2 pk(float lo, float hi) { return make_float2(lo, hi); }
__device__ __forceinline__ float lo(f2 v) { return v.x; }
__device__ __forceinline__ float hi(f2 v) { return v.y; }
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ f2 mul2(f2 a, f2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ f2 add2(f2 a, f2 b) { return __fadd2_rn(a, b); }
// ex2 of both halves.
__device__ __forceinline__ f2 ex2x2(f2 x) { return pk(ex2(lo(x)), ex2(hi(x))); }

// ---------------------------------------------------------------- softplus, silu

// log1p(e) / e on [0, 1]: degree-8 polynomial, coefficients from gen_log1p_poly.py
// (least squares at Chebyshev nodes); e * P(e) is within 2e-7 relative of log1p(e).
#define SSK_LOG1P_C8 0.005253457929939032f
#define SSK_LOG1P_C7 -0.02958850748836994f
#define SSK_LOG1P_C6 0.07836166769266129f
#define SSK_LOG1P_C5 -0.13674770295619965f
#define SSK_LOG1P_C4 0.19111430644989014f
#define SSK_LOG1P_C3 -0.24844369292259216f
#define SSK_LOG1P_C2 0.33319270610809326f
#define SSK_LOG1P_C1 -0.49999502301216125f

__device__ __forceinline__ float log1p_over(float e) {
  float p = SSK_LOG1P_C8;
  p = fmaf(p, e, SSK_LOG1P_C7);
  p = fmaf(p, e, SSK_LOG1P_C6);
  p = fmaf(p, e, SSK_LOG1P_C5);
  p = fmaf(p, e, SSK_LOG1P_C4);
  p = fmaf(p, e, SSK_LOG1P_C3);
  p = fmaf(p, e, SSK_LOG1P_C2);
  p = fmaf(p, e, SSK_LOG1P_C1);
  return fmaf(p, e, 1.0f);
}

__device__ __forceinline__ f2 splat(float v) { return pk(v, v); }

__device__ __forceinline__ f2 log1p_over2(f2 e) {
  f2 p = splat(SSK_LOG1P_C8);
  p = fma2(p, e, splat(SSK_LOG1P_C7));
  p = fma2(p, e, splat(SSK_LOG1P_C6));
  p = fma2(p, e, splat(SSK_LOG1P_C5));
  p = fma2(p, e, splat(SSK_LOG1P_C4));
  p = fma2(p, e, splat(SSK_LOG1P_C3));
  p = fma2(p, e, splat(SSK_LOG1P_C2));
  p = fma2(p, e, splat(SSK_LOG1P_C1));
  return fma2(p, e, splat(1.0f));
}

// softplus(x) = ln(1 + e^x) = max(x, 0) + log1p(e^-|x|): one MUFU.EX2 and a polynomial.
__device__ __forceinline__ float softplus(float x) {
  const float e = ex2(fabsf(x) * -kLog2e);
  return fmaf(e, log1p_over(e), fmaxf(x, 0.f));
}

// softplus of both halves.
__device__ __forceinline__ f2 softplus2(f2 x) {
  const float x0 = lo(x), x1 = hi(x);
  const f2 e = pk(ex2(fabsf(x0) * -kLog2e), ex2(fabsf(x1) * -kLog2e));
  return fma2(e, log1p_over2(e), pk(fmaxf(x0, 0.f), fmaxf(x1, 0.f)));
}

// silu(z) = z * sigmoid(z) = z / (1 + e^-z).  For z -> -inf, e^-z -> inf and rcp -> 0.
__device__ __forceinline__ float silu(float z) { return z * rcp(1.f + ex2(-z * kLog2e)); }

// silu of both halves.
__device__ __forceinline__ f2 silu2(f2 z) {
  const f2 d = add2(ex2x2(mul2(z, splat(-kLog2e))), splat(1.f));
  return mul2(z, pk(rcp(lo(d)), rcp(hi(d))));
}

// ---------------------------------------------------------------- zero-order hold

constexpr float kLn2 = 0.6931471805599453f;

// Input weight of the zero-order hold, (exp(dt A) - 1) / A, for a pair of states,
// given arg = dt * A * log2(e), e = exp2(arg), dt as a pair and inv_a = 1/A (0
// where A = 0).  Where |dt A| >= 1/10 it is (e - 1) / A: e carries a relative
// error of about 2^-22, so e - 1 is good to about 2.4e-7 / 0.1 = 2.4e-6 relative.
// Below, where e - 1 would cancel, it is dt * E(dt A) with E(y) = (exp(y) - 1) / y
// = 1 + y/2 + y^2/6 + y^3/24 + ..., cut after y^3 (truncation below 1e-6
// relative for |y| < 1/10; the series also gives the limit dt at A = 0).  The series
// is evaluated in arg = y / ln 2 directly (its coefficients carry the powers of ln 2),
// and the bound is taken on |arg| < 0.1 / ln 2.
constexpr float kHoldSeriesBelow = 0.1f;
constexpr float kHoldArgBelow = kHoldSeriesBelow / kLn2;

__device__ __forceinline__ f2 hold_series_arg2(f2 arg) {
  f2 p = splat(kLn2 * kLn2 * kLn2 / 24.f);
  p = fma2(p, arg, splat(kLn2 * kLn2 / 6.f));
  p = fma2(p, arg, splat(kLn2 / 2.f));
  return fma2(p, arg, splat(1.f));
}

__device__ __forceinline__ f2 hold2(f2 arg, f2 e, f2 dtp, f2 inv_a) {
  const f2 small = mul2(hold_series_arg2(arg), dtp);
  const f2 large = mul2(add2(e, splat(-1.f)), inv_a);
  return pk(fabsf(lo(arg)) < kHoldArgBelow ? lo(small) : lo(large),
            fabsf(hi(arg)) < kHoldArgBelow ? hi(small) : hi(large));
}

// The same weight when the two exponentials at the ends of the step are known:
// w_next = exp(A (R + dt)) and w_cur = exp(A R) give (w_next - w_cur) / A =
// w_cur * (exp(dt A) - 1) / A, used by the local passes.
__device__ __forceinline__ f2 hold_between2(f2 w_next, f2 w_cur, f2 arg_dt, f2 dtp, f2 inv_a) {
  const f2 small = mul2(mul2(hold_series_arg2(arg_dt), dtp), w_cur);
  const f2 large = mul2(add2(w_next, mul2(w_cur, splat(-1.f))), inv_a);
  return pk(fabsf(lo(arg_dt)) < kHoldArgBelow ? lo(small) : lo(large),
            fabsf(hi(arg_dt)) < kHoldArgBelow ? hi(small) : hi(large));
}

// ---------------------------------------------------------------- bf16

// bf16 bit pattern (low 16 bits of `bits`) widened exactly to fp32.
__device__ __forceinline__ float bf16_lo(uint32_t bits) { return __uint_as_float(bits << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t bits) { return __uint_as_float(bits & 0xffff0000u); }
// Two bf16 in one 32-bit word, widened to an fp32 pair.
__device__ __forceinline__ f2 bf16x2(uint32_t bits) { return pk(bf16_lo(bits), bf16_hi(bits)); }

// Element loads from the input arrays (fp32 or bf16 bit patterns).
template <bool BF>
struct In;

template <>
struct In<false> {
  static constexpr unsigned kBytes = 4;
  static __device__ __forceinline__ const void* addr(const void* p, int64_t i) { return static_cast<const float*>(p) + i; }
  static __device__ __forceinline__ float one(const void* p, int64_t i) { return __ldg(static_cast<const float*>(p) + i); }
  // Raw storage of 8 consecutive elements (two 16-byte loads from a 16-byte aligned offset).
  struct Raw8 { float4 a, b; };
  static __device__ __forceinline__ Raw8 load8(const void* p, int64_t i) {
    const float4* q = reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
    return Raw8{__ldg(q), __ldg(q + 1)};
  }
  // Elements (2j, 2j+1) of a Raw8, as an fp32 pair.
  static __device__ __forceinline__ f2 pair(const Raw8& r, int j) {
    const float4& q = j < 2 ? r.a : r.b;
    return (j & 1) ? pk(q.z, q.w) : pk(q.x, q.y);
  }
  static __device__ __forceinline__ Raw8 pack8(const float (&v)[8]) {
    return Raw8{make_float4(v[0], v[1], v[2], v[3]), make_float4(v[4], v[5], v[6], v[7])};
  }
  // 8 elements live in kVec 16-byte chunks; chunk v at shared address sa + v * stride_bytes.
  static constexpr int kVec = 2;
  static __device__ __forceinline__ Raw8 from_smem(unsigned sa, unsigned stride_bytes) {
    const uint4 a = lds16(sa), b = lds16(sa + stride_bytes);
    return Raw8{make_float4(__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z), __uint_as_float(a.w)),
                make_float4(__uint_as_float(b.x), __uint_as_float(b.y), __uint_as_float(b.z), __uint_as_float(b.w))};
  }
};

template <>
struct In<true> {
  static constexpr unsigned kBytes = 2;
  static __device__ __forceinline__ const void* addr(const void* p, int64_t i) {
    return static_cast<const unsigned short*>(p) + i;
  }
  static __device__ __forceinline__ float one(const void* p, int64_t i) {
    return bf16_lo(__ldg(static_cast<const unsigned short*>(p) + i));
  }
  struct Raw8 { uint4 a; };
  static __device__ __forceinline__ Raw8 load8(const void* p, int64_t i) {
    return Raw8{__ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(p) + i))};
  }
  static __device__ __forceinline__ f2 pair(const Raw8& r, int j) {
    const uint32_t w = j == 0 ? r.a.x : j == 1 ? r.a.y : j == 2 ? r.a.z : r.a.w;
    return bf16x2(w);
  }
  // Values that are exact bf16 numbers (widened by one()), back to their bit patterns.
  static __device__ __forceinline__ Raw8 pack8(const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) w[p] = (__float_as_uint(v[2 * p]) >> 16) | (__float_as_uint(v[2 * p + 1]) & 0xffff0000u);
    return Raw8{make_uint4(w[0], w[1], w[2], w[3])};
  }
  static constexpr int kVec = 1;
  static __device__ __forceinline__ Raw8 from_smem(unsigned sa, unsigned) { return Raw8{lds16(sa)}; }
};

// A per-thread ring of 8-step input groups in shared memory, filled by
// cp.async ahead of use.  Slot s holds, for each of NA input arrays, this
// thread's kVec 16-byte chunks; chunk v of array k of thread i sits at byte
// ((s * NA + k) * kVec + v) * kThreads * 16 + i * 16, so a warp's reads of one
// chunk are 512 contiguous bytes.  `src[k]` is the global address of this
// thread's group 0 of array k and `step` the byte distance between groups
// (negative to walk backward).
template <bool BF, int NA, int kThreads, int kSlots>
struct Ring {
  using L = In<BF>;
  static constexpr unsigned kChunkStride = kThreads * 16;
  static constexpr unsigned kArr = L::kVec * kChunkStride;
  static constexpr unsigned kSlot = NA * kArr;
  static constexpr unsigned kBytes = kSlots * kSlot;
  unsigned base;
  const char* src[NA];
  int64_t step;

  __device__ __forceinline__ void put(int gi) const {
    const unsigned s = base + (unsigned)(gi % kSlots) * kSlot;
    const int64_t off = (int64_t)gi * step;
#pragma unroll
    for (int k = 0; k < NA; ++k)
#pragma unroll
      for (int v = 0; v < L::kVec; ++v) cp_async16(s + k * kArr + v * kChunkStride, src[k] + off + 16 * v);
  }
  __device__ __forceinline__ typename L::Raw8 get(int gi, int k) const {
    return L::from_smem(base + (unsigned)(gi % kSlots) * kSlot + k * kArr, kChunkStride);
  }
};

}  // namespace ssk
