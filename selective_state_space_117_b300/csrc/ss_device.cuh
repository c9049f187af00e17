// Device-side helpers of the selective scan kernels (sm_103a).
//
// Transcendentals use the PTX approximate instructions directly
// (ex2.approx, rcp.approx: the MUFU unit).  exp(x) is computed as
// ex2(x * log2(e)); A is pre-multiplied by log2(e) once per thread so the
// per-state discretization exp(dt * A) is one multiply and one MUFU.EX2.
//
// Pairs of fp32 values travel in one 64-bit register ("f2") and are combined
// with the packed fma/mul/add.rn.f32x2 instructions of sm_100+, which issue
// two FP32 operations per instruction slot.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ssk {

constexpr float kLog2e = 1.4426950408889634f;

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

// ---------------------------------------------------------------- packed pairs

typedef unsigned long long f2;

__device__ __forceinline__ f2 pk(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float lo(f2 v) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
  return a;
}
__device__ __forceinline__ float hi(f2 v) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
  return b;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
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
};

template <>
struct In<true> {
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
};

}  // namespace ssk
