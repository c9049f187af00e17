// Device-side helpers of the selective scan kernels (sm_103a).
//
// Transcendentals use the PTX approximate instructions directly:
// ex2.approx (MUFU.EX2), lg2.approx and rcp.approx.  exp(x) is computed as
// ex2(x * log2(e)); A is pre-multiplied by log2(e) once per thread so that
// the per-state discretization exp(dt * A) is one FMUL and one MUFU.EX2.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ssk {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float lg2(float x) {
  float r;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float rcp(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// bf16 bit pattern (low 16 bits of `bits`) widened exactly to fp32.
__device__ __forceinline__ float bf16_lo(uint32_t bits) { return __uint_as_float(bits << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t bits) { return __uint_as_float(bits & 0xffff0000u); }

// softplus(x) = ln(1 + e^x).
//   x > 20        : x                     (the remainder ln(1 + e^-x) < 2.1e-9)
//   e^x < 1/8     : Taylor series of ln(1 + e) to e^6 (relative error < e^6/7 < 6e-7)
//   otherwise     : ln2 * log2(1 + e)     (1 + e >= 1.125, so its rounding costs < 1e-6 relative)
__device__ __forceinline__ float softplus(float x) {
  const float e = ex2(fminf(x, 20.f) * kLog2e);
  const float s = e * (1.f - e * (0.5f - e * (1.f / 3.f - e * (0.25f - e * (0.2f - e * (1.f / 6.f))))));
  const float l = lg2(1.f + e) * kLn2;
  const float r = e < 0.125f ? s : l;
  return x > 20.f ? x : r;
}

// silu(z) = z * sigmoid(z) = z / (1 + e^-z).  For z -> -inf, e^-z -> inf and rcp -> 0.
__device__ __forceinline__ float silu(float z) { return z * rcp(1.f + ex2(-z * kLog2e)); }

// Element loads from the input arrays (fp32 or bf16 bit patterns).
template <bool BF>
struct In;

template <>
struct In<false> {
  static __device__ __forceinline__ float one(const void* p, int64_t i) { return __ldg(static_cast<const float*>(p) + i); }
  // 8 consecutive elements starting at a 16-byte aligned offset i.
  static __device__ __forceinline__ void eight(const void* p, int64_t i, float (&v)[8]) {
    const float4* q = reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
    const float4 a = __ldg(q), b = __ldg(q + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

template <>
struct In<true> {
  static __device__ __forceinline__ float one(const void* p, int64_t i) {
    return bf16_lo(__ldg(static_cast<const unsigned short*>(p) + i));
  }
  static __device__ __forceinline__ void eight(const void* p, int64_t i, float (&v)[8]) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(p) + i));
    v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
    v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
  }
};

}  // namespace ssk
