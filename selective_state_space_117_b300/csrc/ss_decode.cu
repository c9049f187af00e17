// Launcher of the one-token decode step.
#include "ss_device.cuh"
#include "ss_dispatch.cuh"
#include "ss_launch.h"

namespace ssk {

// One decode step.  A channel's NT states are split over NT/4 consecutive lanes,
// 4 states (one 16-byte vector) per lane, so a warp reads and writes its state
// rows as contiguous 512-byte runs.  The lanes of a channel recompute dt from
// the same broadcast loads; the readout sum crosses them with xor shuffles.
template <int NT, bool BF, bool HAS_Z>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(const DecodeArgs a) {
  using L = In<BF>;
  constexpr int G = NT / 4;                      // lanes per channel (1, 2, 4, 8 or 16)
  const int64_t gid = (int64_t)blockIdx.x * kDecodeThreads + threadIdx.x;
  const int64_t c = gid / G;                     // flattened (b, d)
  const int l = (int)(gid % G);
  if (c >= a.batch * a.dim) return;              // the lanes of a channel leave together
  const int lane = threadIdx.x & 31;
  const unsigned gmask = (G >= 32) ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
  const int N = (int)a.dstate;
  const int64_t b = c / a.dim, d = c % a.dim;
  const int n0 = 4 * l;

  const float x = L::one(a.delta, c) + (a.delta_bias ? a.delta_bias[d] : 0.f);
  const float dt = a.softplus ? softplus(x) : x;
  const float uu = L::one(a.u, c);
  const float du = dt * uu;

  float hv[4], Av[4], Bv[4], Cv[4];
  float* st = a.state + c * N + n0;
  const bool mine = n0 < N;                      // with N % 4 == 0 a lane owns 4 states or none
  if (a.vec && !mine) {
#pragma unroll
    for (int i = 0; i < 4; ++i) hv[i] = Av[i] = Bv[i] = Cv[i] = 0.f;
  } else if (a.vec) {                            // N % 4 == 0 and 16-byte aligned rows
    const float4 h4 = *reinterpret_cast<const float4*>(st);
    const float4 a4 = __ldg(reinterpret_cast<const float4*>(a.A + d * N + n0));
    hv[0] = h4.x; hv[1] = h4.y; hv[2] = h4.z; hv[3] = h4.w;
    Av[0] = a4.x; Av[1] = a4.y; Av[2] = a4.z; Av[3] = a4.w;
    if (BF) {
      const uint2 b2 = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(a.B) + b * N + n0));
      const uint2 c2 = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(a.C) + b * N + n0));
      Bv[0] = bf16_lo(b2.x); Bv[1] = bf16_hi(b2.x); Bv[2] = bf16_lo(b2.y); Bv[3] = bf16_hi(b2.y);
      Cv[0] = bf16_lo(c2.x); Cv[1] = bf16_hi(c2.x); Cv[2] = bf16_lo(c2.y); Cv[3] = bf16_hi(c2.y);
    } else {
      const float4 b4 = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.B) + b * N + n0));
      const float4 c4 = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.C) + b * N + n0));
      Bv[0] = b4.x; Bv[1] = b4.y; Bv[2] = b4.z; Bv[3] = b4.w;
      Cv[0] = c4.x; Cv[1] = c4.y; Cv[2] = c4.z; Cv[3] = c4.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool ok = n0 + i < N;
      hv[i] = ok ? st[i] : 0.f;
      Av[i] = ok ? a.A[d * N + n0 + i] : 0.f;
      Bv[i] = ok ? L::one(a.B, b * N + n0 + i) : 0.f;
      Cv[i] = ok ? L::one(a.C, b * N + n0 + i) : 0.f;
    }
  }
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    hv[i] = fmaf(ex2(dt * (Av[i] * kLog2e)), hv[i], du * Bv[i]);
    acc = fmaf(Cv[i], hv[i], acc);
  }
  if (a.vec) {
    if (mine) *reinterpret_cast<float4*>(st) = make_float4(hv[0], hv[1], hv[2], hv[3]);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (n0 + i < N) st[i] = hv[i];
  }
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(gmask, acc, off);
  if (l == 0) {
    float yv = fmaf(a.D ? a.D[d] : 0.f, uu, acc);
    if (HAS_Z) yv *= silu(L::one(a.z, c));
    a.y[c] = yv;
  }
}

int launch_decode(const DecodeArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s) {
  (void)grid;
  SSK_DISPATCH_NT(a.dstate, {
    const int64_t threads = a.batch * a.dim * (NT / 4);
    const dim3 g2((unsigned)((threads + kDecodeThreads - 1) / kDecodeThreads));
    if (bf16) {
      if (has_z) decode_kernel<NT, true, true><<<g2, kDecodeThreads, 0, s>>>(a);
      else decode_kernel<NT, true, false><<<g2, kDecodeThreads, 0, s>>>(a);
    } else {
      if (has_z) decode_kernel<NT, false, true><<<g2, kDecodeThreads, 0, s>>>(a);
      else decode_kernel<NT, false, false><<<g2, kDecodeThreads, 0, s>>>(a);
    }
  });
  return 0;
}

}  // namespace ssk
