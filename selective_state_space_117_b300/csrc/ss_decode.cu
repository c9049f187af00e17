// Launcher of the one-token decode step.
#include "ss_device.cuh"
#include "ss_dispatch.cuh"
#include "ss_launch.h"

namespace ssk {

template <int NT, bool BF, bool HAS_Z>
__global__ void __launch_bounds__(kThreads) decode_kernel(const DecodeArgs a) {
  using L = In<BF>;
  const int64_t d = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t b = blockIdx.y;
  if (d >= a.dim) return;
  const int N = (int)a.dstate;
  const int64_t c = b * a.dim + d;
  const float x = L::one(a.delta, c) + (a.delta_bias ? a.delta_bias[d] : 0.f);
  const float dt = a.softplus ? softplus(x) : x;
  const float uu = L::one(a.u, c);
  const float du = dt * uu;
  float* st = a.state + c * N;
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    if (n < N) {
      const float Bn = L::one(a.B, b * N + n), Cn = L::one(a.C, b * N + n);
      const float hn = fmaf(ex2(dt * (a.A[d * N + n] * kLog2e)), st[n], du * Bn);
      st[n] = hn;
      if (n & 1) acc1 = fmaf(Cn, hn, acc1); else acc0 = fmaf(Cn, hn, acc0);
    }
  }
  float yv = fmaf(a.D ? a.D[d] : 0.f, uu, acc0 + acc1);
  if (HAS_Z) yv *= silu(L::one(a.z, c));
  a.y[c] = yv;
}


int launch_decode(const DecodeArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s) {
  SSK_DISPATCH_NT(a.dstate, {
    if (bf16) {
      if (has_z) decode_kernel<NT, true, true><<<grid, kThreads, 0, s>>>(a);
      else decode_kernel<NT, true, false><<<grid, kThreads, 0, s>>>(a);
    } else {
      if (has_z) decode_kernel<NT, false, true><<<grid, kThreads, 0, s>>>(a);
      else decode_kernel<NT, false, false><<<grid, kThreads, 0, s>>>(a);
    }
  });
  return 0;
}

}  // namespace ssk
