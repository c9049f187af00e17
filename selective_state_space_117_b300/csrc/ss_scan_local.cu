// Launchers of the chunked scan's first two phases: the zero-start local scan
// of every chunk (mode kLocal) and the carry pass across chunks.
#include "ss_dispatch.cuh"
#include "ss_kernels.cuh"
#include "ss_launch.h"

namespace ssk {

// Exclusive scan over chunks of the pairs (P_k, H_k) = (exp(A * sum_k dt), chunk end state),
// one thread per (b, d, n):  carry_0 = 0,  carry_{k+1} = P_k * carry_k + H_k.
// Overwrites ws_H[k] with carry_k (the true state entering chunk k) and writes
// the final state after the last chunk.
__global__ void __launch_bounds__(256) carry_kernel(const ScanArgs a) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t N = a.dstate;
  if (i >= a.batch * a.dim * N) return;
  const int64_t n = i % N, bd = i / N, d = bd % a.dim;
  const float A2 = a.A[d * N + n] * kLog2e;
  float H = 0.f;
  for (int64_t k = 0; k < a.nchunks; ++k) {
    const int64_t o = (bd * a.nchunks + k) * N + n;
    const float he = a.ws_H[o];
    const float S = a.ws_S[bd * a.nchunks + k];
    a.ws_H[o] = H;
    H = fmaf(ex2(A2 * S), H, he);
  }
  if (a.last_state) a.last_state[bd * N + n] = H;
}


int launch_scan_local(const ScanArgs& a, bool bf16, dim3 grid, cudaStream_t s) {
  SSK_DISPATCH_NT(a.dstate, {
    if (bf16) scan_kernel<NT, true, false, kLocal><<<grid, kThreads, 0, s>>>(a);
    else scan_kernel<NT, false, false, kLocal><<<grid, kThreads, 0, s>>>(a);
  });
  return 0;
}

int launch_carry(const ScanArgs& a, cudaStream_t s) {
  const int64_t total = a.batch * a.dim * a.dstate;
  if (total == 0) return 0;
  const int64_t blocks = (total + 255) / 256;
  carry_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
  return 0;
}

}  // namespace ssk
