// The carry pass across chunks, and the ring-staged local pass (local_kernel)
// with the Euler input weight.
#include "ss_ring_launch.cuh"

namespace ssk {

// Exclusive scan over chunks of the pairs (P_k, H_k) = (exp(A * S_k), chunk end state) under
// (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2), one thread per (b, d, n):
//   carry_0 = h0 (zeros without one),   carry_{k+1} = P_k * carry_k + H_k.
// Overwrites the workspace's H_k with carry_k (the true state entering chunk k) for every chunk.
// Only the chunks the local pass covered (0 .. local_chunks - 1) are combined: the forward scan
// leaves out its last chunk, whose end state is the final state that its fix-up pass writes.
// The dependent chain is latency-bound: loads run in batches of 8 chunks, and the next batch is
// requested before the current one is consumed.
__global__ void __launch_bounds__(256) carry_kernel(const ScanArgs a) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t N = a.dstate;
  if (i >= a.batch * a.dim * N) return;
  const int64_t n = i % N, bd = i / N, d = bd % a.dim;
  const float A2 = a.A[d * N + n] * kLog2e;
  const int64_t K = a.nchunks, BD = a.batch * a.dim;
  // Debug build: the column of every chunk's entry (the last one farthest out), and h0.
  if (!span_ok(a.err, (K - 1) * BD * N + bd * N + n, 1, K * BD * N) || !span_ok(a.err, (K - 1) * BD + bd, 1, K * BD))
    return;
  float* H = a.ws_H + bd * N + n;            // chunk k at H[k * BD * N]
  const float* S = a.ws_S + bd;              // chunk k at S[k * BD]
  float c = a.h0 ? a.h0[bd * N + n] : 0.f;  // the state entering chunk 0
  float he[8], sk[8], hn[8] = {}, sn[8] = {};
  auto load = [&](int64_t k0, float (&hv)[8], float (&sv)[8]) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool ok = k0 + u < K;
      hv[u] = ok ? H[(k0 + u) * BD * N] : 0.f;
      sv[u] = ok ? S[(k0 + u) * BD] : 0.f;
    }
  };
  load(0, he, sk);
  for (int64_t k0 = 0; k0 < K; k0 += 8) {
    if (k0 + 8 < K) load(k0 + 8, hn, sn);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (k0 + u < K) {
        H[(k0 + u) * BD * N] = c;
        if (k0 + u < a.local_chunks) c = fmaf(ex2(A2 * sk[u]), c, he[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      he[u] = hn[u];
      sk[u] = sn[u];
    }
  }
}

int launch_carry(const ScanArgs& a, cudaStream_t s) {
  const int64_t total = a.batch * a.dim * a.dstate;
  if (total == 0) return 0;
  const int64_t blocks = (total + 255) / 256;
  carry_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
  return 0;
}

template int launch_scan_local_t<false>(const ScanArgs&, bool, dim3, cudaStream_t);

}  // namespace ssk
