// Throughput of the MUFU unit's base-2 exponential (ex2.approx.ftz.f32, the
// instruction every decay exp(dt A) of the scan becomes), measured on the
// running GPU: the denominator of the roofline's exponential term.
//
// Each thread runs kEx2Chains independent chains of links x <- ex2(x) * (-1/2):
// one MUFU.EX2 and one FMUL per link.  The values stay in (-1/2, 0) (the chain
// settles near the fixed point of x = -2^x / 2), so no link underflows or
// overflows and every link is real work.  With kEx2Threads-thread blocks, several
// blocks per SM and kEx2Chains chains per thread, many more exponentials are in
// flight than the MUFU pipe's latency covers, and each exponential costs the
// issue slot of itself and of one multiply, so the pipe's throughput bounds the
// loop.  The sum of the chains is written only if it takes an impossible value,
// which keeps every link live without a store per thread.
#include "ss_launch.h"
#include "ss_device.cuh"

namespace ssk {

namespace {

__global__ void __launch_bounds__(kEx2Threads) ex2_rate_kernel(int iters, float* sink) {
  float x[kEx2Chains];
#pragma unroll
  for (int c = 0; c < kEx2Chains; ++c) x[c] = -0.25f - 1e-4f * (float)((threadIdx.x + c) & 63);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kEx2Chains; ++c) x[c] = ex2(x[c]) * -0.5f;
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kEx2Chains; ++c) s += x[c];
  if (s > 1.0f) sink[blockIdx.x] = s;   // never true: every x stays negative
}

}  // namespace

int launch_ex2_rate(int64_t blocks, int iters, float* sink, cudaStream_t s) {
  ex2_rate_kernel<<<(unsigned)blocks, kEx2Threads, 0, s>>>(iters, sink);
  return 0;
}

}  // namespace ssk
