// Diagnostic kernel for the failure path of the bounded waits: one thread
// waits, with the same bounded mbarrier wait the TMA and bulk-copy kernels
// use, on a barrier that nothing ever arrives on.  The wait gives up after its
// poll limit, records the timeout in the device status word and the kernel
// returns, leaving the context usable.
#include "ss_launch.h"
#include "ss_tma.cuh"

namespace ssk {

namespace {

__global__ void wait_timeout_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival completes phase 0; none is ever made
    mbar_init_fence();
    mbar_wait(&bar, 0, err);
  }
}

// The check of a span of 4 elements starting at 2 in an array of 5: outside, so the debug
// build records it.  Nothing is accessed either way.
__global__ void bounds_check_kernel(int* err) {
  if (threadIdx.x == 0) (void)span_ok(err, 2, 4, 5);
}

}  // namespace

int launch_bounds_check(int* err, cudaStream_t s) {
  bounds_check_kernel<<<1, 32, 0, s>>>(err);
  return 0;
}

int launch_wait_timeout(int* err, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(err);
  return 0;
}

}  // namespace ssk
