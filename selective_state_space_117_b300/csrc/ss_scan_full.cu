// Launcher of the single-pass scan (mode kFull).
#include "ss_dispatch.cuh"
#include "ss_kernels.cuh"
#include "ss_launch.h"

namespace ssk {

int launch_scan_full(const ScanArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s) {
  SSK_DISPATCH_NT(a.dstate, {
    if (bf16) {
      if (has_z) scan_kernel<NT, true, true, kFull><<<grid, kThreads, 0, s>>>(a);
      else scan_kernel<NT, true, false, kFull><<<grid, kThreads, 0, s>>>(a);
    } else {
      if (has_z) scan_kernel<NT, false, true, kFull><<<grid, kThreads, 0, s>>>(a);
      else scan_kernel<NT, false, false, kFull><<<grid, kThreads, 0, s>>>(a);
    }
  });
  return 0;
}

}  // namespace ssk
