// Launcher of the chunked scan's fix-up phase (mode kFixup): every chunk runs
// again from its carried-in state and writes y.
#include "ss_dispatch.cuh"
#include "ss_kernels.cuh"
#include "ss_launch.h"

namespace ssk {

int launch_scan_fixup(const ScanArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s) {
  SSK_DISPATCH_NT(a.dstate, {
    if (bf16) {
      if (has_z) scan_kernel<NT, true, true, kFixup><<<grid, kThreads, 0, s>>>(a);
      else scan_kernel<NT, true, false, kFixup><<<grid, kThreads, 0, s>>>(a);
    } else {
      if (has_z) scan_kernel<NT, false, true, kFixup><<<grid, kThreads, 0, s>>>(a);
      else scan_kernel<NT, false, false, kFixup><<<grid, kThreads, 0, s>>>(a);
    }
  });
  return 0;
}

}  // namespace ssk
