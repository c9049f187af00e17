// Launcher of the single-pass scan (mode kFull).
#include "ss_dispatch.cuh"
#include "ss_kernels.cuh"
#include "ss_launch.h"
#include "ss_occupancy.cuh"

namespace ssk {

template <int NT, bool BF, bool Z>
static void go_full(const ScanArgs& a, dim3 grid, cudaStream_t s) {
  auto k = scan_kernel<NT, BF, Z, kFull>;
  size_t dyn = 0;
  balanced_smem((const void*)k, kCh, (int64_t)grid.x * grid.y, 0, &dyn);
  k<<<grid, kCh, dyn, s>>>(a);
}

int launch_scan_full(const ScanArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s) {
  SSK_DISPATCH_NT(a.dstate, {
    if (bf16) {
      if (has_z) go_full<NT, true, true>(a, grid, s);
      else go_full<NT, true, false>(a, grid, s);
    } else {
      if (has_z) go_full<NT, false, true>(a, grid, s);
      else go_full<NT, false, false>(a, grid, s);
    }
  });
  return 0;
}

}  // namespace ssk
