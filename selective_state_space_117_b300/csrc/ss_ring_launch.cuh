// Launchers of the ring-staged scan kernels (scan_kernel in modes full and
// fix-up, local_kernel), templated on the discretisation.  Each .cu file
// instantiates one family for one discretisation, so the many kernel
// instantiations compile in parallel.
#pragma once

#include "ss_dispatch.cuh"
#include "ss_kernels.cuh"
#include "ss_launch.h"
#include "ss_occupancy.cuh"

namespace ssk {

template <int NT, bool BF, bool Z, int MODE, bool ZOH>
void go_ring_scan(const ScanArgs& a, dim3 grid, cudaStream_t s) {
  auto k = scan_kernel<NT, BF, Z, MODE, ZOH>;
  size_t dyn = 0;
  balanced_smem((const void*)k, kCh, (int64_t)grid.x * grid.y, 0, &dyn);
  k<<<grid, kCh, dyn, s>>>(a);
}

template <int MODE, bool ZOH>
int launch_ring_scan(const ScanArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s) {
  SSK_DISPATCH_NT(a.dstate, {
    if (bf16) {
      if (has_z) go_ring_scan<NT, true, true, MODE, ZOH>(a, grid, s);
      else go_ring_scan<NT, true, false, MODE, ZOH>(a, grid, s);
    } else {
      if (has_z) go_ring_scan<NT, false, true, MODE, ZOH>(a, grid, s);
      else go_ring_scan<NT, false, false, MODE, ZOH>(a, grid, s);
    }
  });
  return 0;
}

template <bool ZOH>
int launch_scan_full_t(const ScanArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s) {
  return launch_ring_scan<kFull, ZOH>(a, bf16, has_z, grid, s);
}

template <bool ZOH>
int launch_scan_fixup_t(const ScanArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s) {
  return launch_ring_scan<kFixup, ZOH>(a, bf16, has_z, grid, s);
}

template <int NT, bool BF, bool ZOH>
void go_ring_local(const ScanArgs& a, dim3 grid, cudaStream_t s) {
  auto k = local_kernel<NT, BF, ZOH>;
  size_t dyn = 0;
  balanced_smem((const void*)k, kCh, (int64_t)grid.x * grid.y, 0, &dyn);
  k<<<grid, kCh, dyn, s>>>(a);
}

template <bool ZOH>
int launch_scan_local_t(const ScanArgs& a, bool bf16, dim3 grid, cudaStream_t s) {
  SSK_DISPATCH_NT(a.dstate, {
    if (bf16) go_ring_local<NT, true, ZOH>(a, grid, s);
    else go_ring_local<NT, false, ZOH>(a, grid, s);
  });
  return 0;
}

}  // namespace ssk
