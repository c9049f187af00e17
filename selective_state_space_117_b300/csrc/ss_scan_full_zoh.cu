// Ring-staged single-pass scan (mode kFull), zero-order-hold input weight.
#include "ss_ring_launch.cuh"

namespace ssk {
template int launch_scan_full_t<true>(const ScanArgs&, bool, bool, dim3, cudaStream_t);
}  // namespace ssk
