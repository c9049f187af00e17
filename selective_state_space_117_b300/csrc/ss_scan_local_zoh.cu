// Ring-staged local pass of the chunked scan, zero-order-hold input weight.
#include "ss_ring_launch.cuh"

namespace ssk {
template int launch_scan_local_t<true>(const ScanArgs&, bool, dim3, cudaStream_t);
}  // namespace ssk
