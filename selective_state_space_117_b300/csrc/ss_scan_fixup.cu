// Ring-staged fix-up pass of the chunked scan (mode kFixup), Euler input weight.
#include "ss_ring_launch.cuh"

namespace ssk {
template int launch_scan_fixup_t<false>(const ScanArgs&, bool, bool, dim3, cudaStream_t);
}  // namespace ssk
