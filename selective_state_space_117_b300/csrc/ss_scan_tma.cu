// TMA kernels with the Euler input weight.
#include "ss_tma_launch.cuh"

namespace ssk {
template int launch_scan_tma_t<false>(const ScanArgs&, bool, bool, int, dim3, cudaStream_t);
template int launch_local_tma_t<false>(const ScanArgs&, bool, dim3, cudaStream_t);
bool tma_available(const ScanArgs& a, bool bf16, int mode) { return tma_usable(a, bf16, mode); }
}  // namespace ssk
