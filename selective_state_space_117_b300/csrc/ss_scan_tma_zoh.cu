// TMA kernels with the zero-order-hold input weight.
#include "ss_tma_launch.cuh"

namespace ssk {
template int launch_scan_tma_t<true>(const ScanArgs&, bool, bool, int, dim3, cudaStream_t);
template int launch_local_tma_t<true>(const ScanArgs&, bool, dim3, cudaStream_t);
}  // namespace ssk
