// Host-side launchers of the selective scan kernels (one translation unit per
// kernel family so the template instantiations compile in parallel).
#pragma once

#include <cuda_runtime.h>

#include "ss_types.h"

namespace ssk {

// Each returns 0 when a kernel was launched, -1 when dstate is unsupported.
int launch_scan_full(const ScanArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s);
int launch_scan_local(const ScanArgs& a, bool bf16, dim3 grid, cudaStream_t s);
int launch_scan_fixup(const ScanArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s);
int launch_carry(const ScanArgs& a, cudaStream_t s);
int launch_decode(const DecodeArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s);

// Causal depthwise conv1d (width 4) with optional SiLU; segments of a row per warp.
int launch_conv1d(const ConvArgs& a, bool bf16, bool silu_on, cudaStream_t s);
int64_t conv1d_segments(int64_t seqlen);

// TMA forward scan (mode kFull or kFixup).  tma_usable says whether the
// shapes, alignments and driver allow it; launch_scan_tma returns 0 when it
// launched, nonzero when a tensor map could not be built (nothing launched).
bool tma_usable(const ScanArgs& a, bool bf16, int mode);
int launch_scan_tma(const ScanArgs& a, bool bf16, bool has_z, int mode, dim3 grid, cudaStream_t s);
// TMA local pass of the chunked scan (tma_usable with mode kLocal); same return convention.
int launch_local_tma(const ScanArgs& a, bool bf16, dim3 grid, cudaStream_t s);

}  // namespace ssk
