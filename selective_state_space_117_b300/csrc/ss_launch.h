// Host-side launchers of the selective scan kernels (one translation unit per
// kernel family so the template instantiations compile in parallel).
#pragma once

#include <cuda_runtime.h>

#include "ss_types.h"

namespace ssk {

// Each returns 0 when a kernel was launched, -1 when dstate is unsupported.
// The _t templates take the discretisation (ZOH: zero-order hold) and are
// instantiated in separate files; the plain names pick one from a.zoh.
template <bool ZOH> int launch_scan_full_t(const ScanArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s);
template <bool ZOH> int launch_scan_fixup_t(const ScanArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s);
template <bool ZOH> int launch_scan_local_t(const ScanArgs& a, bool bf16, dim3 grid, cudaStream_t s);
inline int launch_scan_full(const ScanArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s) {
  return a.zoh ? launch_scan_full_t<true>(a, bf16, has_z, grid, s) : launch_scan_full_t<false>(a, bf16, has_z, grid, s);
}
inline int launch_scan_fixup(const ScanArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s) {
  return a.zoh ? launch_scan_fixup_t<true>(a, bf16, has_z, grid, s)
               : launch_scan_fixup_t<false>(a, bf16, has_z, grid, s);
}
inline int launch_scan_local(const ScanArgs& a, bool bf16, dim3 grid, cudaStream_t s) {
  return a.zoh ? launch_scan_local_t<true>(a, bf16, grid, s) : launch_scan_local_t<false>(a, bf16, grid, s);
}
int launch_carry(const ScanArgs& a, cudaStream_t s);

// The local pass over channels grouped by decay speed (ss_local_sorted.cu): one warp per
// (32 channels, batch row, chunk) for chunks 0 .. local_chunks - 1, states dropped once their
// weights underflow.  Needs N <= 16, 16-byte aligned rows (vec, vec_bc), whole 16-step tiles
// per chunk and a.perm; returns 0 when launched.
bool local_sorted_available(const ScanArgs& a, bool bf16);
int launch_local_sorted(const ScanArgs& a, bool bf16, cudaStream_t s);
// One decode step.  `reverse`: the blocks take the state's ranges in the opposite order
// (the caller alternates it from step to step so that a step first reads the part of the
// state that the previous step wrote last, which is the part most likely still in L2).
int launch_decode(const DecodeArgs& a, bool bf16, bool has_z, int reverse, cudaStream_t s);

// Backward pass (ss_bwd.cu): launch_bwd_locals (both local passes in one kernel; fills ws_S,
// ws_H and ws_G), then the forward carry (launch_carry), then launch_bwd (adjoint carry and
// main pass).  Each returns 0 when launched.
int launch_bwd_locals(const BwdArgs& a, bool bf16, bool has_z, cudaStream_t s);
int launch_bwd(const BwdArgs& a, bool bf16, bool has_z, cudaStream_t s);
// Channel tiles of the main backward kernel (its grid is tiles x chunks x batch).
int bwd_main_ctiles(int64_t dim, int64_t dstate);

// Full-sequence scan with one warp per channel (lanes split time): available for
// N <= 16, seqlen % 8 == 0 and 16-byte aligned rows (either input weight); returns 0 when launched,
// else the cudaError_t of the failed attribute call.
bool warp_scan_available(const ScanArgs& a, bool bf16);
int launch_scan_warp(const ScanArgs& a, bool bf16, bool has_z, cudaStream_t s);

// Diagnostic: one bounded mbarrier wait that runs out and records the timeout in *err.
int launch_wait_timeout(int* err, cudaStream_t s);
// Diagnostic: one debug-build index check of a span outside its array (nothing is accessed);
// records kDevBounds in *err in the SS_DEBUG_BOUNDS build, nothing in the normal one.
int launch_bounds_check(int* err, cudaStream_t s);

// Measurement: `blocks` blocks of kEx2Threads threads, each thread running kEx2Chains
// chains of `iters` ex2.approx.ftz.f32 links (ss_peak.cu); sink is written never.
constexpr int kEx2Threads = 256;
constexpr int kEx2Chains = 8;
int launch_ex2_rate(int64_t blocks, int iters, float* sink, cudaStream_t s);

// Causal depthwise conv1d (width 4) with optional SiLU; segments of a row per warp.
int launch_conv1d(const ConvArgs& a, bool bf16, bool silu_on, cudaStream_t s);
int64_t conv1d_segments(int64_t seqlen);

// TMA kernels.  tma_available says whether the shapes, alignments and driver
// allow them (mode kFull, kLocal or kFixup); the launchers return 0 when they
// launched, nonzero when a tensor map could not be built (nothing launched).
bool tma_available(const ScanArgs& a, bool bf16, int mode);
template <bool ZOH>
int launch_scan_tma_t(const ScanArgs& a, bool bf16, bool has_z, int mode, dim3 grid, cudaStream_t s);
template <bool ZOH> int launch_local_tma_t(const ScanArgs& a, bool bf16, dim3 grid, cudaStream_t s);
inline int launch_scan_tma(const ScanArgs& a, bool bf16, bool has_z, int mode, dim3 grid, cudaStream_t s) {
  return a.zoh ? launch_scan_tma_t<true>(a, bf16, has_z, mode, grid, s)
               : launch_scan_tma_t<false>(a, bf16, has_z, mode, grid, s);
}
inline int launch_local_tma(const ScanArgs& a, bool bf16, dim3 grid, cudaStream_t s) {
  return a.zoh ? launch_local_tma_t<true>(a, bf16, grid, s) : launch_local_tma_t<false>(a, bf16, grid, s);
}

}  // namespace ssk
