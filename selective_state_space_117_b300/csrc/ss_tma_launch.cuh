// Launchers of the TMA kernels (forward scan in modes kFull and kFixup, local
// pass): tensor maps for u, delta, z, B, C and y, then one launch with the maps
// as grid constants.  Templated on the discretisation; each .cu file
// instantiates one.
#pragma once

#include <cudaTypedefs.h>

#include <mutex>

#include "ss_dispatch.cuh"
#include "ss_kernels_tma.cuh"
#include "ss_launch.h"
#include "ss_occupancy.cuh"

namespace ssk {

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A (batch, rows, L) row-major array as a 3-D tensor map with boxes of
// (box_t steps, box_rows rows, 1 batch row).
inline bool encode3d(CUtensorMap* m, bool bf16, bool f32_out, const void* base, int64_t L, int64_t rows, int64_t batch,
              unsigned box_t, unsigned box_rows, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int64_t es = f32_out ? 4 : (bf16 ? 2 : 4);
  const CUtensorMapDataType dt =
      (f32_out || !bf16) ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[3] = {(cuuint64_t)L, (cuuint64_t)rows, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)(L * es), (cuuint64_t)(L * es * rows)};
  cuuint32_t box[3] = {box_t, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline CUtensorMapSwizzle swizzle_for(int row_bytes) {
  return row_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                         : (row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int NT, bool BF, bool Z, int MODE, bool ZOH>
int go_tma(const ScanArgs& a, dim3 grid, cudaStream_t s) {
  using Lay = TmaLayout<NT, BF, Z>;
  TmaMaps m;
  const int64_t rows = a.dim;
  const CUtensorMapSwizzle sin = swizzle_for(Lay::RB);
  if (!encode3d(&m.u, BF, false, a.u, a.seqlen, rows, a.batch, kTmaSteps, kCh, sin) ||
      !encode3d(&m.delta, BF, false, a.delta, a.seqlen, rows, a.batch, kTmaSteps, kCh, sin) ||
      !encode3d(&m.B, BF, false, a.B, a.seqlen, a.dstate, a.batch, kTmaSteps, (unsigned)a.dstate,
                CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode3d(&m.C, BF, false, a.C, a.seqlen, a.dstate, a.batch, kTmaSteps, (unsigned)a.dstate,
                CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode3d(&m.y, BF, true, a.y, a.seqlen, rows, a.batch, kTmaSteps, kCh, swizzle_for(Lay::YB)))
    return 1;
  if (Z) {
    if (!encode3d(&m.z, BF, false, a.z, a.seqlen, rows, a.batch, kTmaSteps, kCh, sin)) return 1;
  } else {
    m.z = m.u;
  }
  auto k = scan_tma_kernel<NT, BF, Z, MODE, ZOH>;
  size_t dyn = Lay::kAlloc;
  if (!balanced_smem((const void*)k, kCh, (int64_t)grid.x * grid.y, Lay::kAlloc, &dyn)) return 1;
  k<<<grid, kCh, dyn, s>>>(a, m);
  return 0;
}

template <int NT, bool BF, bool ZOH>
int go_local_tma(const ScanArgs& a, dim3 grid, cudaStream_t s) {
  using Lay = LocalTmaLayout<NT, BF>;
  TmaMaps m;
  constexpr int RB = kTmaSteps * In<BF>::kBytes;
  const CUtensorMapSwizzle sin = swizzle_for(RB);
  if (!encode3d(&m.u, BF, false, a.u, a.seqlen, a.dim, a.batch, kTmaSteps, kCh, sin) ||
      !encode3d(&m.delta, BF, false, a.delta, a.seqlen, a.dim, a.batch, kTmaSteps, kCh, sin) ||
      !encode3d(&m.B, BF, false, a.B, a.seqlen, a.dstate, a.batch, kTmaSteps, (unsigned)a.dstate,
                CU_TENSOR_MAP_SWIZZLE_NONE))
    return 1;
  m.z = m.C = m.y = m.u;  // unused by the local pass
  auto k = local_tma_kernel<NT, BF, ZOH>;
  size_t dyn = Lay::kAlloc;
  if (!balanced_smem((const void*)k, kCh, (int64_t)grid.x * grid.y, Lay::kAlloc, &dyn)) return 1;
  k<<<grid, kCh, dyn, s>>>(a, m);
  return 0;
}

template <int MODE, bool ZOH>
int dispatch_tma(const ScanArgs& a, bool bf16, bool has_z, dim3 grid, cudaStream_t s) {
  SSK_DISPATCH_NT(a.dstate, {
    if (bf16)
      return has_z ? go_tma<NT, true, true, MODE, ZOH>(a, grid, s) : go_tma<NT, true, false, MODE, ZOH>(a, grid, s);
    return has_z ? go_tma<NT, false, true, MODE, ZOH>(a, grid, s) : go_tma<NT, false, false, MODE, ZOH>(a, grid, s);
  });
  return 1;
}

template <bool ZOH>
int launch_local_tma_t(const ScanArgs& a, bool bf16, dim3 grid, cudaStream_t s) {
  SSK_DISPATCH_NT(a.dstate, {
    return bf16 ? go_local_tma<NT, true, ZOH>(a, grid, s) : go_local_tma<NT, false, ZOH>(a, grid, s);
  });
  return 1;
}

inline bool tma_usable(const ScanArgs& a, bool bf16, int mode) {
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) % 16) == 0; };
  if (!encode_fn()) return false;
  if (a.dstate < 1 || a.dstate > 64 || a.seqlen % kGroup != 0) return false;
  if (mode != kFull && a.chunk_len % kTmaSteps != 0) return false;
  if (!al(a.u) || !al(a.delta) || !al(a.z) || !al(a.B) || !al(a.C) || !al(a.y)) return false;
  if (a.seqlen > (int64_t)INT32_MAX || a.dim > (int64_t)INT32_MAX) return false;
  (void)bf16;
  return true;
}

template <bool ZOH>
int launch_scan_tma_t(const ScanArgs& a, bool bf16, bool has_z, int mode, dim3 grid, cudaStream_t s) {
  return mode == kFixup ? dispatch_tma<kFixup, ZOH>(a, bf16, has_z, grid, s)
                        : dispatch_tma<kFull, ZOH>(a, bf16, has_z, grid, s);
}

}  // namespace ssk
