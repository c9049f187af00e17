// Tensor-memory-accelerator (TMA) and mbarrier primitives (sm_90+ PTX, used on sm_103a).
//
// Bulk tensor copies move whole 2-D/3-D boxes between global and shared
// memory without per-thread address work: one elected thread issues them, an
// mbarrier counts the bytes of each load, and bulk-group fences track the
// stores.  Every wait on an mbarrier is bounded: after one second on the
// global timer it records an error in the caller's status word and gives up
// instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ss_device.cuh"

namespace ssk {

// A wait gives up after kWaitNs of the global timer.  A poll of an incomplete
// phase can itself suspend the thread for a few microseconds, so the limit is
// kept in time, not in polls; kMaxSpins only backs it up should the timer not
// advance.
constexpr unsigned long long kWaitNs = 1000000000ull;
constexpr int kMaxSpins = 1 << 26;

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive once and announce `bytes` of transactions for the current phase.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait until the phase with the given parity has completed.  Returns false
// (and sets *err) if it did not complete within kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (int i = 0; i < kMaxSpins; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 64) __nanosleep(128);
    if ((i & 255) == 255 && global_ns() - t0 > kWaitNs) break;
  }
  if (err) atomicOr(err, kDevTimeout);
  return false;
}

// 3-D tiled bulk load of the box at element coordinates (x, y, z) into dst,
// completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// 3-D tiled bulk store of the box at (x, y, z) from src (out-of-range parts are clipped).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(smem_addr(src))
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// All but the newest N committed bulk stores have finished reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// All but the newest N committed bulk stores are complete.
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later async-proxy reads.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Byte offset of 16-byte chunk j of row r in a tile whose rows are RB bytes
// and which TMA wrote with the swizzle mode of span RB (32, 64 or 128 bytes):
// the chunk index is XORed with address bits 7.. of the row's offset.
template <int RB>
__device__ __forceinline__ unsigned swz(int r, int j) {
  static_assert(RB == 32 || RB == 64 || RB == 128, "swizzle span");
  constexpr int kMask = RB / 16 - 1;
  const int bits = (r * RB) >> 7;
  return (unsigned)(r * RB + ((j ^ (bits & kMask)) << 4));
}

__device__ __forceinline__ void sts16(unsigned sa, float4 v) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(sa), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

// 8 consecutive elements of row r, group g (elements 8g..8g+7) of a swizzled
// input tile with RB-byte rows.
template <bool BF, int RB>
__device__ __forceinline__ typename In<BF>::Raw8 tile_row8(unsigned base, int r, int g) {
  if constexpr (BF) {
    return typename In<BF>::Raw8{lds16(base + swz<RB>(r, g))};
  } else {
    const uint4 a = lds16(base + swz<RB>(r, 2 * g)), b = lds16(base + swz<RB>(r, 2 * g + 1));
    return typename In<BF>::Raw8{
        make_float4(__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z), __uint_as_float(a.w)),
        make_float4(__uint_as_float(b.x), __uint_as_float(b.y), __uint_as_float(b.z), __uint_as_float(b.w))};
  }
}

}  // namespace ssk
