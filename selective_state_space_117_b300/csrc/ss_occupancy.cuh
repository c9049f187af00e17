// Launch helper that sizes residency to the work: a grid of `units` equal
// blocks runs in ceil(units / (SMs * blocks_per_SM)) waves, and a last wave
// that fills only part of the GPU idles the rest of it.  The helper picks the
// blocks per SM b in [ceil(3 bmax / 4), bmax] that minimises waves * b (the time
// of the busiest SM when every resident block shares it evenly; ties go to the
// larger b) and caps residency at b by requesting dynamic shared memory.  It
// goes no lower than 3/4 of bmax: with fewer blocks an SM no longer has enough
// warps to keep its pipes busy, so its throughput drops.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <unordered_map>

namespace ssk {

struct DevInfo {
  int sms = 0;
  int smem_per_sm = 0;     // bytes of shared memory per SM
  int smem_optin = 0;      // largest per-block request allowed after opting in
};

inline bool device_info(DevInfo* out) {
  static std::mutex mu;
  static std::unordered_map<int, DevInfo> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it == cache.end()) {
    DevInfo d;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return false;
    it = cache.emplace(dev, d).first;
  }
  *out = it->second;
  return true;
}

inline int pick_blocks_per_sm(int64_t units, int sms, int bmax) {
  int best = bmax;
  int64_t best_cost = INT64_MAX;
  for (int b = bmax; b >= (3 * bmax + 3) / 4 && b >= 1; --b) {
    const int64_t slots = (int64_t)sms * b;
    const int64_t waves = (units + slots - 1) / slots;
    const int64_t cost = waves * b;
    if (cost < best_cost) {
      best_cost = cost;
      best = b;
    }
  }
  return best;
}

// Per (kernel, device): the resident-block limit and the kernel's static shared memory.
struct KernelInfo {
  int bmax = 0;
  int static_smem = 0;
};

inline bool kernel_info(const void* kernel, int threads, size_t base, KernelInfo* out) {
  static std::mutex mu;
  static std::unordered_map<const void*, KernelInfo> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache[dev].find(kernel);
  if (it == cache[dev].end()) {
    KernelInfo k;
    cudaFuncAttributes fa;
    if (base > 48 * 1024 &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)base) != cudaSuccess)
      return false;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k.bmax, kernel, threads, base) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, kernel) != cudaSuccess)
      return false;
    k.static_smem = (int)fa.sharedSizeBytes;
    it = cache[dev].emplace(kernel, k).first;
  }
  *out = it->second;
  return true;
}

// Dynamic shared memory to request so that at most the chosen number of
// blocks of `kernel` are resident per SM for a grid of `units` blocks, given
// that the kernel itself needs `base` bytes of dynamic shared memory.  On
// return *dyn >= base.  Returns false when a CUDA query or attribute call
// fails (the caller should not launch then).
inline bool balanced_smem(const void* kernel, int threads, int64_t units, size_t base, size_t* dyn) {
  *dyn = base;
  DevInfo di;
  KernelInfo ki;
  if (!device_info(&di) || !kernel_info(kernel, threads, base, &ki)) return false;
  size_t want = base;
  if (ki.bmax > 1) {
    const int b = pick_blocks_per_sm(units, di.sms, ki.bmax);
    if (b < ki.bmax) {
      constexpr int kReserved = 1024;  // per-block shared memory the runtime reserves
      const int64_t per_block = di.smem_per_sm / (b + 1) + 1;  // b + 1 blocks no longer fit
      const int64_t need = per_block - kReserved - ki.static_smem;
      if (need > (int64_t)base && need + ki.static_smem <= di.smem_optin) want = (size_t)need;
    }
  }
  // Static plus dynamic shared memory above 48 KB needs the kernel's opt-in.
  if (want + ki.static_smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)want) != cudaSuccess)
    return false;
  *dyn = want;
  return true;
}

}  // namespace ssk
