// host_cache.h — per-device, thread-safe caches of host-side launch set-up:
// the SM count, and the kernel attributes that cudaFuncSetAttribute sets per
// function in the current device's context.
#pragma once

#include <cuda_runtime.h>

#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

namespace lrkv {

// SM count the launch plans are made for: LRKV_SM_COUNT when set to a
// positive number (planning without a device, e.g. to size workspaces ahead
// of time; any value gives correct results, the grids follow it), else the
// current device's (0 on error).
inline int device_sm_count() {
  if (const char* env = std::getenv("LRKV_SM_COUNT")) {
    const int n = std::atoi(env);
    if (n > 0) return n;
  }
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cache[dev] = n;
  return n;
}

// Raises `func`'s dynamic shared-memory limit to at least `bytes` on the
// current device (a no-op when an earlier call set as much) and, with
// `max_shared_carveout`, asks for the largest shared-memory carveout.
inline cudaError_t ensure_kernel_smem(const void* func, int bytes, bool max_shared_carveout = false) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void*>, int> set_bytes;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_tuple(dev, func);
  auto it = set_bytes.find(key);
  if (it != set_bytes.end() && it->second >= bytes) return cudaSuccess;
  if (bytes > 48 * 1024 && (e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) !=
                               cudaSuccess)
    return e;
  if (max_shared_carveout &&
      (e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
    return e;
  set_bytes[key] = bytes;
  return cudaSuccess;
}

}  // namespace lrkv
