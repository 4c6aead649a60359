// Host-side launch helpers shared by the library's CUDA translation units (each unit keeps its own caches).
#pragma once
#include <cuda_runtime.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

namespace kvtc {

// SM count of a device, queried once per device.
static int sm_count(int device) {
  static std::atomic<int> cached[64];
  const bool slot = device >= 0 && device < 64;
  if (slot) {
    const int v = cached[device].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 148;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device);
  n = n > 0 ? n : 148;
  if (slot) cached[device].store(n, std::memory_order_relaxed);
  return n;
}

static int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev;
}

// Raise a kernel's dynamic shared-memory ceiling on the current device, once: cudaFuncSetAttribute runs only
// when a launch asks for more than the value last set for that (kernel, device).
static cudaError_t ensure_dyn_smem(const void* fn, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> set_to;
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(mu);
  size_t& cur = set_to[{fn, dev}];
  if (bytes <= cur) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) cur = bytes;
  return e;
}

}  // namespace kvtc
