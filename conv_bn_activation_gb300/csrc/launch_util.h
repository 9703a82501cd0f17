// Host-side launch helpers shared by the kernel files.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>

namespace cb {

// Raises a kernel's dynamic shared-memory limit to at least `smem` bytes,
// calling cudaFuncSetAttribute only when this device has not been raised
// that far yet (the call costs microseconds, a launch about as much).
template <auto Kernel>
cudaError_t smem_attr_once(size_t smem) {
  constexpr int kMaxDevices = 64;
  static std::atomic<size_t> raised[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices)
    return cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (raised[dev].load(std::memory_order_acquire) >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  size_t cur = raised[dev].load(std::memory_order_relaxed);
  while (cur < smem && !raised[dev].compare_exchange_weak(cur, smem, std::memory_order_acq_rel)) {
  }
  return cudaSuccess;
}

}  // namespace cb
