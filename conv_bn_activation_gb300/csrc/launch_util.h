// Host-side launch helpers shared by the kernel files.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdlib>
#include <utility>

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

// Programmatic dependent launch is on unless CB_PDL=0 (read once).
inline bool pdl_enabled() {
  static const bool on = [] {
    const char* s = std::getenv("CB_PDL");
    return !(s && s[0] == '0');
  }();
  return on;
}

// The last kernel this host thread launched through launch_pdl (kernel,
// grid, block, dynamic shared memory, cluster size): read back by
// cb_last_launch for occupancy reports.
struct LaunchRecord {
  const void* kernel = nullptr;
  dim3 grid, block;
  size_t smem = 0;
  int cluster = 1;
};
inline LaunchRecord& last_launch() {
  static thread_local LaunchRecord r;
  return r;
}
inline void record_launch(const void* kernel, dim3 grid, dim3 block, size_t smem, int cluster) {
  LaunchRecord& r = last_launch();
  r.kernel = kernel;
  r.grid = grid;
  r.block = block;
  r.smem = smem;
  r.cluster = cluster;
}

// Launches `kernel` on stream s with programmatic stream serialisation: the
// kernel may be launched before the previous kernel of the stream has
// finished and must call pdl_wait() before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  record_launch(reinterpret_cast<const void*>(kernel), grid, block, smem, 1);
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_pdl for a kernel launched in clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_x);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  record_launch(reinterpret_cast<const void*>(kernel), grid, block, smem, cluster_x);
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace cb
