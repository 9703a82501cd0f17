// The channel-major instantiation of the halo-tile implicit GEMM
// (igemm_halo.cuh): 256 pixels x 128 output channels per tile.
#include "igemm_halo.cuh"
#include "launch_util.h"

namespace cb {

int igemm_read_trace_halo_cm(unsigned long long* out, int max_records) { return igemm_read_trace_tu(out, max_records); }

cudaError_t launch_igemm_halo_cm(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int grid,
                                 size_t smem, cudaStream_t s) {
  cudaError_t e = smem_attr_once<igemm_halo_kernel<256, 128, true>>(smem);
  if (e != cudaSuccess) return e;
  if (a.split_k == 2)
    return launch_pdl_cluster(igemm_halo_kernel<256, 128, true>, dim3(grid), dim3(kHaloThreads), smem, s, 2, xmap,
                              wmap, a);
  return launch_pdl(igemm_halo_kernel<256, 128, true>, dim3(grid), dim3(kHaloThreads), smem, s, xmap, wmap, a);
}

int halo_max_pairs_cm(size_t smem) {
  if (smem_attr_once<igemm_halo_kernel<256, 128, true>>(smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kHaloThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, igemm_halo_kernel<256, 128, true>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace cb
