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
  return launch_pdl(igemm_halo_kernel<256, 128, true>, dim3(grid), dim3(kHaloThreads), smem, s, xmap, wmap, a);
}

}  // namespace cb
