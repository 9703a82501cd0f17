// The bf16-operand instantiations of the halo-tile implicit GEMM
// (igemm_halo.cuh, kind::f16 MMAs): pixel-major 128 x {32, 64, 128, 256} and
// channel-major 256 x 128 tiles of 128-byte pixel rows (64 bf16 channels per
// chunk).  The 64- and 32-byte-row tiles are in igemm_halo_bf16_kc16.cu.
#include "igemm_halo.cuh"
#include "launch_util.h"

namespace cb {

cudaError_t launch_igemm_halo_bf16_narrow(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a,
                                          int co, int grid, size_t smem, cudaStream_t s);

template <int PX, int CO, bool CM>
static cudaError_t halo_launch_bf16(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int grid,
                                    size_t smem, cudaStream_t s) {
  cudaError_t e = smem_attr_once<igemm_halo_kernel<PX, CO, CM, 32, __nv_bfloat16>>(smem);
  if (e != cudaSuccess) return e;
  if (a.split_k == 2)
    return launch_pdl_cluster(igemm_halo_kernel<PX, CO, CM, 32, __nv_bfloat16>, dim3(grid), dim3(kHaloThreads), smem,
                              s, 2, xmap, wmap, a);
  return launch_pdl(igemm_halo_kernel<PX, CO, CM, 32, __nv_bfloat16>, dim3(grid), dim3(kHaloThreads), smem, s, xmap,
                    wmap, a);
}

cudaError_t launch_igemm_halo_bf16(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int px,
                                   int co, bool cm, int grid, size_t smem, cudaStream_t s) {
  if (a.kc == 16 || a.kc == 8) return !cm && px == 128 ? launch_igemm_halo_bf16_narrow(xmap, wmap, a, co, grid, smem, s)
                                                       : cudaErrorInvalidValue;
  if (a.kc != 32) return cudaErrorInvalidValue;
  if (cm) return px == 256 && co == 128 ? halo_launch_bf16<256, 128, true>(xmap, wmap, a, grid, smem, s)
                                        : cudaErrorInvalidValue;
  if (px != 128) return cudaErrorInvalidValue;
  switch (co) {
    case 32: return halo_launch_bf16<128, 32, false>(xmap, wmap, a, grid, smem, s);
    case 64: return halo_launch_bf16<128, 64, false>(xmap, wmap, a, grid, smem, s);
    case 128: return halo_launch_bf16<128, 128, false>(xmap, wmap, a, grid, smem, s);
    case 256: return halo_launch_bf16<128, 256, false>(xmap, wmap, a, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cb
