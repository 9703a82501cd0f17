// The bf16-operand halo-tile implicit GEMM (igemm_halo.cuh) with 64-byte
// pixel rows (32 bf16 channels per chunk; stride-2 phase tiles too),
// pixel-major 128 x {32, 64, 128}, and with 32-byte rows (16 channels),
// pixel-major 128 x 32, at stride 1 and (phase tiles) 2.
#include "igemm_halo.cuh"
#include "launch_util.h"

namespace cb {

template <int CO, int KC>
static cudaError_t launch_co_bf16(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int grid,
                                  size_t smem, cudaStream_t s) {
  cudaError_t e = smem_attr_once<igemm_halo_kernel<128, CO, false, KC, __nv_bfloat16>>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(igemm_halo_kernel<128, CO, false, KC, __nv_bfloat16>, dim3(grid), dim3(kHaloThreads), smem, s,
                    xmap, wmap, a);
}

cudaError_t launch_igemm_halo_bf16_narrow(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a,
                                          int co, int grid, size_t smem, cudaStream_t s) {
  if (a.split_k != 1) return cudaErrorInvalidValue;
  if (a.kc == 8) return co == 32 ? launch_co_bf16<32, 8>(xmap, wmap, a, grid, smem, s) : cudaErrorInvalidValue;
  if (co == 32) return launch_co_bf16<32, 16>(xmap, wmap, a, grid, smem, s);
  if (co == 64) return launch_co_bf16<64, 16>(xmap, wmap, a, grid, smem, s);
  if (co == 128) return launch_co_bf16<128, 16>(xmap, wmap, a, grid, smem, s);
  return cudaErrorInvalidValue;
}

}  // namespace cb
