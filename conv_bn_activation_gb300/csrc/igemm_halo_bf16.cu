// The bf16-operand instantiations of the halo-tile implicit GEMM
// (igemm_halo.cuh, kind::f16 MMAs): pixel-major 128 x {32, 64, 128, 256} and
// channel-major 256 x 128 tiles of 128-byte pixel rows (64 bf16 channels per
// chunk).  The 64- and 32-byte-row tiles are in igemm_halo_bf16_kc16.cu, the
// 192 x 128 channel-major tile in igemm_halo_cm192.cu.
#include "igemm_halo.cuh"

namespace cb {

cudaError_t launch_igemm_halo_bf16_narrow(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a,
                                          int co, int grid, size_t smem, cudaStream_t s);

cudaError_t launch_igemm_halo_bf16(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int px,
                                   int co, bool cm, int grid, size_t smem, cudaStream_t s) {
  if (a.kc == 16 || a.kc == 8) return !cm && px == 128 ? launch_igemm_halo_bf16_narrow(xmap, wmap, a, co, grid, smem, s)
                                                       : cudaErrorInvalidValue;
  if (a.kc != 32) return cudaErrorInvalidValue;
  if (cm) return px == 256 && co == 128 ? halo_launch<256, 128, true, 32, __nv_bfloat16>(xmap, wmap, a, grid, smem, s)
                                        : cudaErrorInvalidValue;
  if (px != 128) return cudaErrorInvalidValue;
  switch (co) {
    case 32: return halo_launch<128, 32, false, 32, __nv_bfloat16>(xmap, wmap, a, grid, smem, s);
    case 64: return halo_launch<128, 64, false, 32, __nv_bfloat16>(xmap, wmap, a, grid, smem, s);
    case 128: return halo_launch<128, 128, false, 32, __nv_bfloat16>(xmap, wmap, a, grid, smem, s);
    case 256: return halo_launch<128, 256, false, 32, __nv_bfloat16>(xmap, wmap, a, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cb
