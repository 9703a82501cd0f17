// The 16- and 8-channel-chunk instantiations of the halo-tile implicit GEMM
// (igemm_halo.cuh): layers whose input channels are a multiple of 16 but not
// of 32, and stride-2 layers (64-byte pixel rows, 64-byte swizzle),
// pixel-major 128 x {32, 64, 128}.
#include "igemm_halo.cuh"
#include "launch_util.h"

namespace cb {

int igemm_read_trace_halo_kc16(unsigned long long* out, int max_records) {
  return igemm_read_trace_tu(out, max_records);
}

template <int CO, int KC = 16>
static cudaError_t launch_co(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int grid,
                             size_t smem, cudaStream_t s) {
  cudaError_t e = smem_attr_once<igemm_halo_kernel<128, CO, false, KC>>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(igemm_halo_kernel<128, CO, false, KC>, dim3(grid), dim3(kHaloThreads), smem, s, xmap, wmap, a);
}

// 8-channel chunks (32-byte rows, 32-byte swizzle): layers with Ci % 16 == 8
// at stride 1, pixel-major 128 x 32.
cudaError_t launch_igemm_halo_kc8(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int co,
                                  int grid, size_t smem, cudaStream_t s) {
  if (a.split_k != 1 || a.stride != 1) return cudaErrorInvalidValue;
  if (co == 32) return launch_co<32, 8>(xmap, wmap, a, grid, smem, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_igemm_halo_kc16(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int co,
                                   int grid, size_t smem, cudaStream_t s) {
  if (a.split_k != 1) return cudaErrorInvalidValue;
  if (co == 32) return launch_co<32>(xmap, wmap, a, grid, smem, s);
  if (co == 64) return launch_co<64>(xmap, wmap, a, grid, smem, s);
  if (co == 128) return launch_co<128>(xmap, wmap, a, grid, smem, s);
  return cudaErrorInvalidValue;
}

}  // namespace cb
