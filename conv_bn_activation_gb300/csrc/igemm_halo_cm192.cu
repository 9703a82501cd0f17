// The 192-pixel channel-major instantiations of the halo-tile implicit GEMM
// (igemm_halo.cuh): 192 pixels x 128 output channels per tile, fp32 (TF32
// MMAs) and bf16 operands (kind::f16) of 128-byte pixel rows.
#include "igemm_halo.cuh"

namespace cb {

int igemm_read_trace_halo_cm192(unsigned long long* out, int max_records) {
  return igemm_read_trace_tu(out, max_records);
}

cudaError_t launch_igemm_halo_cm192(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int grid,
                                    size_t smem, cudaStream_t s) {
  if (a.kc != 32) return cudaErrorInvalidValue;
  return a.bf16 ? halo_launch<192, 128, true, 32, __nv_bfloat16>(xmap, wmap, a, grid, smem, s)
                : halo_launch<192, 128, true>(xmap, wmap, a, grid, smem, s);
}

int halo_max_pairs_cm192(size_t smem) { return halo_pairs<192, 128, true>(smem); }

}  // namespace cb
