// The channel-major instantiation of the halo-tile implicit GEMM
// (igemm_halo.cuh): 256 pixels x 128 output channels per tile.
#include "igemm_halo.cuh"

namespace cb {

int igemm_read_trace_halo_cm(unsigned long long* out, int max_records) { return igemm_read_trace_tu(out, max_records); }

cudaError_t launch_igemm_halo_cm256(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int grid,
                                    size_t smem, cudaStream_t s) {
  return halo_launch<256, 128, true>(xmap, wmap, a, grid, smem, s);
}

int halo_max_pairs_cm256(size_t smem) { return halo_pairs<256, 128, true>(smem); }

}  // namespace cb
