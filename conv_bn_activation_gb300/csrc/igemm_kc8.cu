// Tensor-core implicit GEMM instantiated for 8-channel K steps (see igemm_tc.cuh).
#include "igemm_tc.cuh"

namespace cb {

cudaError_t launch_igemm_kc8(const CUtensorMap& amap, const CUtensorMap& bmap, const IgemmArgs& a, int bn, int grid,
                              size_t smem, cudaStream_t s) {
  return igemm_launch_kc<8>(amap, bmap, a, bn, grid, smem, s);
}

int igemm_read_trace_kc8(unsigned long long* out, int max_records) {
  return igemm_read_trace_tu(out, max_records);
}

}  // namespace cb
