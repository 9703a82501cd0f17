// Tensor-core implicit GEMM instantiated for 32-channel K steps (see igemm_tc.cuh).
#include "igemm_tc.cuh"

namespace cb {

cudaError_t launch_igemm_kc32(const CUtensorMap& amap, const CUtensorMap& bmap, const IgemmArgs& a, int bn, int grid,
                              size_t smem, cudaStream_t s) {
  return igemm_launch_kc<32>(amap, bmap, a, bn, grid, smem, s);
}

int igemm_read_trace_kc32(unsigned long long* out, int max_records) {
  return igemm_read_trace_tu(out, max_records);
}

}  // namespace cb
