// Tensor-core implicit GEMM with bf16 operands (kind::f16) instantiated for
// K steps of 16 x 4 bytes, i.e. 32 bf16 channels (see igemm_tc.cuh).
#include "igemm_tc.cuh"

namespace cb {

cudaError_t launch_igemm_bf16_kc16(const CUtensorMap& amap, const CUtensorMap& bmap, const IgemmArgs& a, int bn,
                                   int grid, size_t smem, cudaStream_t s) {
  return igemm_launch_kc<16, __nv_bfloat16>(amap, bmap, a, bn, grid, smem, s);
}

}  // namespace cb
