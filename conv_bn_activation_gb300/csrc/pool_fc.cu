// Global average pool + linear layer (the DepthwiseMNIST head on "How I sped
// up convolutions": AdaptiveAvgPool2d(1), flatten, Linear).  One CTA per
// image: threads first average their channels over H x W (consecutive
// threads read consecutive channels of a pixel, so the reads coalesce), then
// each output feature is a dot product over the pooled vector in shared
// memory.  The whole head moves ~38 KB per image; it exists so that the
// network's last step also runs on the GPU.
#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"

namespace cb {

__global__ void __launch_bounds__(256) pool_fc_kernel(const PoolFcArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ float pooled[];
  const int n = blockIdx.x;
  const float inv = 1.0f / static_cast<float>(a.H * a.W);
  for (int c = threadIdx.x; c < a.C; c += blockDim.x) {
    float acc = 0.0f;
    for (int h = 0; h < a.H; ++h)
      for (int w = 0; w < a.W; ++w) acc += __ldg(a.x + n * a.xs_n + h * a.xs_h + w * a.xs_w + c);
    pooled[c] = acc * inv;
  }
  __syncthreads();
  for (int o = threadIdx.x; o < a.out_features; o += blockDim.x) {
    float acc = __ldg(a.fc_b + o);
    const float* wr = a.fc_w + static_cast<long long>(o) * a.C;
    for (int c = 0; c < a.C; ++c) acc = fmaf(pooled[c], __ldg(wr + c), acc);
    a.out[static_cast<long long>(n) * a.out_features + o] = acc;
  }
}

cudaError_t launch_pool_fc(const PoolFcArgs& a, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  const cudaError_t e = launch_pdl(pool_fc_kernel, dim3(a.N), dim3(256), a.C * sizeof(float), s, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace cb
