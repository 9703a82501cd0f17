// Direct convolution on CUDA cores (fp32), groups = 1, with the fused
// folded-BN / residual / activation epilogue.
//
// This is the path for layers the tensor-core implicit GEMM does not take:
// stems with 1 or 3 input channels (the 1x28x28 MNIST stem, the 640x640x3
// YOLO-style stem, the stem that reads the planar NCHW preprocess output),
// odd channel counts, and views whose alignment a TMA descriptor cannot
// express.  These layers are memory-bound (a 3->16 stride-2 stem moves about
// 7.7 FLOP per byte), so the design goal is one pass over the input and one
// coalesced write of the output:
//  * one thread per output pixel and COB consecutive output channels;
//  * the CTA's COB-channel slice of the weights staged in shared memory as
//    [tap][ci][COB] so that a thread reads COB weights with vector loads;
//  * the input read through arbitrary strides, so NHWC and NCHW inputs share
//    the kernel.
#include "epilogue.cuh"
#include "internal.h"

namespace cb {

template <int COB>
__global__ void __launch_bounds__(256) direct_conv_kernel(const DirectArgs a, int vec_out) {
  extern __shared__ __align__(16) float sw[];
  const int K = a.kh * a.kw * a.Ci;
  const int co0 = blockIdx.y * COB;
  for (int i = threadIdx.x; i < K * COB; i += blockDim.x) {
    const int k = i / COB, q = i % COB;
    const int co = co0 + q;
    sw[i] = co < a.Co ? __ldg(a.w + static_cast<long long>(co) * K + k) : 0.0f;
  }
  __syncthreads();

  const long long M = static_cast<long long>(a.N) * a.OH * a.OW;
  const long long m = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (m >= M) return;
  const int ow = static_cast<int>(m % a.OW);
  const int oh = static_cast<int>((m / a.OW) % a.OH);
  const int n = static_cast<int>(m / (static_cast<long long>(a.OW) * a.OH));

  float acc[COB];
#pragma unroll
  for (int q = 0; q < COB; ++q) acc[q] = 0.0f;

  for (int i = 0; i < a.kh; ++i) {
    const int ih = oh * a.stride - a.pad + i;
    if (ih < 0 || ih >= a.H) continue;
    for (int j = 0; j < a.kw; ++j) {
      const int iw = ow * a.stride - a.pad + j;
      if (iw < 0 || iw >= a.W) continue;
      const float* xp = a.x + n * a.xs_n + ih * a.xs_h + iw * a.xs_w;
      const float* wr = sw + (i * a.kw + j) * a.Ci * COB;
      for (int ci = 0; ci < a.Ci; ++ci) {
        const float xv = __ldg(xp + ci * a.xs_c);
        if (COB % 4 == 0) {
#pragma unroll
          for (int q = 0; q < COB; q += 4) {
            const float4 wv = *reinterpret_cast<const float4*>(wr + ci * COB + q);
            acc[q] = fmaf(xv, wv.x, acc[q]);
            acc[q + 1] = fmaf(xv, wv.y, acc[q + 1]);
            acc[q + 2] = fmaf(xv, wv.z, acc[q + 2]);
            acc[q + 3] = fmaf(xv, wv.w, acc[q + 3]);
          }
        } else {
#pragma unroll
          for (int q = 0; q < COB; ++q) acc[q] = fmaf(xv, wr[ci * COB + q], acc[q]);
        }
      }
    }
  }

  float* yp = a.out.y + n * a.out.ys_n + oh * a.out.ys_h + ow * a.out.ys_w + co0;
  const float* rp = a.ep.res_mode ? a.ep.r + n * a.ep.rs_n + oh * a.ep.rs_h + ow * a.ep.rs_w + co0 : nullptr;
  if (COB % 4 == 0 && vec_out && co0 + COB <= a.Co) {
#pragma unroll
    for (int q = 0; q < COB; q += 4) {
      const float4 r = a.ep.res_mode ? *reinterpret_cast<const float4*>(rp + q) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 o = epi_apply4(make_float4(acc[q], acc[q + 1], acc[q + 2], acc[q + 3]), ldg4(a.ep.scale + co0 + q),
                                  ldg4(a.ep.bias + co0 + q), r, a.ep.act, a.ep.res_mode);
      *reinterpret_cast<float4*>(yp + q) = o;
    }
  } else {
#pragma unroll
    for (int q = 0; q < COB; ++q) {
      if (co0 + q < a.Co) {
        const float r = a.ep.res_mode ? rp[q] : 0.0f;
        yp[q] = epi_apply(acc[q], __ldg(a.ep.scale + co0 + q), __ldg(a.ep.bias + co0 + q), r, a.ep.act,
                          a.ep.res_mode);
      }
    }
  }
}

namespace {
template <int COB>
cudaError_t launch_cob(const DirectArgs& a, int vec_out, cudaStream_t s) {
  const long long M = static_cast<long long>(a.N) * a.OH * a.OW;
  const size_t smem = static_cast<size_t>(a.kh) * a.kw * a.Ci * COB * sizeof(float);
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(direct_conv_kernel<COB>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  dim3 grid(static_cast<unsigned>((M + 255) / 256), static_cast<unsigned>((a.Co + COB - 1) / COB));
  direct_conv_kernel<COB><<<grid, 256, smem, s>>>(a, vec_out);
  return cudaGetLastError();
}
}  // namespace

// Chooses COB so that the CTA's weight slice fits in shared memory.
cudaError_t launch_direct(const DirectArgs& a, cudaStream_t s) {
  const long long M = static_cast<long long>(a.N) * a.OH * a.OW;
  if (M == 0) return cudaSuccess;
  const long long K = static_cast<long long>(a.kh) * a.kw * a.Ci;
  const bool vec_ok = (reinterpret_cast<uintptr_t>(a.out.y) % 16 == 0) && a.out.ys_w % 4 == 0 &&
                      a.out.ys_h % 4 == 0 && a.out.ys_n % 4 == 0 &&
                      (a.ep.res_mode == 0 || ((reinterpret_cast<uintptr_t>(a.ep.r) % 16 == 0) && a.ep.rs_w % 4 == 0 &&
                                              a.ep.rs_h % 4 == 0 && a.ep.rs_n % 4 == 0));
  const int vec = vec_ok ? 1 : 0;
  const long long budget = 200 * 1024 / sizeof(float);
  if (a.Co >= 16 && K * 16 <= budget) return launch_cob<16>(a, vec, s);
  if (a.Co >= 8 && K * 8 <= budget) return launch_cob<8>(a, vec, s);
  if (K * 4 <= budget) return launch_cob<4>(a, vec, s);
  if (K <= budget) return launch_cob<1>(a, 0, s);
  return cudaErrorInvalidValue;
}

}  // namespace cb
