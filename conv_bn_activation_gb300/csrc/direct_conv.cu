// Direct convolution on CUDA cores (fp32), groups = 1, with the fused
// folded-BN / residual / activation epilogue: a shared-memory tiled kernel
// for layers with few input channels and a generic one for the rest.
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
#include "launch_util.h"
#include "internal.h"
#include "ptx.cuh"

namespace cb {

template <int COB>
__global__ void __launch_bounds__(256) direct_conv_kernel(const DirectArgs a, int vec_out) {
  pdl_wait();
  pdl_launch_dependents();
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

// ------------------------------------------------ small-channel tiled kernel
// Layers with at most 16 input channels (stems reading 1 or 3 channels,
// NHWC or planar; 8- and 16-channel 3x3 layers).  A CTA computes a TH x 32
// tile of output pixels for COB output channels.  The input tile and its
// halo are staged once in shared memory in planar form -- one plane per
// input channel, and for stride 2 the even and odd input columns in separate
// half-planes -- so that the 32 threads of a warp (32 consecutive output
// columns) read 32 consecutive words per tap.  The CTA's weights sit in
// shared memory as [tap][ci][COB] and are read as broadcast float4s; each
// thread accumulates PX pixels (rows) x COB channels in registers.
constexpr int kTileW = 32;

template <int S, int KS, int COB, int PX, int CI>
__global__ void __launch_bounds__(256) direct_tile_kernel(const DirectArgs a, int th, int vec_out) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ __align__(16) float sm[];
  const int Ci = CI ? CI : a.Ci;  // compile-time for the common channel counts
  const int rows_in = (th - 1) * S + KS;
  const int cols_in = (kTileW - 1) * S + KS;
  const int half = (cols_in + 1) / 2;              // half-plane width for stride 2
  const int pitch = S == 2 ? 2 * half : cols_in;   // words per staged row
  const int plane = rows_in * pitch;
  float* xs = sm;
  float* ws = sm + ((Ci * plane + 3) & ~3);      // [tap][ci][COB], 16-byte aligned for float4 reads

  const int co_blocks = (a.Co + COB - 1) / COB;
  const int n = blockIdx.z / co_blocks;
  const int co0 = (blockIdx.z % co_blocks) * COB;
  const int oh0 = blockIdx.y * th, ow0 = blockIdx.x * kTileW;
  const int ih0 = oh0 * S - a.pad, iw0 = ow0 * S - a.pad;

  // weights of this output-channel block
  const int taps = KS * KS;
  for (int i = threadIdx.x; i < taps * Ci * COB; i += blockDim.x) {
    const int q = i % COB, tc = i / COB;  // tc = tap * Ci + ci
    const int co = co0 + q;
    ws[i] = co < a.Co ? __ldg(a.w + static_cast<long long>(co) * taps * Ci + tc) : 0.0f;
  }
  // input tile with halo, zero outside the image.  Each thread owns fixed
  // (column, channel) positions of a staged row and copies them for all rows,
  // eight rows' loads in flight at a time.
  const int per_row = cols_in * Ci;
  constexpr int U = 8;
  for (int rem = threadIdx.x; rem < per_row; rem += blockDim.x) {
    int c, ci;
    if (a.xs_c == 1) {  // channel-contiguous input: walk (col, ci) so reads coalesce
      c = rem / Ci;
      ci = rem - c * Ci;
    } else {            // planar input: walk (ci, col)
      ci = rem / cols_in;
      c = rem - ci * cols_in;
    }
    const int iw = iw0 + c;
    const bool col_ok = iw >= 0 && iw < a.W;
    const float* gp = a.x + n * a.xs_n + static_cast<long long>(ci) * a.xs_c + static_cast<long long>(iw) * a.xs_w;
    float* sp = xs + ci * plane + (S == 2 ? (c & 1) * half + (c >> 1) : c);
    for (int r0 = 0; r0 < rows_in; r0 += U) {
      float v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int ih = ih0 + r0 + u;
        v[u] = (col_ok && r0 + u < rows_in && ih >= 0 && ih < a.H) ? __ldg(gp + static_cast<long long>(ih) * a.xs_h)
                                                                  : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (r0 + u < rows_in) sp[(r0 + u) * pitch] = v[u];
    }
  }
  __syncthreads();

  const int col = threadIdx.x % kTileW;
  const int rowg = (threadIdx.x / kTileW) * PX;
  float acc[PX][COB];
#pragma unroll
  for (int p = 0; p < PX; ++p)
#pragma unroll
    for (int q = 0; q < COB; ++q) acc[p][q] = 0.0f;

  for (int kh = 0; kh < KS; ++kh) {
#pragma unroll
    for (int kw = 0; kw < KS; ++kw) {
      const int sc = S == 2 ? (kw & 1) * half + col + (kw >> 1) : col + kw;
      const float* wp = ws + (kh * KS + kw) * Ci * COB;
      for (int ci = 0; ci < Ci; ++ci) {
        float wv[COB];
#pragma unroll
        for (int q = 0; q < COB; q += 4) {
          const float4 t = *reinterpret_cast<const float4*>(wp + ci * COB + q);
          wv[q] = t.x, wv[q + 1] = t.y, wv[q + 2] = t.z, wv[q + 3] = t.w;
        }
        const float* xp = xs + ci * plane + (rowg * S + kh) * pitch + sc;
#pragma unroll
        for (int p = 0; p < PX; ++p) {
          const float xv = xp[p * S * pitch];
#pragma unroll
          for (int q = 0; q < COB; ++q) acc[p][q] = fmaf(xv, wv[q], acc[p][q]);
        }
      }
    }
  }

  const int ow = ow0 + col;
#pragma unroll
  for (int p = 0; p < PX; ++p) {
    const int oh = oh0 + rowg + p;
    if (oh >= a.OH || ow >= a.OW || rowg + p >= th) continue;
    float* yp = a.out.y + n * a.out.ys_n + oh * a.out.ys_h + ow * a.out.ys_w + co0;
    const float* rp = a.ep.res_mode ? a.ep.r + n * a.ep.rs_n + oh * a.ep.rs_h + ow * a.ep.rs_w + co0 : nullptr;
    if (vec_out && co0 + COB <= a.Co) {
#pragma unroll
      for (int q = 0; q < COB; q += 4) {
        const float4 r = a.ep.res_mode ? *reinterpret_cast<const float4*>(rp + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(yp + q) =
            epi_apply4(make_float4(acc[p][q], acc[p][q + 1], acc[p][q + 2], acc[p][q + 3]),
                       ldg4(a.ep.scale + co0 + q), ldg4(a.ep.bias + co0 + q), r, a.ep.act, a.ep.res_mode);
      }
    } else {
#pragma unroll
      for (int q = 0; q < COB; ++q)
        if (co0 + q < a.Co)
          yp[q] = epi_apply(acc[p][q], __ldg(a.ep.scale + co0 + q), __ldg(a.ep.bias + co0 + q),
                            a.ep.res_mode ? rp[q] : 0.0f, a.ep.act, a.ep.res_mode);
    }
  }
}

namespace {
template <int S, int KS, int COB, int CI>
cudaError_t launch_tile(const DirectArgs& a, int vec_out, cudaStream_t s) {
  constexpr int PX = 2;
  // tile height: as tall as fits in 64 KB of shared memory (8 rows per 256 threads x PX)
  int th = 256 / kTileW * PX;
  auto smem_for = [&](int t) {
    const int rows_in = (t - 1) * S + KS, cols_in = (kTileW - 1) * S + KS;
    const int pitch = S == 2 ? 2 * ((cols_in + 1) / 2) : cols_in;
    return static_cast<size_t>(((a.Ci * rows_in * pitch + 3) & ~3) + KS * KS * a.Ci * COB) * sizeof(float);
  };
  while (th > PX && smem_for(th) > 64 * 1024) th -= PX;
  const size_t smem = smem_for(th);
  if (smem > 64 * 1024) return cudaErrorInvalidValue;
  if (smem > 48 * 1024) {
    const cudaError_t e = smem_attr_once<direct_tile_kernel<S, KS, COB, PX, CI>>(smem);
    if (e != cudaSuccess) return e;
  }
  const int co_blocks = (a.Co + COB - 1) / COB;
  dim3 grid((a.OW + kTileW - 1) / kTileW, (a.OH + th - 1) / th, a.N * co_blocks);
  return launch_pdl(direct_tile_kernel<S, KS, COB, PX, CI>, grid, dim3(kTileW * (th / PX)), smem, s, a, th, vec_out);
}

template <int S, int KS, int COB>
cudaError_t launch_tile_ci(const DirectArgs& a, int vec_out, cudaStream_t s) {
  if (KS == 3) {
    switch (a.Ci) {
      case 1: return launch_tile<S, KS, COB, 1>(a, vec_out, s);
      case 3: return launch_tile<S, KS, COB, 3>(a, vec_out, s);
      case 8: return launch_tile<S, KS, COB, 8>(a, vec_out, s);
      case 16: return launch_tile<S, KS, COB, 16>(a, vec_out, s);
      default: break;
    }
  }
  return launch_tile<S, KS, COB, 0>(a, vec_out, s);
}

template <int S, int KS>
cudaError_t launch_tile_cob(const DirectArgs& a, int vec_out, cudaStream_t s) {
  if (a.Co <= 8) return launch_tile_ci<S, KS, 8>(a, vec_out, s);
  return launch_tile_ci<S, KS, 16>(a, vec_out, s);
}

template <int COB>
cudaError_t launch_cob(const DirectArgs& a, int vec_out, cudaStream_t s) {
  const long long M = static_cast<long long>(a.N) * a.OH * a.OW;
  const size_t smem = static_cast<size_t>(a.kh) * a.kw * a.Ci * COB * sizeof(float);
  if (smem > 48 * 1024) {
    const cudaError_t e = smem_attr_once<direct_conv_kernel<COB>>(smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(static_cast<unsigned>((M + 255) / 256), static_cast<unsigned>((a.Co + COB - 1) / COB));
  return launch_pdl(direct_conv_kernel<COB>, grid, dim3(256), smem, s, a, vec_out);
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
  if (a.Ci <= 16 && a.kh == a.kw && (a.kh == 1 || a.kh == 3) && (a.stride == 1 || a.stride == 2) &&
      a.N <= 65535 / ((a.Co + 7) / 8)) {
    if (a.stride == 1) return a.kh == 3 ? launch_tile_cob<1, 3>(a, vec, s) : launch_tile_cob<1, 1>(a, vec, s);
    return a.kh == 3 ? launch_tile_cob<2, 3>(a, vec, s) : launch_tile_cob<2, 1>(a, vec, s);
  }
  const long long budget = 200 * 1024 / sizeof(float);
  if (a.Co >= 16 && K * 16 <= budget) return launch_cob<16>(a, vec, s);
  if (a.Co >= 8 && K * 8 <= budget) return launch_cob<8>(a, vec, s);
  if (K * 4 <= budget) return launch_cob<4>(a, vec, s);
  if (K <= budget) return launch_cob<1>(a, 0, s);
  return cudaErrorInvalidValue;
}

}  // namespace cb
