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
// NHWC or planar; 8- and 16-channel 3x3 layers).  Persistent CTAs walk
// TH x 32 tiles of output pixels.  A tile's input (with its halo) is staged
// in shared memory in planar form -- one plane per input channel, and for
// stride 2 the even and odd input columns in separate half-planes -- so that
// the 32 threads of a warp (32 consecutive output columns) read 32
// consecutive words per tap.  The staging is asynchronous (4-byte cp.async,
// zero-filled outside the image, which is the padding) into the second of
// two buffers while the current tile is computed.  The weights of every
// output channel sit in shared memory as [tap][ci][Co padded to COB] and are
// read as broadcast float4s; each thread accumulates PX pixels (rows) x COB
// channels in registers, one COB-channel block after another, all from the
// one staged tile.
constexpr int kTileW = 32;
constexpr int kStagePos = 5;  // staged-row positions per thread (the launch checks they cover a row)

__device__ __forceinline__ void cp_async4(float* dst, const float* src, bool in) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(in ? 4 : 0)
               : "memory");
}

struct TileGeom {
  int th, rows_in, cols_in, half, pitch, plane, tile_floats;  // tile_floats: one staged tile, 16-byte multiple
};

template <int S, int KS>
__host__ __device__ inline TileGeom tile_geom(int th, int ci) {
  TileGeom g;
  g.th = th;
  g.rows_in = (th - 1) * S + KS;
  g.cols_in = (kTileW - 1) * S + KS;
  g.half = (g.cols_in + 1) / 2;                  // half-plane width for stride 2
  g.pitch = S == 2 ? 2 * g.half : g.cols_in;     // words per staged row
  g.plane = g.rows_in * g.pitch;
  g.tile_floats = (ci * g.plane + 3) & ~3;
  return g;
}

// COB output channels of one pixel through the compile-time epilogue.
template <int COB, int ACT, int RES>
__device__ __forceinline__ void store_cob(const float (&acc)[COB], float* yp, const float* rp, const DirectArgs& a,
                                          int co0, int vec_out) {
  if (vec_out && co0 + COB <= a.Co) {
#pragma unroll
    for (int q = 0; q < COB; q += 4) {
      const float4 r = RES ? *reinterpret_cast<const float4*>(rp + q) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 sc = ldg4(a.ep.scale + co0 + q), bi = ldg4(a.ep.bias + co0 + q);
      *reinterpret_cast<float4*>(yp + q) =
          make_float4(epi_t<ACT, RES>(acc[q], sc.x, bi.x, r.x), epi_t<ACT, RES>(acc[q + 1], sc.y, bi.y, r.y),
                      epi_t<ACT, RES>(acc[q + 2], sc.z, bi.z, r.z), epi_t<ACT, RES>(acc[q + 3], sc.w, bi.w, r.w));
    }
  } else {
#pragma unroll
    for (int q = 0; q < COB; ++q)
      if (co0 + q < a.Co)
        yp[q] = epi_t<ACT, RES>(acc[q], __ldg(a.ep.scale + co0 + q), __ldg(a.ep.bias + co0 + q), RES ? rp[q] : 0.0f);
  }
}

template <int S, int KS, int COB, int PX, int CI>
__global__ void __launch_bounds__(256, 2) direct_tile_kernel(const DirectArgs a, int th, int vec_out, int tiles_x,
                                                          int tiles_y, int co_pad) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ __align__(16) float sm[];
  const int Ci = CI ? CI : a.Ci;  // compile-time for the common channel counts
  const TileGeom tg = tile_geom<S, KS>(th, Ci);
  float* const xbuf1 = sm + tg.tile_floats;  // second tile buffer (the first is sm)
  float* ws = sm + 2 * tg.tile_floats;  // [tap][ci][co_pad], 16-byte aligned for float4 reads
  const int taps = KS * KS;
  for (int i = threadIdx.x; i < taps * Ci * co_pad; i += blockDim.x) {
    const int q = i % co_pad, tc = i / co_pad;  // tc = tap * Ci + ci
    ws[i] = q < a.Co ? __ldg(a.w + static_cast<long long>(q) * taps * Ci + tc) : 0.0f;
  }

  const int num_tiles = a.N * tiles_y * tiles_x;
  // Each thread owns up to kPos fixed (column, channel) positions of a staged
  // row -- position rem = threadIdx.x + k * blockDim.x, in the order that
  // makes a warp's reads coalesce (channel-fastest for NHWC, column-fastest
  // for planar input) -- decoded once, and copies them for every row.
  constexpr int kPos = kStagePos;
  const int per_row = tg.cols_in * Ci;
  int pos_c[kPos], pos_off[kPos];
  long long pos_goff[kPos];
#pragma unroll
  for (int k = 0; k < kPos; ++k) {
    const int rem = threadIdx.x + k * static_cast<int>(blockDim.x);
    int c = 0, ci = 0;
    if (a.xs_c == 1) {
      c = rem / Ci;
      ci = rem - c * Ci;
    } else {
      ci = rem / tg.cols_in;
      c = rem - ci * tg.cols_in;
    }
    pos_c[k] = rem < per_row ? c : -1;
    pos_off[k] = ci * tg.plane + (S == 2 ? (c & 1) * tg.half + (c >> 1) : c);
    pos_goff[k] = static_cast<long long>(c) * a.xs_w + static_cast<long long>(ci) * a.xs_c;
  }
  // Issue the copies of tile t into buffer xs.
  auto stage = [&](int t, float* xs) {
    const int tx = t % tiles_x, ty = (t / tiles_x) % tiles_y, n = t / (tiles_x * tiles_y);
    const int ih0 = ty * th * S - a.pad, iw0 = tx * kTileW * S - a.pad;
    const float* xn = a.x + n * a.xs_n + static_cast<long long>(iw0) * a.xs_w;
#pragma unroll
    for (int k = 0; k < kPos; ++k) {
      if (pos_c[k] < 0) continue;
      const int iw = iw0 + pos_c[k];
      const bool col_ok = iw >= 0 && iw < a.W;
      const float* gp = xn + pos_goff[k];
      float* sp = xs + pos_off[k];
      for (int r = 0; r < tg.rows_in; ++r) {
        const int ih = ih0 + r;
        const bool in = col_ok && ih >= 0 && ih < a.H;
        cp_async4(sp + r * tg.pitch, in ? gp + static_cast<long long>(ih) * a.xs_h : a.x, in);
      }
    }
  };

  const int col = threadIdx.x % kTileW;
  const int rowg = (threadIdx.x / kTileW) * PX;
  int tile = blockIdx.x;
  if (tile < num_tiles) stage(tile, sm);
  asm volatile("cp.async.commit_group;" ::: "memory");
  for (int it = 0; tile < num_tiles; tile += gridDim.x, ++it) {
    float* xs = (it & 1) ? xbuf1 : sm;
    const int next = tile + gridDim.x;
    if (next < num_tiles) stage(next, (it & 1) ? sm : xbuf1);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");  // this tile (and the weights) are in place
    __syncthreads();

    const int tx = tile % tiles_x, ty = (tile / tiles_x) % tiles_y, n = tile / (tiles_x * tiles_y);
    const int oh0 = ty * th, ow0 = tx * kTileW;
    const int ow = ow0 + col;
    for (int co0 = 0; co0 < a.Co; co0 += COB) {
      float acc[PX][COB];
#pragma unroll
      for (int p = 0; p < PX; ++p)
#pragma unroll
        for (int q = 0; q < COB; ++q) acc[p][q] = 0.0f;

      if constexpr (S == 1 && KS == 3 && CI > 0) {
        // Stride 1: a staged row is kTileW + 2 words (a compile-time pitch).
        // Per (input channel, filter column) the thread loads the PX + 2
        // input rows its PX outputs touch once and reuses them for the
        // three filter rows: (PX + 2) + 3 * COB / 4 shared loads per
        // 3 * PX * COB FMAs, all at immediate offsets from two pointers that
        // advance once per channel.
        constexpr int kPitch = kTileW + 2;
        const float* xb = xs + rowg * kPitch + col;
        const float* wb = ws + co0;
#pragma unroll 1
        for (int ci = 0; ci < CI; ++ci, xb += tg.plane, wb += co_pad) {
#pragma unroll
          for (int kw = 0; kw < 3; ++kw) {
            float xv[PX + 2];
#pragma unroll
            for (int r = 0; r < PX + 2; ++r) xv[r] = xb[r * kPitch + kw];
#pragma unroll
            for (int kh = 0; kh < 3; ++kh) {
              float wv[COB];
              const float* wp = wb + (kh * 3 + kw) * CI * co_pad;
#pragma unroll
              for (int q = 0; q < COB; q += 4) {
                const float4 t4 = *reinterpret_cast<const float4*>(wp + q);
                wv[q] = t4.x, wv[q + 1] = t4.y, wv[q + 2] = t4.z, wv[q + 3] = t4.w;
              }
#pragma unroll
              for (int p = 0; p < PX; ++p)
#pragma unroll
                for (int q = 0; q < COB; ++q) acc[p][q] = fmaf(xv[p + kh], wv[q], acc[p][q]);
            }
          }
        }
      } else {
        for (int kh = 0; kh < KS; ++kh) {
#pragma unroll
          for (int kw = 0; kw < KS; ++kw) {
            const int sc = S == 2 ? (kw & 1) * tg.half + col + (kw >> 1) : col + kw;
            const float* wp = ws + (kh * KS + kw) * Ci * co_pad + co0;
            for (int ci = 0; ci < Ci; ++ci) {
              float wv[COB];
#pragma unroll
              for (int q = 0; q < COB; q += 4) {
                const float4 t4 = *reinterpret_cast<const float4*>(wp + ci * co_pad + q);
                wv[q] = t4.x, wv[q + 1] = t4.y, wv[q + 2] = t4.z, wv[q + 3] = t4.w;
              }
              const float* xp = xs + ci * tg.plane + (rowg * S + kh) * tg.pitch + sc;
#pragma unroll
              for (int p = 0; p < PX; ++p) {
                const float xv = xp[p * S * tg.pitch];
#pragma unroll
                for (int q = 0; q < COB; ++q) acc[p][q] = fmaf(xv, wv[q], acc[p][q]);
              }
            }
          }
        }
      }

#pragma unroll
      for (int p = 0; p < PX; ++p) {
        const int oh = oh0 + rowg + p;
        if (oh >= a.OH || ow >= a.OW || rowg + p >= th) continue;
        float* yp = a.out.y + n * a.out.ys_n + oh * a.out.ys_h + ow * a.out.ys_w + co0;
        const float* rp = a.ep.res_mode ? a.ep.r + n * a.ep.rs_n + oh * a.ep.rs_h + ow * a.ep.rs_w + co0 : nullptr;
        switch (a.ep.act * 3 + a.ep.res_mode) {  // uniform: one compile-time epilogue per output row
          case 0: store_cob<COB, 0, 0>(acc[p], yp, rp, a, co0, vec_out); break;
          case 1: store_cob<COB, 0, 1>(acc[p], yp, rp, a, co0, vec_out); break;
          case 2: store_cob<COB, 0, 2>(acc[p], yp, rp, a, co0, vec_out); break;
          case 3: store_cob<COB, 1, 0>(acc[p], yp, rp, a, co0, vec_out); break;
          case 4: store_cob<COB, 1, 1>(acc[p], yp, rp, a, co0, vec_out); break;
          case 5: store_cob<COB, 1, 2>(acc[p], yp, rp, a, co0, vec_out); break;
          case 6: store_cob<COB, 2, 0>(acc[p], yp, rp, a, co0, vec_out); break;
          case 7: store_cob<COB, 2, 1>(acc[p], yp, rp, a, co0, vec_out); break;
          default: store_cob<COB, 2, 2>(acc[p], yp, rp, a, co0, vec_out); break;
        }
      }
    }
    __syncthreads();  // a later tile's copies overwrite this buffer
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

namespace {

template <int S, int KS, int COB, int CI>
cudaError_t launch_tile(const DirectArgs& a, int vec_out, int sms, cudaStream_t s) {
  // output rows per thread: 4 for the 8 -> (at most) 8 channel 3x3 stride-1
  // layer (each staged weight float4 then feeds more FMAs), else 2
  constexpr int PX = (S == 1 && KS == 3 && CI == 8 && COB == 8) ? 4 : 2;
  const int co_pad = (a.Co + COB - 1) / COB * COB;
  // Tile height: the tallest (up to 8 row groups of PX rows, 256 threads)
  // whose two staged tiles and weights fit in 100 KB (two CTAs per SM), else
  // the tallest that fits in 200 KB; the threads must cover a staged row in
  // at most kStagePos positions each.
  auto smem_for = [&](int t) {
    const TileGeom g = tile_geom<S, KS>(t, a.Ci);
    return static_cast<size_t>(2 * g.tile_floats + KS * KS * a.Ci * co_pad) * sizeof(float);
  };
  const int per_row = ((kTileW - 1) * S + KS) * a.Ci;
  int th = 0;
  for (int t = 256 / kTileW * PX; t >= PX; t -= PX) {
    if (per_row > kStagePos * kTileW * (t / PX)) continue;
    if (smem_for(t) <= 100 * 1024) {
      th = t;
      break;
    }
    if (th == 0 && smem_for(t) <= 200 * 1024) th = t;
  }
  if (th == 0) return cudaErrorInvalidValue;
  const size_t smem = smem_for(th);
  cudaError_t e = smem_attr_once<direct_tile_kernel<S, KS, COB, PX, CI>>(smem);
  if (e != cudaSuccess) return e;
  const int threads = kTileW * (th / PX);
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, direct_tile_kernel<S, KS, COB, PX, CI>, threads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int tiles_x = (a.OW + kTileW - 1) / kTileW, tiles_y = (a.OH + th - 1) / th;
  const long long tiles = static_cast<long long>(a.N) * tiles_x * tiles_y;
  if (tiles >= (1LL << 31)) return cudaErrorInvalidValue;
  const long long cap = static_cast<long long>(sms) * per_sm;
  const unsigned grid = static_cast<unsigned>(tiles < cap ? tiles : cap);
  return launch_pdl(direct_tile_kernel<S, KS, COB, PX, CI>, dim3(grid), dim3(threads), smem, s, a, th, vec_out,
                    tiles_x, tiles_y, co_pad);
}

template <int S, int KS, int COB>
cudaError_t launch_tile_ci(const DirectArgs& a, int vec_out, int sms, cudaStream_t s) {
  if (KS == 3) {
    switch (a.Ci) {
      case 1: return launch_tile<S, KS, COB, 1>(a, vec_out, sms, s);
      case 3: return launch_tile<S, KS, COB, 3>(a, vec_out, sms, s);
      case 8: return launch_tile<S, KS, COB, 8>(a, vec_out, sms, s);
      case 16: return launch_tile<S, KS, COB, 16>(a, vec_out, sms, s);
      default: break;
    }
  }
  return launch_tile<S, KS, COB, 0>(a, vec_out, sms, s);
}

template <int S, int KS>
cudaError_t launch_tile_cob(const DirectArgs& a, int vec_out, int sms, cudaStream_t s) {
  if (a.Co <= 8) return launch_tile_ci<S, KS, 8>(a, vec_out, sms, s);
  return launch_tile_ci<S, KS, 16>(a, vec_out, sms, s);
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
cudaError_t launch_direct(const DirectArgs& a, int sms, cudaStream_t s) {
  const long long M = static_cast<long long>(a.N) * a.OH * a.OW;
  if (M == 0) return cudaSuccess;
  const long long K = static_cast<long long>(a.kh) * a.kw * a.Ci;
  const bool vec_ok = (reinterpret_cast<uintptr_t>(a.out.y) % 16 == 0) && a.out.ys_w % 4 == 0 &&
                      a.out.ys_h % 4 == 0 && a.out.ys_n % 4 == 0 &&
                      (a.ep.res_mode == 0 || ((reinterpret_cast<uintptr_t>(a.ep.r) % 16 == 0) && a.ep.rs_w % 4 == 0 &&
                                              a.ep.rs_h % 4 == 0 && a.ep.rs_n % 4 == 0));
  const int vec = vec_ok ? 1 : 0;
  if (conv3x3_c8_ok(a)) return launch_conv3x3_c8(a, sms, s);
  if (a.bf16) return cudaErrorInvalidValue;  // bf16 storage: the 8-channel kernel only
  if (a.Ci <= 16 && a.kh == a.kw && (a.kh == 1 || a.kh == 3) && (a.stride == 1 || a.stride == 2)) {
    cudaError_t e;
    if (a.stride == 1)
      e = a.kh == 3 ? launch_tile_cob<1, 3>(a, vec, sms, s) : launch_tile_cob<1, 1>(a, vec, sms, s);
    else
      e = a.kh == 3 ? launch_tile_cob<2, 3>(a, vec, sms, s) : launch_tile_cob<2, 1>(a, vec, sms, s);
    if (e != cudaErrorInvalidValue) return e;  // else: no tile shape fits; the generic kernel below
  }
  const long long budget = 200 * 1024 / sizeof(float);
  if (a.Co >= 16 && K * 16 <= budget) return launch_cob<16>(a, vec, s);
  if (a.Co >= 8 && K * 8 <= budget) return launch_cob<8>(a, vec, s);
  if (K * 4 <= budget) return launch_cob<4>(a, vec, s);
  if (K <= budget) return launch_cob<1>(a, 0, s);
  return cudaErrorInvalidValue;
}

}  // namespace cb
