// Stem convolution 3 -> 16 channels, 3x3, stride 2, pad 1, with the folded-BN
// / activation epilogue, on CUDA cores in fp32 -- and the same kernel with
// the u8 frame preprocess (bilinear resize, u8 rounding, /255) run in its
// input staging, so that the preprocessed image never goes to memory.
//
// The stems of the pages' networks ("YOLO26N Inference Optimisation": the
// 640x640x3 stem; "A fused Ampere preprocess kernel": the network input the
// preprocess feeds) have three input channels, so the layer is a short
// reduction (27 terms) per output and the GEMM view gives the tensor cores
// nothing to chew on: it is bound by HBM (one read of the input, one write
// of the 16-channel output) and by instruction issue.  The design keeps
// both in check:
//  * persistent CTAs of 128 threads walk 8 x 64 tiles of output pixels;
//  * a tile's input (17 rows x 132 columns x 3 channels, zero outside the
//    image = the padding) sits in shared memory as three planes, filled by
//    16-byte cp.async copies of the next tile while the current one is
//    computed: straight into the planes for planar NCHW input; for packed
//    NHWC input into a raw buffer that a de-interleave pass splits; for u8
//    frames, the source rows the tile's bilinear samples need, from which
//    the fill pass computes the preprocessed values (bit-identical to the
//    preprocess kernel: same operations, same order);
//  * each thread owns 2 x 2 output pixels x 16 channels (64 accumulators);
//    per (input channel, filter row) it reads the 5 input columns of each
//    of its two rows with one 16-byte and one 4-byte shared load and reuses
//    them across the 3 filter columns and 2 pixels; the 16 weights of a tap
//    are broadcast 16-byte loads; the FMAs are paired (fma.rn.f32x2, each
//    lane rounded like fmaf), which halves the issue slots they take;
//  * the epilogue applies scale / bias / activation and writes each pixel's
//    16 channels as four 16-byte stores (two adjacent pixels per thread, a
//    warp covering 4 KB of contiguous output row).
#include "epilogue.cuh"
#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"
#include "resample.cuh"

#include <type_traits>

namespace cb {

namespace {

constexpr int kTH = 8;                    // output rows per tile
constexpr int kTW = 64;                   // output columns per tile
constexpr int kThreads = 128;             // 32 column pairs x 4 row pairs
constexpr int kRows = 2 * kTH + 1;        // staged input rows
constexpr int kCols = 2 * kTW + 4;        // staged input columns, from 2 * ow0 - 4 (16-byte aligned)
constexpr int kChunks = kCols / 4;        // 16-byte chunks per staged plane row
constexpr int kPlane = kRows * kCols;     // floats per channel plane
constexpr int kTileF = 3 * kPlane;        // floats per staged tile (a multiple of 4)
constexpr int kRawRow = 3 * kCols;        // floats per packed NHWC row of the tile
constexpr int kFixedF = 27 * 16 + 16 + 16 + 256;  // weights, scale, bias, u8 / 255 table
// bf16 NHWC input (SRC 3): rows staged from input column 2 * ow0 - 8, so that
// the 6-byte pixels start on a 16-byte boundary; 136 pixels = 17 groups of 8
// (48 bytes, three 16-byte copies), plane column = staged pixel - 4.
constexpr int kBfGroups = (kCols + 4) / 8;
constexpr int kBfRawRowB = kBfGroups * 48;        // bytes per staged bf16 row
static_assert(kBfRawRowB <= kRawRow * 4, "a bf16 row fits in an fp32 row's room");

static_assert(kTileF % 4 == 0 && kRawRow % 4 == 0 && kFixedF % 4 == 0, "16-byte aligned regions");

__device__ __forceinline__ void cp_async16_z(void* dst, const void* src, bool in) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(in ? 16 : 0)
               : "memory");
}

struct TilePos {
  int n, oh0, ow0, ih0, iw0;
};

__device__ __forceinline__ TilePos tile_pos(int t, const StemArgs& a) {
  TilePos p;
  const int tx = t % a.tiles_x, rest = t / a.tiles_x;
  const int ty = rest % a.tiles_y;
  p.n = rest / a.tiles_y;
  p.oh0 = ty * kTH;
  p.ow0 = tx * kTW;
  p.ih0 = 2 * p.oh0 - 1;  // input row of staged row 0
  p.iw0 = 2 * p.ow0 - 4;  // input column of staged column 0
  return p;
}

// Source rows and byte range of the u8 frames that the preprocessed pixels
// of one tile sample (rows r_lo..r_hi, bytes [b_lo, b_hi) of each row).
struct SrcSpan {
  int r_lo, r_hi, b_lo, b_hi;
};

__device__ __forceinline__ SrcSpan src_span(const TilePos& p, const StemArgs& a, float scale_y, float scale_x) {
  const int y0 = max(p.ih0, 0), y1 = min(p.ih0 + kRows - 1, a.H - 1);
  const int x0 = max(p.iw0, 0), x1 = min(p.iw0 + kCols - 1, a.W - 1);
  SrcSpan s;
  s.r_lo = axis_sample(y0, a.hs, scale_y).i0;
  s.r_hi = axis_sample(y1, a.hs, scale_y).i1;
  s.b_lo = (3 * axis_sample(x0, a.ws, scale_x).i0) & ~15;
  s.b_hi = (3 * axis_sample(x1, a.ws, scale_x).i1 + 3 + 15) & ~15;
  return s;
}

// Issues the copies of tile t: planar input into `pl` (SRC 0), packed NHWC
// rows into `raw` (SRC 1; SRC 3 for bf16), source rows of the u8 frames into
// `raw` (SRC 2).
template <int SRC>
__device__ __forceinline__ void issue_tile(int t, const StemArgs& a, float* pl, float* raw, float scale_y,
                                           float scale_x) {
  const TilePos p = tile_pos(t, a);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (SRC == 0) {
    const float* x = static_cast<const float*>(a.src);
    for (int row = warp; row < 3 * kRows; row += kThreads / 32) {
      const int ci = row / kRows, r = row - ci * kRows;
      const int ih = p.ih0 + r;
      const bool row_ok = ih >= 0 && ih < a.H;
      const long long base = p.n * a.xs_n + ci * a.xs_c + static_cast<long long>(ih) * a.xs_h;
      float* d = pl + ci * kPlane + r * kCols;
      for (int k = lane; k < kChunks; k += 32) {
        const int col = p.iw0 + 4 * k;
        const bool ok = row_ok && col >= 0 && col < a.W;
        cp_async16_z(d + 4 * k, ok ? x + base + col : x, ok);
      }
    }
  } else if (SRC == 1) {
    const float* x = static_cast<const float*>(a.src);
    for (int r = warp; r < kRows; r += kThreads / 32) {
      const int ih = p.ih0 + r;
      const bool row_ok = ih >= 0 && ih < a.H;
      const long long base = p.n * a.xs_n + static_cast<long long>(ih) * a.xs_h + 3LL * p.iw0;
      float* d = raw + r * kRawRow;
      for (int k = lane; k < 3 * kChunks; k += 32) {
        const int col = p.iw0 + 4 * (k / 3);  // first pixel of the 4-pixel group this chunk is in
        const bool ok = row_ok && col >= 0 && col < a.W;
        cp_async16_z(d + 4 * k, ok ? x + base + 4 * k : x, ok);
      }
    }
  } else if (SRC == 3) {
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.src);
    for (int r = warp; r < kRows; r += kThreads / 32) {
      const int ih = p.ih0 + r;
      const bool row_ok = ih >= 0 && ih < a.H;
      const long long base = p.n * a.xs_n + static_cast<long long>(ih) * a.xs_h + 3LL * (p.iw0 - 4);
      uint8_t* d = reinterpret_cast<uint8_t*>(raw) + r * kBfRawRowB;
      for (int k = lane; k < 3 * kBfGroups; k += 32) {
        const int col = p.iw0 - 4 + 8 * (k / 3);  // first pixel of the 8-pixel group this chunk is in
        const bool ok = row_ok && col >= 0 && col < a.W;
        cp_async16_z(d + 16 * k, ok ? x + base + 8 * k : x, ok);
      }
    }
  } else {
    const uint8_t* src = static_cast<const uint8_t*>(a.src);
    const SrcSpan s = src_span(p, a, scale_y, scale_x);
    const int chunks = (s.b_hi - s.b_lo) >> 4;
    const int rows = s.r_hi - s.r_lo + 1;
    const uint8_t* frame = src + static_cast<long long>(p.n) * a.hs * a.pitch + s.b_lo;
    uint8_t* slots = reinterpret_cast<uint8_t*>(raw);
    for (int i = threadIdx.x; i < rows * chunks; i += kThreads) {
      const int r = i / chunks, k = i - r * chunks;
      cp_async16_z(slots + r * a.row_cap + 16 * k, frame + static_cast<long long>(s.r_lo + r) * a.pitch + 16 * k,
                   true);
    }
  }
}

// Builds the three input planes of tile t from the raw buffer (SRC 1, 2, 3).
template <int SRC>
__device__ __forceinline__ void fill_tile(int t, const StemArgs& a, const float* raw, float* pl, const float* inv255,
                                          float scale_y, float scale_x) {
  if (SRC == 3) {
    // 8 bf16 pixels (24 values, three 16-byte loads) per group, widened to
    // fp32 (exact) and split into the planes; plane column = staged pixel - 4
    for (int i = threadIdx.x; i < kRows * kBfGroups; i += kThreads) {
      const int r = i / kBfGroups, g = i - r * kBfGroups;
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(raw) + r * kBfRawRowB + 48 * g);
      const uint4 u0 = src[0], u1 = src[1], u2 = src[2];
      const uint32_t w[12] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w, u2.x, u2.y, u2.z, u2.w};
      float f[24];
#pragma unroll
      for (int k = 0; k < 12; ++k) {
        f[2 * k] = __uint_as_float(w[k] << 16);
        f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
      }
      float* d = pl + r * kCols + 8 * g - 4;
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        if (g > 0)
          *reinterpret_cast<float4*>(d + c * kPlane) = make_float4(f[c], f[3 + c], f[6 + c], f[9 + c]);
        *reinterpret_cast<float4*>(d + 4 + c * kPlane) = make_float4(f[12 + c], f[15 + c], f[18 + c], f[21 + c]);
      }
    }
  } else if (SRC == 1) {
    for (int i = threadIdx.x; i < kRows * kChunks; i += kThreads) {
      const int r = i / kChunks, g = i - r * kChunks;
      const float4* s = reinterpret_cast<const float4*>(raw + r * kRawRow + 12 * g);
      const float4 u = s[0], v = s[1], w = s[2];  // 4 pixels x (c0, c1, c2)
      float* d = pl + r * kCols + 4 * g;
      *reinterpret_cast<float4*>(d) = make_float4(u.x, u.w, v.z, w.y);
      *reinterpret_cast<float4*>(d + kPlane) = make_float4(u.y, v.x, v.w, w.z);
      *reinterpret_cast<float4*>(d + 2 * kPlane) = make_float4(u.z, v.y, w.x, w.w);
    }
  } else if (SRC == 2) {
    const TilePos p = tile_pos(t, a);
    const SrcSpan s = src_span(p, a, scale_y, scale_x);
    const uint8_t* slots = reinterpret_cast<const uint8_t*>(raw);
    const bool two_to_one = a.ws == 2 * a.W;
    for (int i = threadIdx.x; i < kRows * kChunks; i += kThreads) {
      const int r = i / kChunks, g = i - r * kChunks;
      const int y = p.ih0 + r, xf = p.iw0 + 4 * g;
      float* d = pl + r * kCols + 4 * g;
      if (y < 0 || y >= a.H) {
#pragma unroll
        for (int c = 0; c < 3; ++c) *reinterpret_cast<float4*>(d + c * kPlane) = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      const AxisSample sy = axis_sample(y, a.hs, scale_y);
      const uint8_t* ra = slots + (sy.i0 - s.r_lo) * a.row_cap;  // byte b of a source row at ra[b - b_lo]
      const uint8_t* rb = slots + (sy.i1 - s.r_lo) * a.row_cap;
      if (two_to_one && xf >= 0 && xf + 3 < a.W) {
        // exact 2:1 width: the horizontal weights are 1/2, folded into the
        // row weights (as the preprocess kernel does)
        int o[12];  // [pixel q][channel c]
        blend_pairs(ra + 6 * xf - s.b_lo, rb + 6 * xf - s.b_lo, sy.a, o);
#pragma unroll
        for (int c = 0; c < 3; ++c)
          *reinterpret_cast<float4*>(d + c * kPlane) =
              make_float4(inv255[o[c]], inv255[o[3 + c]], inv255[o[6 + c]], inv255[o[9 + c]]);
      } else {
        // other ratios and the image edges, one pixel at a time (kept out of line: code size)
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          const int x = xf + q;
          const bool in = x >= 0 && x < a.W;
          const AxisSample sx = axis_sample(in ? x : 0, a.ws, scale_x);
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            const int i0 = 3 * sx.i0 + c - s.b_lo, i1 = 3 * sx.i1 + c - s.b_lo;
            const int u = round_u8(bilinear(u8_to_float(ra[i0]), u8_to_float(ra[i1]), u8_to_float(rb[i0]),
                                             u8_to_float(rb[i1]), sx.a, sy.a));
            d[c * kPlane + q] = in ? inv255[u] : 0.0f;
          }
        }
      }
    }
  }
}

// The 2 x 2 output pixels x 16 channels of thread (tx, ty) in tile t, from
// the staged planes, through the epilogue to memory.
template <int ACT, bool RES, typename TO = float>
__device__ __forceinline__ void conv_tile(int t, const StemArgs& a, const float* pl, const float* ws,
                                          const float* sc, const float* bi) {
  const TilePos p = tile_pos(t, a);
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
  float2 acc[2][2][8];
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[r][q][j] = make_float2(0.0f, 0.0f);

#pragma unroll
  for (int ci = 0; ci < 3; ++ci) {
#pragma unroll
    for (int kh = 0; kh < 3; ++kh) {
      // input columns 2*ow - 1 .. 2*ow + 3 of the thread's first pixel ow:
      // one 16-byte load of columns 2*ow .. 2*ow + 3, and column 2*ow - 1
      // from the lane to the left (its last column; lane 0 loads its own:
      // a per-lane 4-byte load at a 16-byte stride would be a 4-way bank
      // conflict)
      float v[2][5];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float* rp = pl + ci * kPlane + (4 * ty + 2 * r + kh) * kCols + 4 * tx;
        const float4 f = *reinterpret_cast<const float4*>(rp + 4);
        v[r][0] = __shfl_up_sync(0xffffffffu, f.w, 1);
        if (tx == 0) v[r][0] = rp[3];
        v[r][1] = f.x, v[r][2] = f.y, v[r][3] = f.z, v[r][4] = f.w;
      }
#pragma unroll
      for (int kw = 0; kw < 3; ++kw) {
        const float4* wp = reinterpret_cast<const float4*>(ws + ((kh * 3 + kw) * 3 + ci) * 16);
        float2 w2[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 f = wp[j];
          w2[2 * j] = make_float2(f.x, f.y);
          w2[2 * j + 1] = make_float2(f.z, f.w);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const float xv = v[r][2 * q + kw];
            const float2 xx = make_float2(xv, xv);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[r][q][j] = __ffma2_rn(xx, w2[j], acc[r][q][j]);
          }
      }
    }
  }

  TO* const y = reinterpret_cast<TO*>(a.out.y) + p.n * a.out.ys_n;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int oh = p.oh0 + 2 * ty + r;
    if (oh >= a.OH) continue;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int ow = p.ow0 + 2 * tx + q;
      if (ow >= a.OW) continue;
      TO* yp = y + oh * a.out.ys_h + ow * a.out.ys_w;
      const TO* rp =
          RES ? reinterpret_cast<const TO*>(a.ep.r) + p.n * a.ep.rs_n + oh * a.ep.rs_h + ow * a.ep.rs_w : nullptr;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 s4 = reinterpret_cast<const float4*>(sc)[j], b4 = reinterpret_cast<const float4*>(bi)[j];
        const float2 lo = acc[r][q][2 * j], hi = acc[r][q][2 * j + 1];
        float4 o;
        if (!RES) {
          o = make_float4(epi_t<ACT, 0>(lo.x, s4.x, b4.x, 0.0f), epi_t<ACT, 0>(lo.y, s4.y, b4.y, 0.0f),
                          epi_t<ACT, 0>(hi.x, s4.z, b4.z, 0.0f), epi_t<ACT, 0>(hi.y, s4.w, b4.w, 0.0f));
        } else {
          const float4 rv = load4(rp + 4 * j);
          if (a.ep.res_mode == 1)
            o = make_float4(epi_t<ACT, 1>(lo.x, s4.x, b4.x, rv.x), epi_t<ACT, 1>(lo.y, s4.y, b4.y, rv.y),
                            epi_t<ACT, 1>(hi.x, s4.z, b4.z, rv.z), epi_t<ACT, 1>(hi.y, s4.w, b4.w, rv.w));
          else
            o = make_float4(epi_t<ACT, 2>(lo.x, s4.x, b4.x, rv.x), epi_t<ACT, 2>(lo.y, s4.y, b4.y, rv.y),
                            epi_t<ACT, 2>(hi.x, s4.z, b4.z, rv.z), epi_t<ACT, 2>(hi.y, s4.w, b4.w, rv.w));
        }
        store4(yp + 4 * j, o);
      }
    }
  }
}

template <int SRC, int ACT>
__global__ void __launch_bounds__(kThreads, 4) stem_kernel(const StemArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ __align__(16) float sm[];
  float* const ws = sm;               // [tap][ci][16 co]
  float* const sc = ws + 27 * 16;
  float* const bi = sc + 16;
  float* const inv255 = bi + 16;      // u / 255 for every u8 code (IEEE division)
  float* const pl0 = sm + kFixedF;    // staged planes
  float* const pl1 = pl0 + kTileF;    // second planes (SRC 0) or the raw buffer (SRC 1, 2)
  for (int i = threadIdx.x; i < 27 * 16; i += kThreads) {
    const int co = i % 16, tap = i / 16;
    ws[i] = __ldg(a.w + co * 27 + tap);
  }
  if (threadIdx.x < 16) {
    sc[threadIdx.x] = __ldg(a.ep.scale + threadIdx.x);
    bi[threadIdx.x] = __ldg(a.ep.bias + threadIdx.x);
  }
  if (SRC == 2)
    for (int i = threadIdx.x; i < 256; i += kThreads) inv255[i] = __fdiv_rn(static_cast<float>(i), 255.0f);
  const float scale_y = SRC == 2 ? __fdiv_rn(static_cast<float>(a.hs), static_cast<float>(a.H)) : 0.0f;
  const float scale_x = SRC == 2 ? __fdiv_rn(static_cast<float>(a.ws), static_cast<float>(a.W)) : 0.0f;

  const int num_tiles = a.N * a.tiles_y * a.tiles_x;
  int tile = blockIdx.x;
  if (SRC == 0) {
    if (tile < num_tiles) issue_tile<0>(tile, a, pl0, nullptr, 0.0f, 0.0f);
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (int it = 0; tile < num_tiles; tile += gridDim.x, ++it) {
      float* cur = (it & 1) ? pl1 : pl0;
      const int next = tile + gridDim.x;
      if (next < num_tiles) issue_tile<0>(next, a, (it & 1) ? pl0 : pl1, nullptr, 0.0f, 0.0f);
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group 1;" ::: "memory");  // this tile's planes are in place
      __syncthreads();
      if (a.ep.res_mode) conv_tile<ACT, true>(tile, a, cur, ws, sc, bi);
      else conv_tile<ACT, false>(tile, a, cur, ws, sc, bi);
      __syncthreads();  // the copies of a later tile overwrite these planes
    }
  } else {
    if (tile < num_tiles) issue_tile<SRC>(tile, a, nullptr, pl1, scale_y, scale_x);
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (; tile < num_tiles; tile += gridDim.x) {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      __syncthreads();  // raw data in place; the previous tile's reads of the planes are done
      fill_tile<SRC>(tile, a, pl1, pl0, inv255, scale_y, scale_x);
      __syncthreads();  // planes built; the raw buffer is free
      const int next = tile + gridDim.x;
      if (next < num_tiles) issue_tile<SRC>(next, a, nullptr, pl1, scale_y, scale_x);
      asm volatile("cp.async.commit_group;" ::: "memory");
      using TO = std::conditional_t<SRC == 3, __nv_bfloat16, float>;  // bf16 input: bf16 output
      if (SRC != 2 && a.ep.res_mode) conv_tile<ACT, true, TO>(tile, a, pl0, ws, sc, bi);  // frames: no residual
      else conv_tile<ACT, false, TO>(tile, a, pl0, ws, sc, bi);
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

template <int SRC, int ACT>
cudaError_t launch_act(const StemArgs& a, size_t smem, int sms, cudaStream_t s) {
  cudaError_t e = smem_attr_once<stem_kernel<SRC, ACT>>(smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stem_kernel<SRC, ACT>, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const long long tiles = static_cast<long long>(a.N) * a.tiles_y * a.tiles_x;
  const long long cap = static_cast<long long>(sms) * per_sm;
  const unsigned grid = static_cast<unsigned>(tiles < cap ? tiles : cap);
  return launch_pdl(stem_kernel<SRC, ACT>, dim3(grid), dim3(kThreads), smem, s, a);
}

template <int SRC>
cudaError_t launch_src(const StemArgs& a, size_t smem, int sms, cudaStream_t s) {
  if (a.ep.act == 0) return launch_act<SRC, 0>(a, smem, sms, s);
  if (a.ep.act == 1) return launch_act<SRC, 1>(a, smem, sms, s);
  return launch_act<SRC, 2>(a, smem, sms, s);
}

}  // namespace

size_t stem_smem_bytes(int src_kind, int src_rows, int row_cap) {
  const size_t fixed = static_cast<size_t>(kFixedF + kTileF) * sizeof(float);
  if (src_kind == 0 || src_kind == 1 || src_kind == 3) return fixed + static_cast<size_t>(kTileF) * sizeof(float);
  return fixed + static_cast<size_t>(src_rows) * row_cap;
}

void stem_tile_grid(int OH, int OW, int* tiles_y, int* tiles_x) {
  *tiles_y = (OH + kTH - 1) / kTH;
  *tiles_x = (OW + kTW - 1) / kTW;
}

void stem_src_bounds(int hs, int ws, int hd, int wd, int* rows, int* row_cap) {
  // At most kRows destination rows (kCols columns) per tile: the samples
  // span at most ceil((kRows - 1) * hs / hd) + 1 source rows past the first,
  // plus the second row of the last sample; columns likewise, plus the
  // 16-byte alignment of both ends.
  *rows = static_cast<int>((static_cast<long long>(kRows) * hs + hd - 1) / hd) + 3;
  const int cols = static_cast<int>((static_cast<long long>(kCols) * ws + wd - 1) / wd) + 3;
  *row_cap = (3 * cols + 32 + 15) & ~15;
}

cudaError_t launch_stem(const StemArgs& a, int src_kind, size_t smem, int sms, cudaStream_t s) {
  if (static_cast<long long>(a.N) * a.tiles_y * a.tiles_x == 0) return cudaSuccess;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  if (src_kind == 0) return launch_src<0>(a, smem, sms, s);
  if (src_kind == 1) return launch_src<1>(a, smem, sms, s);
  if (src_kind == 3) return launch_src<3>(a, smem, sms, s);
  return launch_src<2>(a, smem, sms, s);
}

}  // namespace cb
