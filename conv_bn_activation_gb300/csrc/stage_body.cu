// The body of a YOLO-style stage with C = 16 channels in one kernel, fp32
// on the CUDA cores ("YOLO26N Inference Optimisation": the conv2d_bn_silu
// layers hold most of the GPU time; the stage is the chain's unit).  For the
// stage's stride-2 output x1 (16 channels):
//     a   = act(s1 * conv1x1(x1) + b1)                  16 -> 8
//     b   = act(s2 * conv3x3(a) + b2)                   8 -> 8, pad 1
//     out = act(s3 * conv1x1([a | b]) + b3) + x1        16 -> 16, residual after the activation
// a and b never leave the SM: the three layer launches move about 1.15 GB
// through HBM at 320 x 320 batch 32 (a, b and the concat written and read
// back, x1 read twice); this kernel reads x1 and writes out, 0.42 GB.  The
// work is then about 985 multiply-adds per output pixel, so the FMA pipe,
// not HBM, bounds it, and the design keeps the instructions around the
// paired FMAs few:
//  * Persistent CTAs of 128 threads walk 4 x 32 output tiles, eight CTAs
//    per SM (20 KB of shared memory, at most 64 registers each): so many
//    warps per SM outweigh the 1x1's work over the tiles' halos (6 x 34
//    pixels for 4 x 32; measured at 320 x 320 batch 32: 179 us, against 195
//    us with 16 x 32 tiles and three CTAs per SM, 182-189 us for the shapes
//    in between).  x1 over the tile and its 1-pixel halo (16 channels)
//    arrives by one TMA copy per tile (zero outside the image), with the 64-byte
//    swizzle (bf16: 32-byte) that puts the k-th 16-byte piece of haloed
//    pixel p at k ^ (p / 2 % 4) (bf16: k ^ (p / 4 % 2)): eight neighbouring
//    pixels' pieces then fall in distinct banks.  The next tile's copy is
//    issued as soon as phase 1 has read this one.
//  * Phase 1: a over the haloed tile, two pixels per thread, into
//    shared memory; zero outside the image, which is the 3x3's padding (not
//    act(b1), what the 1x1 would give on the zero-filled x1).
//  * Phase 2: b as in the 8-channel 3x3 kernel (conv3x3_c8.cu): a thread owns
//    kRows output rows of one column (one at this tile height), loads each a
//    row once per filter column and 4-channel half and reuses it for the 3
//    filter rows; b stays in the thread's registers.
//  * Phase 3: out for the same pixels, 8 output channels per pass, from a
//    (the tile's centre, shared memory) and b (registers), the residual x1
//    from global memory (L2: the tile was just read).  Two barriers per
//    tile.
//  * Every product is a paired FMA (fma.rn.f32x2): an accumulator pair holds
//    the sums over the even and the odd input channels of one (pixel,
//    output channel), so that both operands come already paired: an input
//    channel pair from shared memory and the matching weight pair.
//  * The weights (and the folded BN) are in the launch's parameter block,
//    laid out [input channel pair][output channel][2]; every loop that reads
//    them is unrolled, so each read is a constant offset into the constant
//    bank and costs no load instruction and no shared-memory bandwidth (read
//    from shared memory, the weight pairs took most of the L1 bandwidth,
//    which bounded the kernel).
#include "epilogue.cuh"
#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"

#include <cuda_bf16.h>

namespace cb {
namespace {

constexpr int kTW = 32, kTH = 4;               // output tile
constexpr int kRows = 1;                       // output rows per thread (phases 2 and 3)
constexpr int kThreads = 32 * kTH / kRows;     // 128: one warp per kRows rows x 32 columns
constexpr int kMinBlocks = 8;                  // CTAs per SM (registers: 65536 / (128 x 8) = 64)
constexpr int kInW = kTW + 2, kInH = kTH + 2;  // the tile with its halo: where a is needed
constexpr int kInPx = kInW * kInH;             // 204
constexpr int kABytes = kInPx * 32;            // a: 8 fp32 channels over the haloed tile

template <typename T>
struct XTile {
  static constexpr int kPixBytes = 16 * static_cast<int>(sizeof(T));  // 64 (fp32) or 32 (bf16)
  static constexpr int kBytes = kInPx * kPixBytes;
  // Byte offset of channels 4q .. 4q + 3 of haloed pixel p in the swizzled tile.
  __device__ static int off(int p, int q) {
    if constexpr (sizeof(T) == 4) return p * 64 + ((q ^ ((p >> 1) & 3)) << 4);
    return p * 32 + (((q >> 1) ^ ((p >> 2) & 1)) << 4) + ((q & 1) << 3);
  }
};

template <typename T>
constexpr int smem_bytes() {
  return 1024 + XTile<T>::kBytes + kABytes + 16;
}

// a pixels: two 16-byte pieces (channels 0-3, 4-7) swizzled by column
// (the layout of conv3x3_c8.cu: a warp's 32 neighbouring columns conflict-free).
__device__ __forceinline__ int ab_off(int r, int c, int w, int j) {
  return (r * w + c) * 32 + ((j ^ ((c >> 2) & 1)) << 4);
}

template <typename T>
__device__ __forceinline__ float4 x_quad(const uint8_t* xt, int p, int q) {
  if constexpr (sizeof(T) == 4) return *reinterpret_cast<const float4*>(xt + XTile<T>::off(p, q));
  const uint2 v = *reinterpret_cast<const uint2*>(xt + XTile<T>::off(p, q));
  return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u), __uint_as_float(v.y << 16),
                     __uint_as_float(v.y & 0xFFFF0000u));
}

template <int ACT>
__device__ __forceinline__ float act_t(float z) {
  if constexpr (ACT == 1) return fmaxf(z, 0.0f);
  if constexpr (ACT == 2) return silu(z);
  return z;
}

template <int ACT, typename T>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
    stage_body_kernel(const __grid_constant__ CUtensorMap xmap, const StageBodyArgs a, int tiles_x, int tiles_y) {
  using X = XTile<T>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* const xt = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* const at = xt + X::kBytes;
  uint64_t* const xfull = reinterpret_cast<uint64_t*>(at + kABytes);
  const float* const w1 = a.w1;  // the parameter block: constant-bank reads
  const float* const w2 = a.w2;
  const float* const w3 = a.w3;
  const float* const sb = a.sb;
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(xfull + 1);

  const int num_tiles = a.N * tiles_y * tiles_x;
  auto issue = [&](int t) {  // thread 0: the TMA copy of tile t's haloed x1
    const int tx = t % tiles_x, rest = t / tiles_x, ty = rest % tiles_y, n = rest / tiles_y;
    mbar_arrive_expect_tx(xfull, static_cast<uint32_t>(X::kBytes));
    tma_load_4d(xt, &xmap, xfull, 0, tx * kTW - 1, ty * kTH - 1, n);
  };
  if (threadIdx.x == 0) {
    mbar_init(xfull, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&xmap);
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0 && static_cast<int>(blockIdx.x) < num_tiles) issue(blockIdx.x);
  const Watchdog wd{a.err, abort_flag, a.timeout_ns};
  const int col = threadIdx.x & 31, row0 = (threadIdx.x >> 5) * kRows;
  bool pending = false;  // thread 0: a copy issued and not yet waited for
  if (threadIdx.x == 0) pending = static_cast<int>(blockIdx.x) < num_tiles;
  int it = 0;
  for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
    const int tx = tile % tiles_x, rest = tile / tiles_x, ty = rest % tiles_y, n = rest / tiles_y;
    const int ih0 = ty * kTH - 1, iw0 = tx * kTW - 1;
    // this tile's x1 in place; every thread's phase 3 of the previous tile
    // is done with a
    if (!__syncthreads_and(mbar_wait(xfull, static_cast<uint32_t>(it) & 1u, wd))) break;
    if (threadIdx.x == 0) pending = false;

    // ------------------------------------------------ phase 1: a = act(bn(1x1(x1)))
    for (int p0 = threadIdx.x; p0 < kInPx; p0 += 2 * kThreads) {
      const int pp[2] = {p0, p0 + kThreads};
      const bool live1 = pp[1] < kInPx;
      float2 acc[2][8];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[i][q] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // input channels 4k .. 4k + 3
        float4 xq[2];
        xq[0] = x_quad<T>(xt, pp[0], k);
        xq[1] = live1 ? x_quad<T>(xt, pp[1], k) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // channel pair 2k + h
          const float* wp = w1 + (2 * k + h) * 16;
#pragma unroll
          for (int q = 0; q < 8; q += 2) {
            const float4 w4 = make_float4(wp[2 * q], wp[2 * q + 1], wp[2 * q + 2], wp[2 * q + 3]);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float2 xp = h ? make_float2(xq[i].z, xq[i].w) : make_float2(xq[i].x, xq[i].y);
              acc[i][q] = __ffma2_rn(xp, make_float2(w4.x, w4.y), acc[i][q]);
              acc[i][q + 1] = __ffma2_rn(xp, make_float2(w4.z, w4.w), acc[i][q + 1]);
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (i == 1 && !live1) break;
        const int r = pp[i] / kInW, c = pp[i] - r * kInW;
        const int ih = ih0 + r, iw = iw0 + c;
        // outside the image a is +0: every value computed, then masked (a select
        // made the compiler branch around each value's exponential)
        const uint32_t keep = ih >= 0 && ih < a.H && iw >= 0 && iw < a.W ? 0xFFFFFFFFu : 0u;
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          v[q] = __uint_as_float(__float_as_uint(act_t<ACT>(fmaf(acc[i][q].x + acc[i][q].y, sb[q], sb[8 + q]))) & keep);
        *reinterpret_cast<float4*>(at + ab_off(r, c, kInW, 0)) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(at + ab_off(r, c, kInW, 1)) = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
    __syncthreads();  // a complete; the x1 tile is free
    const int next = tile + gridDim.x;
    if (threadIdx.x == 0 && next < num_tiles) {
      issue(next);
      pending = true;
    }

    // ------------------------------------------------ phase 2: b = act(bn(3x3(a)))
    float bv[kRows][8];
    {
      float2 acc[kRows][8];
#pragma unroll
      for (int p = 0; p < kRows; ++p)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[p][q] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int kw = 0; kw < 3; ++kw) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {  // input channels 4j .. 4j + 3
          float4 xr[kRows + 2];
#pragma unroll
          for (int r = 0; r < kRows + 2; ++r)
            xr[r] = *reinterpret_cast<const float4*>(at + ab_off(row0 + r, col + kw, kInW, j));
#pragma unroll
          for (int kh = 0; kh < 3; ++kh) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // channel pair 2j + h
              const float* wp = w2 + ((kh * 3 + kw) * 4 + 2 * j + h) * 16;
#pragma unroll
              for (int q = 0; q < 8; q += 2) {
                const float4 w4 = make_float4(wp[2 * q], wp[2 * q + 1], wp[2 * q + 2], wp[2 * q + 3]);
#pragma unroll
                for (int p = 0; p < kRows; ++p) {
                  const float4 x4 = xr[p + kh];
                  const float2 xp = h ? make_float2(x4.z, x4.w) : make_float2(x4.x, x4.y);
                  acc[p][q] = __ffma2_rn(xp, make_float2(w4.x, w4.y), acc[p][q]);
                  acc[p][q + 1] = __ffma2_rn(xp, make_float2(w4.z, w4.w), acc[p][q + 1]);
                }
              }
            }
          }
        }
      }
#pragma unroll
      for (int p = 0; p < kRows; ++p)
#pragma unroll
        for (int q = 0; q < 8; ++q) bv[p][q] = act_t<ACT>(fmaf(acc[p][q].x + acc[p][q].y, sb[16 + q], sb[24 + q]));
    }

    // ------------------------------------------------ phase 3: out = act(bn(1x1([a | b]))) + x1
    const int ow = tx * kTW + col;
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // output channels 8 half .. 8 half + 7
      float2 acc[kRows][8];
#pragma unroll
      for (int p = 0; p < kRows; ++p)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[p][q] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // input channels 4j .. 4j + 3 of [a | b]
        float4 xr[kRows];
#pragma unroll
        for (int p = 0; p < kRows; ++p)
          xr[p] = j < 2 ? *reinterpret_cast<const float4*>(at + ab_off(row0 + p + 1, col + 1, kInW, j))
                        : make_float4(bv[p][4 * (j - 2)], bv[p][4 * (j - 2) + 1], bv[p][4 * (j - 2) + 2],
                                      bv[p][4 * (j - 2) + 3]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // channel pair 2j + h
          const float* wp = w3 + (2 * j + h) * 32 + half * 16;
#pragma unroll
          for (int q = 0; q < 8; q += 2) {
            const float4 w4 = make_float4(wp[2 * q], wp[2 * q + 1], wp[2 * q + 2], wp[2 * q + 3]);
#pragma unroll
            for (int p = 0; p < kRows; ++p) {
              const float2 xp = h ? make_float2(xr[p].z, xr[p].w) : make_float2(xr[p].x, xr[p].y);
              acc[p][q] = __ffma2_rn(xp, make_float2(w4.x, w4.y), acc[p][q]);
              acc[p][q + 1] = __ffma2_rn(xp, make_float2(w4.z, w4.w), acc[p][q + 1]);
            }
          }
        }
      }
#pragma unroll
      for (int p = 0; p < kRows; ++p) {
        const int oh = ty * kTH + row0 + p;
        if (oh >= a.H || ow >= a.W) continue;
        const T* rp = reinterpret_cast<const T*>(a.x) + n * a.xs_n + oh * a.xs_h + ow * a.xs_w + 8 * half;
        T* yp = reinterpret_cast<T*>(a.y) + n * a.ys_n + oh * a.ys_h + ow * a.ys_w + 8 * half;
        const float4 r0 = load4(rp), r1 = load4(rp + 4);
        const float r[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          v[q] = act_t<ACT>(fmaf(acc[p][q].x + acc[p][q].y, sb[32 + 8 * half + q], sb[48 + 8 * half + q])) + r[q];
        store4(yp, make_float4(v[0], v[1], v[2], v[3]));
        store4(yp + 4, make_float4(v[4], v[5], v[6], v[7]));
      }
    }
  }
  // after a timeout: let a copy still in flight land before the CTA exits
  if (pending) mbar_wait_drain(xfull, static_cast<uint32_t>(it) & 1u, 20000000ull);
}

template <int ACT, typename T>
cudaError_t launch_t(const CUtensorMap& xmap, const StageBodyArgs& a, int sms, cudaStream_t s) {
  constexpr size_t smem = smem_bytes<T>();
  cudaError_t e = smem_attr_once<stage_body_kernel<ACT, T>>(smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stage_body_kernel<ACT, T>, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int tiles_x = (a.W + kTW - 1) / kTW, tiles_y = (a.H + kTH - 1) / kTH;
  const long long tiles = static_cast<long long>(a.N) * tiles_x * tiles_y;
  if (tiles >= (1LL << 31) - static_cast<long long>(sms) * per_sm) return cudaErrorInvalidValue;
  const long long cap = static_cast<long long>(sms) * per_sm;
  const unsigned grid = static_cast<unsigned>(tiles < cap ? tiles : cap);
  return launch_pdl(stage_body_kernel<ACT, T>, dim3(grid), dim3(kThreads), smem, s, xmap, a, tiles_x, tiles_y);
}

template <typename T>
cudaError_t launch_type(const CUtensorMap& xmap, const StageBodyArgs& a, int sms, cudaStream_t s) {
  if (a.act == 0) return launch_t<0, T>(xmap, a, sms, s);
  if (a.act == 1) return launch_t<1, T>(xmap, a, sms, s);
  return launch_t<2, T>(xmap, a, sms, s);
}

}  // namespace

void stage_body_box(int* box_c, int* box_w, int* box_h) {
  *box_c = 16;
  *box_w = kInW;
  *box_h = kInH;
}

cudaError_t launch_stage_body(const CUtensorMap& xmap, const StageBodyArgs& a, int sms, cudaStream_t s) {
  if (a.N == 0 || a.H == 0 || a.W == 0) return cudaSuccess;
  return a.bf16 ? launch_type<__nv_bfloat16>(xmap, a, sms, s) : launch_type<float>(xmap, a, sms, s);
}

}  // namespace cb
