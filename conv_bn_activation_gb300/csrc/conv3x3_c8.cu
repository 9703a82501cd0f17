// 3x3 stride-1 pad-1 convolution with 8 input and 8 output channels, fp32
// on the CUDA cores, with the fused folded-BN / residual / activation
// epilogue: the 8 -> 8 channel layer of the YOLO-style chain's first stage
// ("YOLO26N Inference Optimisation": the conv2d_bn_silu kernels hold most of
// the GPU time, and the per-layer variance is the signal to chase).
//
// At 576 multiply-adds per output pixel the layer is bound by the FMA pipe,
// not by HBM, so the design minimises the instructions around the FMAs:
//  * Input tiles (18 x 34 pixels for 16 x 32 outputs) stay NHWC in shared
//    memory: 16-byte cp.async copies of 4 channels (zero-filled outside the
//    image, which is the padding), double-buffered over persistent CTAs of
//    four warps, four CTAs per SM (measured: 97 us against 104 us with
//    32-row tiles in eight-warp CTAs, two per SM, whose staging and
//    epilogue phases left the FMA pipe idle more of the time; 99 us with
//    8-row tiles).
//    The two 16-byte halves of a pixel are XOR-swizzled by column so that a
//    warp's 16-byte loads of 32 neighbouring pixels are conflict-free.
//  * The products go out as packed pairs (fma.rn.f32x2, each lane an fmaf):
//    an accumulator pair holds the sums over the even and the odd input
//    channels of one (pixel, output channel), so both operands of every
//    packed FMA come from memory already paired -- an input channel pair of
//    one pixel (half of a 16-byte load) and the matching weight pair, which
//    the weights' shared-memory layout [tap][channel pair][co][2] provides.
//    The two halves are added once per output.
//  * A thread owns 4 output rows of one column (all 8 channels); per filter
//    column and 4-channel half it loads the 6 input rows once and reuses
//    them for the three filter rows.
#include "epilogue.cuh"
#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"

namespace cb {
namespace {

constexpr int kC8Rows = 4;                   // output rows per thread
constexpr int kC8TileW = 32, kC8TileH = 16;  // output tile
constexpr int kC8Threads = 32 * kC8TileH / kC8Rows;  // one warp per 4 rows x 32 columns
constexpr int kC8MinBlocks = 512 / kC8Threads;       // 16 warps per SM at 128 registers
constexpr int kC8InW = kC8TileW + 2, kC8InH = kC8TileH + 2;
constexpr int kC8WFloats = 9 * 4 * 8 * 2;            // [tap][channel pair][co][2]
// T: the storage type of x, y and the residual (fp32, or bf16 widened to
// fp32 as it leaves shared memory; the arithmetic is fp32 either way)
template <typename T>
constexpr int c8_tile_bytes() { return kC8InH * kC8InW * 8 * static_cast<int>(sizeof(T)); }
template <typename T>
constexpr int c8_smem_bytes() { return 2 * c8_tile_bytes<T>() + (kC8WFloats + 16) * 4; }  // tiles, weights, BN

// Byte offset of the 16-byte piece j of staged pixel (r, c): fp32 pixels are
// two pieces (4 channels each), XOR-swizzled by column; a bf16 pixel is one.
template <typename T>
__device__ __forceinline__ int c8_off(int r, int c, int j) {
  if constexpr (sizeof(T) == 2) return (r * kC8InW + c) * 16;
  return (r * kC8InW + c) * 32 + ((j ^ ((c >> 2) & 1)) << 4);
}

// Channels 4j .. 4j + 3 of a staged pixel as fp32.
template <typename T>
__device__ __forceinline__ float4 c8_load4(const uint8_t* xs, int r, int c, int j) {
  if constexpr (sizeof(T) == 2) return load4(reinterpret_cast<const __nv_bfloat16*>(xs + c8_off<T>(r, c, 0)) + 4 * j);
  return *reinterpret_cast<const float4*>(xs + c8_off<T>(r, c, j));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool in) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(in ? 16 : 0) : "memory");
}

// sb: the 8 scales then the 8 biases, in shared memory.
template <int ACT, int RES, typename T>
__device__ __forceinline__ void c8_store(const float2 (&acc)[8], const float* sb, T* yp, const T* rp) {
  float o[8];
#pragma unroll
  for (int q = 0; q < 8; q += 4) {
    const float4 s4 = *reinterpret_cast<const float4*>(sb + q), b4 = *reinterpret_cast<const float4*>(sb + 8 + q);
    // the even- and odd-channel halves, then scale and bias two channels at a time
    const float2 z0 = __ffma2_rn(make_float2(acc[q].x + acc[q].y, acc[q + 1].x + acc[q + 1].y),
                                 make_float2(s4.x, s4.y), make_float2(b4.x, b4.y));
    const float2 z1 = __ffma2_rn(make_float2(acc[q + 2].x + acc[q + 2].y, acc[q + 3].x + acc[q + 3].y),
                                 make_float2(s4.z, s4.w), make_float2(b4.z, b4.w));
    o[q] = z0.x, o[q + 1] = z0.y, o[q + 2] = z1.x, o[q + 3] = z1.y;
  }
  float r[8] = {};
  if constexpr (RES != 0) {
    const float4 r0 = load4(rp), r1 = load4(rp + 4);
    r[0] = r0.x, r[1] = r0.y, r[2] = r0.z, r[3] = r0.w, r[4] = r1.x, r[5] = r1.y, r[6] = r1.z, r[7] = r1.w;
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    float z = o[q];
    if constexpr (RES == 1) z += r[q];
    if constexpr (ACT == 1) z = fmaxf(z, 0.0f);
    if constexpr (ACT == 2) z = silu(z);
    if constexpr (RES == 2) z += r[q];
    o[q] = z;
  }
  store4(yp, make_float4(o[0], o[1], o[2], o[3]));
  store4(yp + 4, make_float4(o[4], o[5], o[6], o[7]));
}

template <int ACT, int RES, typename T>
__global__ void __launch_bounds__(kC8Threads, kC8MinBlocks) conv3x3_c8_kernel(const DirectArgs a, int tiles_x, int tiles_y) {
  constexpr int kC8TileBytes = c8_tile_bytes<T>();
  constexpr int kPieces = sizeof(T) == 2 ? 1 : 2;  // 16-byte pieces per pixel
  extern __shared__ __align__(16) uint8_t c8_smem[];
  float* ws = reinterpret_cast<float*>(c8_smem + 2 * kC8TileBytes);
  pdl_wait();
  pdl_launch_dependents();
  // weights [co][tap][ci] (OHWI) -> [tap][ci / 2][co][ci % 2]
  for (int i = threadIdx.x; i < kC8WFloats; i += kC8Threads) {
    const int e = i & 1, co = (i >> 1) & 7, cp = (i >> 4) & 3, tap = i >> 6;
    ws[i] = __ldg(a.w + (co * 9 + tap) * 8 + 2 * cp + e);
  }
  float* sb = ws + kC8WFloats;
  if (threadIdx.x < 16) sb[threadIdx.x] = __ldg(threadIdx.x < 8 ? a.ep.scale + threadIdx.x : a.ep.bias + threadIdx.x - 8);

  const int num_tiles = a.N * tiles_y * tiles_x;
  const uint32_t s0 = smem_u32(c8_smem);
  // The sixteen-byte copies of a tile's (kC8InH x kC8InW) pixels, spread over the threads.
  auto stage = [&](int t, uint32_t buf) {
    const int tx = t % tiles_x, ty = (t / tiles_x) % tiles_y, n = t / (tiles_x * tiles_y);
    const int ih0 = ty * kC8TileH - 1, iw0 = tx * kC8TileW - 1;
    const T* x = reinterpret_cast<const T*>(a.x);
    const T* xn = x + n * a.xs_n;
    for (int i = threadIdx.x; i < kC8InH * kC8InW * kPieces; i += kC8Threads) {
      const int r = i / (kC8InW * kPieces), rem = i - r * (kC8InW * kPieces);
      const int c = rem / kPieces, j = rem - c * kPieces;
      const int ih = ih0 + r, iw = iw0 + c;
      const bool in = ih >= 0 && ih < a.H && iw >= 0 && iw < a.W;
      cp_async16(buf + c8_off<T>(r, c, j), in ? xn + ih * a.xs_h + iw * a.xs_w + (16 / sizeof(T)) * j : x, in);
    }
  };

  const int col = threadIdx.x & 31, row0 = (threadIdx.x >> 5) * kC8Rows;
  int tile = blockIdx.x;
  if (tile < num_tiles) stage(tile, s0);
  asm volatile("cp.async.commit_group;" ::: "memory");
  for (int it = 0; tile < num_tiles; tile += gridDim.x, ++it) {
    const int next = tile + gridDim.x;
    if (next < num_tiles) stage(next, s0 + ((it + 1) & 1) * kC8TileBytes);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");  // this tile (and, the first time, the weights)
    __syncthreads();

    const uint8_t* xs = c8_smem + (it & 1) * kC8TileBytes;
    float2 acc[kC8Rows][8];
#pragma unroll
    for (int p = 0; p < kC8Rows; ++p)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[p][q] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int kw = 0; kw < 3; ++kw) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {  // input channels 4j .. 4j + 3
        float4 xr[kC8Rows + 2];
#pragma unroll
        for (int r = 0; r < kC8Rows + 2; ++r)
          xr[r] = c8_load4<T>(xs, row0 + r, col + kw, j);
#pragma unroll
        for (int kh = 0; kh < 3; ++kh) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // channel pair 2j + h
            const float* wp = ws + ((kh * 3 + kw) * 4 + 2 * j + h) * 16;
#pragma unroll
            for (int q = 0; q < 8; q += 2) {
              const float4 w4 = *reinterpret_cast<const float4*>(wp + 2 * q);  // (c, c+1) for co q, then co q + 1
#pragma unroll
              for (int p = 0; p < kC8Rows; ++p) {
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

    const int tx = tile % tiles_x, ty = (tile / tiles_x) % tiles_y, n = tile / (tiles_x * tiles_y);
    const int ow = tx * kC8TileW + col;
#pragma unroll
    for (int p = 0; p < kC8Rows; ++p) {
      const int oh = ty * kC8TileH + row0 + p;
      if (oh >= a.OH || ow >= a.OW) continue;
      T* yp = reinterpret_cast<T*>(a.out.y) + n * a.out.ys_n + oh * a.out.ys_h + ow * a.out.ys_w;
      const T* rp =
          RES ? reinterpret_cast<const T*>(a.ep.r) + n * a.ep.rs_n + oh * a.ep.rs_h + ow * a.ep.rs_w : nullptr;
      c8_store<ACT, RES, T>(acc[p], sb, yp, rp);
    }
    __syncthreads();  // a later tile's copies overwrite this buffer
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

template <int ACT, int RES, typename T>
cudaError_t launch_c8(const DirectArgs& a, int sms, cudaStream_t s) {
  constexpr size_t smem = c8_smem_bytes<T>();
  cudaError_t e = smem_attr_once<conv3x3_c8_kernel<ACT, RES, T>>(smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, conv3x3_c8_kernel<ACT, RES, T>, kC8Threads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int tiles_x = (a.OW + kC8TileW - 1) / kC8TileW, tiles_y = (a.OH + kC8TileH - 1) / kC8TileH;
  const long long tiles = static_cast<long long>(a.N) * tiles_x * tiles_y;
  if (tiles >= (1LL << 31)) return cudaErrorInvalidValue;
  const long long cap = static_cast<long long>(sms) * per_sm;
  const unsigned grid = static_cast<unsigned>(tiles < cap ? tiles : cap);
  return launch_pdl(conv3x3_c8_kernel<ACT, RES, T>, dim3(grid), dim3(kC8Threads), smem, s, a, tiles_x, tiles_y);
}

template <typename T>
cudaError_t launch_c8_t(const DirectArgs& a, int sms, cudaStream_t s) {
  switch (a.ep.act * 3 + a.ep.res_mode) {
    case 0: return launch_c8<0, 0, T>(a, sms, s);
    case 1: return launch_c8<0, 1, T>(a, sms, s);
    case 2: return launch_c8<0, 2, T>(a, sms, s);
    case 3: return launch_c8<1, 0, T>(a, sms, s);
    case 4: return launch_c8<1, 1, T>(a, sms, s);
    case 5: return launch_c8<1, 2, T>(a, sms, s);
    case 6: return launch_c8<2, 0, T>(a, sms, s);
    case 7: return launch_c8<2, 1, T>(a, sms, s);
    default: return launch_c8<2, 2, T>(a, sms, s);
  }
}

}  // namespace

bool conv3x3_c8_ok(const DirectArgs& a) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  // x pixels in 16-byte pieces (fp32: strides multiples of 4 elements, bf16
  // of 8); y and the residual in 16-byte (fp32) or 8-byte (bf16) pieces
  const long long xm = a.bf16 ? 8 : 4;
  const bool res_ok = a.ep.res_mode == 0 || (al16(a.ep.r) && a.ep.rs_n % 4 == 0 && a.ep.rs_h % 4 == 0 && a.ep.rs_w % 4 == 0);
  return a.Ci == 8 && a.Co == 8 && a.kh == 3 && a.kw == 3 && a.stride == 1 && a.pad == 1 && a.xs_c == 1 &&
         al16(a.x) && a.xs_n % xm == 0 && a.xs_h % xm == 0 && a.xs_w % xm == 0 && al16(a.out.y) &&
         a.out.ys_n % 4 == 0 && a.out.ys_h % 4 == 0 && a.out.ys_w % 4 == 0 && res_ok && a.N > 0;
}

cudaError_t launch_conv3x3_c8(const DirectArgs& a, int sms, cudaStream_t s) {
  if (!conv3x3_c8_ok(a)) return cudaErrorInvalidValue;
  return a.bf16 ? launch_c8_t<__nv_bfloat16>(a, sms, s) : launch_c8_t<float>(a, sms, s);
}

}  // namespace cb
