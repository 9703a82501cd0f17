// u8 frame preprocess: bilinear resize (half-pixel centres) -> u8 rounding ->
// /255 -> planar fp32, as one pass ("A fused Ampere preprocess kernel", path
// B) and as three passes (path A: resize, normalize, layout) for comparison.
//
// Fused kernel layout: one CTA per (destination row, frame).  The CTA copies
// the two source rows its samples need into shared memory with 16-byte
// coalesced loads (the page found its fused kernel's 16 scalar u8 reads per
// thread to be the weak side), then each thread produces 4 consecutive
// destination pixels of all three channels and writes one float4 per
// channel plane.  Each u8 byte is read from DRAM once per frame (row reuse
// between neighbouring destination rows hits L2) and each fp32 output is
// written once.
//
// Arithmetic (coordinates, weights, the bilinear value, the u8 rounding and
// the division) is IEEE fp32 with every operation rounded separately, in the
// order: f = (d + 0.5) * (S / D) - 0.5; i0 = floor(f); a = f - i0 (border
// clamps); v = (1-ay)*((1-ax)*p00 + ax*p01) + ay*((1-ax)*p10 + ax*p11);
// u = floor(v + 0.5); out = u / 255.
#include <cstdint>

#include "internal.h"

namespace cb {

struct AxisSample {
  int i0, i1;
  float a;
};

__device__ __forceinline__ AxisSample axis_sample(int d, int S, int D) {
  const float scale = __fdiv_rn(static_cast<float>(S), static_cast<float>(D));
  const float f = __fsub_rn(__fmul_rn(__fadd_rn(static_cast<float>(d), 0.5f), scale), 0.5f);
  const float fl = floorf(f);
  int k = static_cast<int>(fl);
  float t = __fsub_rn(f, fl);
  if (k < 0) {
    k = 0;
    t = 0.0f;
  }
  if (k >= S - 1) {
    k = S - 1;
    t = 0.0f;
  }
  AxisSample s;
  s.i0 = k;
  s.i1 = (k + 1 < S) ? k + 1 : S - 1;
  s.a = t;
  return s;
}

__device__ __forceinline__ float bilinear(float p00, float p01, float p10, float p11, float ax, float ay) {
  const float bx = __fsub_rn(1.0f, ax), by = __fsub_rn(1.0f, ay);
  const float top = __fadd_rn(__fmul_rn(bx, p00), __fmul_rn(ax, p01));
  const float bot = __fadd_rn(__fmul_rn(bx, p10), __fmul_rn(ax, p11));
  return __fadd_rn(__fmul_rn(by, top), __fmul_rn(ay, bot));
}

__device__ __forceinline__ float round_u8(float v) {
  float u = floorf(__fadd_rn(v, 0.5f));
  return fminf(fmaxf(u, 0.0f), 255.0f);
}

// Copy `bytes` bytes of a source row into shared memory.
__device__ __forceinline__ void stage_row(uint8_t* dst, const uint8_t* src, int bytes, bool vec) {
  if (vec) {
    const int n16 = bytes >> 4;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (int i = threadIdx.x; i < n16; i += blockDim.x) d4[i] = __ldg(s4 + i);
    for (int i = (n16 << 4) + threadIdx.x; i < bytes; i += blockDim.x) dst[i] = __ldg(src + i);
  } else {
    for (int i = threadIdx.x; i < bytes; i += blockDim.x) dst[i] = __ldg(src + i);
  }
}

template <bool TO_U8>
__global__ void __launch_bounds__(256) preprocess_row_kernel(const uint8_t* __restrict__ src, int hs, int ws,
                                                             long long pitch, void* __restrict__ out, int hd,
                                                             int wd, int vec_in, int vec_out) {
  extern __shared__ __align__(16) uint8_t rows[];
  const int row_bytes = ws * 3;
  const int row_alloc = (row_bytes + 15) & ~15;
  const int dy = blockIdx.x, n = blockIdx.y;
  const AxisSample sy = axis_sample(dy, hs, hd);
  const uint8_t* frame = src + static_cast<long long>(n) * hs * pitch;
  uint8_t* r0 = rows;
  uint8_t* r1 = rows + row_alloc;
  stage_row(r0, frame + sy.i0 * pitch, row_bytes, vec_in != 0);
  stage_row(r1, frame + sy.i1 * pitch, row_bytes, vec_in != 0);
  __syncthreads();

  const int groups = (wd + 3) >> 2;
  for (int g = threadIdx.x; g < groups; g += blockDim.x) {
    float o[3][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int dx = g * 4 + q;
      if (dx < wd) {
        const AxisSample sx = axis_sample(dx, ws, wd);
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const float p00 = r0[sx.i0 * 3 + c], p01 = r0[sx.i1 * 3 + c];
          const float p10 = r1[sx.i0 * 3 + c], p11 = r1[sx.i1 * 3 + c];
          o[c][q] = round_u8(bilinear(p00, p01, p10, p11, sx.a, sy.a));
        }
      } else {
#pragma unroll
        for (int c = 0; c < 3; ++c) o[c][q] = 0.0f;
      }
    }
    if (TO_U8) {
      uint8_t* op = static_cast<uint8_t*>(out) + (static_cast<long long>(n) * hd + dy) * wd * 3;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int dx = g * 4 + q;
        if (dx < wd)
          for (int c = 0; c < 3; ++c) op[dx * 3 + c] = static_cast<uint8_t>(o[c][q]);
      }
    } else {
      float* base = static_cast<float*>(out);
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        float* op = base + ((static_cast<long long>(n) * 3 + c) * hd + dy) * wd;
        const float4 v = make_float4(__fdiv_rn(o[c][0], 255.0f), __fdiv_rn(o[c][1], 255.0f),
                                     __fdiv_rn(o[c][2], 255.0f), __fdiv_rn(o[c][3], 255.0f));
        if (vec_out && g * 4 + 3 < wd) {
          *reinterpret_cast<float4*>(op + g * 4) = v;
        } else {
          const float vv[4] = {v.x, v.y, v.z, v.w};
          for (int q = 0; q < 4; ++q)
            if (g * 4 + q < wd) op[g * 4 + q] = vv[q];
        }
      }
    }
  }
}

static size_t row_smem(int ws) { return 2 * static_cast<size_t>((ws * 3 + 15) & ~15); }

template <bool TO_U8>
static cudaError_t launch_rows(const uint8_t* src, int n, int hs, int ws, long long pitch, void* out, int hd, int wd,
                               bool vec_out, cudaStream_t s) {
  if (n == 0 || hd == 0 || wd == 0) return cudaSuccess;
  const bool vec_in = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (pitch % 16 == 0);
  const size_t smem = row_smem(ws);
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(preprocess_row_kernel<TO_U8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
  int threads = ((wd + 3) / 4 + 31) / 32 * 32;
  if (threads > 256) threads = 256;
  if (threads < 64) threads = 64;
  dim3 grid(hd, n);
  preprocess_row_kernel<TO_U8><<<grid, threads, smem, s>>>(src, hs, ws, pitch, out, hd, wd, vec_in ? 1 : 0,
                                                           vec_out ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_preprocess_fused(const uint8_t* src, int n, int hs, int ws, long long pitch, float* dst, int hd,
                                    int wd, cudaStream_t s) {
  const bool vec_out = (reinterpret_cast<uintptr_t>(dst) % 16 == 0) && (wd % 4 == 0);
  return launch_rows<false>(src, n, hs, ws, pitch, dst, hd, wd, vec_out, s);
}

cudaError_t launch_preprocess_resize(const uint8_t* src, int n, int hs, int ws, long long pitch, uint8_t* out,
                                     int hd, int wd, cudaStream_t s) {
  return launch_rows<true>(src, n, hs, ws, pitch, out, hd, wd, false, s);
}

// Pass 2: u8 -> fp32 / 255 (HWC kept).
__global__ void __launch_bounds__(256) normalize_kernel(const uint8_t* __restrict__ in, long long count,
                                                        float* __restrict__ out) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < count; i += stride)
    out[i] = __fdiv_rn(static_cast<float>(in[i]), 255.0f);
}

cudaError_t launch_preprocess_normalize(const uint8_t* in, long long count, float* out, cudaStream_t s) {
  if (count == 0) return cudaSuccess;
  long long blocks = (count + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  normalize_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(in, count, out);
  return cudaGetLastError();
}

// Pass 3: fp32 HWC [n, h, w, 3] -> fp32 CHW [n, 3, h, w].
__global__ void __launch_bounds__(256) layout_kernel(const float* __restrict__ in, int n, int h, int w,
                                                     float* __restrict__ out) {
  const long long plane = static_cast<long long>(h) * w;
  const long long total = static_cast<long long>(n) * plane;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total; i += stride) {
    const long long img = i / plane, p = i - img * plane;
    const float* src = in + i * 3;
    float* dst = out + img * 3 * plane + p;
    dst[0] = src[0];
    dst[plane] = src[1];
    dst[2 * plane] = src[2];
  }
}

cudaError_t launch_preprocess_layout(const float* in, int n, int h, int w, float* out, cudaStream_t s) {
  const long long total = static_cast<long long>(n) * h * w;
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  layout_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(in, n, h, w, out);
  return cudaGetLastError();
}

}  // namespace cb
