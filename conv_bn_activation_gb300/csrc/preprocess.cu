// u8 frame preprocess: bilinear resize (half-pixel centres) -> u8 rounding ->
// /255 -> planar fp32, as one pass ("A fused Ampere preprocess kernel", path
// B) and as three passes (path A: resize, normalize, layout) for comparison.
//
// Kernel layout: one CTA per (destination row pair, frame) for the fused
// path (one per destination row for the u8 resize pass of the three-pass
// path).  The CTA copies the source rows its samples need into shared
// memory with 16-byte coalesced loads (the page found its fused kernel's 16
// scalar u8 reads per thread to be the weak side), then each thread
// produces 4 consecutive destination pixels of all three channels and
// writes one float4 per channel plane.  Each u8 byte is read from DRAM once
// per frame (row reuse between neighbouring CTAs hits L2) and each fp32
// output is written once.
//
// Arithmetic (coordinates, weights, the bilinear value, the u8 rounding and
// the division) is IEEE fp32 with every operation rounded separately, in the
// order: f = (d + 0.5) * (S / D) - 0.5; i0 = floor(f); a = f - i0 (border
// clamps); v = (1-ay)*((1-ax)*p00 + ax*p01) + ay*((1-ax)*p10 + ax*p11);
// u = floor(v + 0.5); out = u / 255.
#include <cstdint>

#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"
#include "resample.cuh"

namespace cb {

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
  pdl_wait();
  pdl_launch_dependents();
  // u / 255 for every u8 code, each an IEEE fp32 division, looked up instead
  // of divided per output.
  __shared__ float inv255[256];
  extern __shared__ __align__(16) uint8_t rows[];
  if (!TO_U8)
    for (int i = threadIdx.x; i < 256; i += blockDim.x) inv255[i] = __fdiv_rn(static_cast<float>(i), 255.0f);
  const int row_bytes = ws * 3;
  const int row_alloc = (row_bytes + 15) & ~15;
  const int dy = blockIdx.x, n = blockIdx.y;
  const float scale_x = __fdiv_rn(static_cast<float>(ws), static_cast<float>(wd));
  const AxisSample sy = axis_sample(dy, hs, __fdiv_rn(static_cast<float>(hs), static_cast<float>(hd)));
  const uint8_t* frame = src + static_cast<long long>(n) * hs * pitch;
  uint8_t* r0 = rows;
  uint8_t* r1 = rows + row_alloc;
  stage_row(r0, frame + sy.i0 * pitch, row_bytes, vec_in != 0);
  stage_row(r1, frame + sy.i1 * pitch, row_bytes, vec_in != 0);
  __syncthreads();

  const int groups = (wd + 3) >> 2;
  // 2:1 horizontal ratio (the 1280 -> 640 workload): destination column dx
  // samples source columns 2dx and 2dx + 1 with weight 1/2 (what axis_sample
  // gives for it), so 4 destination pixels read 24 consecutive bytes per row,
  // fetched as six 32-bit words.
  const bool two_to_one = (ws == 2 * wd) && (row_alloc % 8 == 0);
  for (int g = threadIdx.x; g < groups; g += blockDim.x) {
    int o[3][4];
    if (two_to_one && g * 4 + 3 < wd) {
      const uint32_t* w0 = reinterpret_cast<const uint32_t*>(r0 + g * 24);
      const uint32_t* w1 = reinterpret_cast<const uint32_t*>(r1 + g * 24);
      uint32_t a0[6], a1[6];
#pragma unroll
      for (int i = 0; i < 6; ++i) a0[i] = w0[i], a1[i] = w1[i];
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const int b0 = q * 6 + c, b1 = q * 6 + 3 + c;  // byte offsets of the two samples
          const float p00 = u8_to_float((a0[b0 >> 2] >> ((b0 & 3) * 8)) & 0xFF);
          const float p01 = u8_to_float((a0[b1 >> 2] >> ((b1 & 3) * 8)) & 0xFF);
          const float p10 = u8_to_float((a1[b0 >> 2] >> ((b0 & 3) * 8)) & 0xFF);
          const float p11 = u8_to_float((a1[b1 >> 2] >> ((b1 & 3) * 8)) & 0xFF);
          o[c][q] = round_u8(bilinear(p00, p01, p10, p11, 0.5f, sy.a));
        }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int dx = g * 4 + q;
        if (dx < wd) {
          const AxisSample sx = axis_sample(dx, ws, scale_x);
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            const float p00 = u8_to_float(r0[sx.i0 * 3 + c]), p01 = u8_to_float(r0[sx.i1 * 3 + c]);
            const float p10 = u8_to_float(r1[sx.i0 * 3 + c]), p11 = u8_to_float(r1[sx.i1 * 3 + c]);
            o[c][q] = round_u8(bilinear(p00, p01, p10, p11, sx.a, sy.a));
          }
        } else {
#pragma unroll
          for (int c = 0; c < 3; ++c) o[c][q] = 0;
        }
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
        const float4 v = make_float4(inv255[o[c][0]], inv255[o[c][1]], inv255[o[c][2]], inv255[o[c][3]]);
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

// 16-byte asynchronous global -> shared copy.
__device__ __forceinline__ void cp_async16_pp(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// The source rows of one destination row pair: 0 = s0.i0, 1 = s0.i1,
// 2 = s1.i0 (or slot 1 again when it is the same row), 3 = s1.i1.
struct PairRows {
  AxisSample s0, s1;
  bool two_rows, shared_row;
};

__device__ __forceinline__ PairRows pair_rows(int dy0, int hs, int hd, float scale_y) {
  PairRows r;
  r.two_rows = dy0 + 1 < hd;
  r.s0 = axis_sample(dy0, hs, scale_y);
  r.s1 = r.two_rows ? axis_sample(dy0 + 1, hs, scale_y) : r.s0;
  r.shared_row = r.s1.i0 == r.s0.i1;
  return r;
}

// Fused path: persistent CTAs walk (destination row pair, frame) items.  The
// two rows of a pair share a source row whenever the height ratio is below
// 2 (720 -> 480: rows 3k, 3k+1 and 3k+1, 3k+2), which is then staged and
// summed once.  The source rows of the next item are copied (cp.async)
// into the second of two shared-memory buffers while the current item is
// computed.  At a 2:1 width ratio the value is
//   by * ((p00 + p01) / 2) + ay * ((p10 + p11) / 2)
// with each product and the sum rounded separately -- the same IEEE
// operations as bilinear() with ax = 1/2, the halving moved into the row
// weights (hb = by / 2, exact) -- then the same u8 rounding and /255 table.
// async_rows: 16-byte aligned source rows of a multiple of 16 bytes (else
// each item stages its rows synchronously).
__global__ void __launch_bounds__(256) preprocess_pair_kernel(const uint8_t* __restrict__ src, int n, int hs, int ws,
                                                              long long pitch, float* __restrict__ out, int hd,
                                                              int wd, int async_rows, int vec_in, int vec_out) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float inv255[256];
  extern __shared__ __align__(16) uint8_t rows[];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) inv255[i] = __fdiv_rn(static_cast<float>(i), 255.0f);
  const int row_bytes = ws * 3;
  const int row_alloc = (row_bytes + 15) & ~15;
  const int pairs = (hd + 1) / 2;
  const int items = pairs * n;
  const float scale_x = __fdiv_rn(static_cast<float>(ws), static_cast<float>(wd));
  const float scale_y = __fdiv_rn(static_cast<float>(hs), static_cast<float>(hd));
  const int groups = (wd + 3) >> 2;
  const bool two_to_one = (ws == 2 * wd) && (row_alloc % 8 == 0);
  auto slots = [&](int buf, uint8_t* (&sl)[4], bool shared_row) {
    uint8_t* base = rows + static_cast<size_t>(buf) * 4 * row_alloc;
    sl[0] = base;
    sl[1] = base + row_alloc;
    sl[2] = shared_row ? sl[1] : base + 2 * row_alloc;
    sl[3] = base + 3 * row_alloc;
  };
  // Copies the source rows of `item` into buffer `buf` (asynchronously when
  // async_rows, else with plain loads).
  auto stage_item = [&](int item, int buf) {
    const int f = item / pairs, dy0 = (item - f * pairs) * 2;
    const PairRows pr = pair_rows(dy0, hs, hd, scale_y);
    uint8_t* sl[4];
    slots(buf, sl, pr.shared_row);
    const uint8_t* frame = src + static_cast<long long>(f) * hs * pitch;
    const int src_rows[4] = {pr.s0.i0, pr.s0.i1, pr.s1.i0, pr.s1.i1};
    const bool need[4] = {true, true, pr.two_rows && !pr.shared_row, pr.two_rows};
    if (async_rows) {
      const int chunks = row_bytes >> 4;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (!need[k]) continue;
        const uint8_t* rp = frame + src_rows[k] * pitch;
        for (int i = threadIdx.x; i < chunks; i += blockDim.x) cp_async16_pp(sl[k] + 16 * i, rp + 16 * i);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (need[k]) stage_row(sl[k], frame + src_rows[k] * pitch, row_bytes, vec_in != 0);
    }
  };

  int item = blockIdx.x;
  if (item < items) stage_item(item, 0);
  asm volatile("cp.async.commit_group;" ::: "memory");
  for (int it = 0; item < items; item += gridDim.x, ++it) {
    const int buf = it & 1;
    const int next = item + gridDim.x;
    if (next < items) stage_item(next, buf ^ 1);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");  // this item's rows have landed
    __syncthreads();

    const int f = item / pairs, dy0 = (item - f * pairs) * 2;
    const PairRows pr = pair_rows(dy0, hs, hd, scale_y);
    uint8_t* sl[4];
    slots(buf, sl, pr.shared_row);
    const float hb0 = 0.5f * __fsub_rn(1.0f, pr.s0.a), ha0 = 0.5f * pr.s0.a;
    const float hb1 = 0.5f * __fsub_rn(1.0f, pr.s1.a), ha1 = 0.5f * pr.s1.a;
    // One destination row at a time (fewer live registers, more CTAs per SM).
    auto store_row = [&](int g, int j, const int (&o)[3][4]) {
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        float* op = out + ((static_cast<long long>(f) * 3 + c) * hd + dy0 + j) * wd;
        const float4 v = make_float4(inv255[o[c][0]], inv255[o[c][1]], inv255[o[c][2]], inv255[o[c][3]]);
        if (vec_out && g * 4 + 3 < wd) {
          *reinterpret_cast<float4*>(op + g * 4) = v;
        } else {
          const float vv[4] = {v.x, v.y, v.z, v.w};
          for (int q = 0; q < 4; ++q)
            if (g * 4 + q < wd) op[g * 4 + q] = vv[q];
        }
      }
    };
    for (int g = threadIdx.x; g < groups; g += blockDim.x) {
      int o[3][4];
      if (two_to_one && g * 4 + 3 < wd) {
        float ht[12], hb[12];
        pair_sums(sl[0], g, ht);
        pair_sums(sl[1], g, hb);
#pragma unroll
        for (int i = 0; i < 12; ++i) o[i % 3][i / 3] = round_u8(__fadd_rn(__fmul_rn(hb0, ht[i]), __fmul_rn(ha0, hb[i])));
        store_row(g, 0, o);
        if (pr.two_rows) {
          if (pr.shared_row) {
#pragma unroll
            for (int i = 0; i < 12; ++i) ht[i] = hb[i];
          } else {
            pair_sums(sl[2], g, ht);
          }
          pair_sums(sl[3], g, hb);
#pragma unroll
          for (int i = 0; i < 12; ++i)
            o[i % 3][i / 3] = round_u8(__fadd_rn(__fmul_rn(hb1, ht[i]), __fmul_rn(ha1, hb[i])));
          store_row(g, 1, o);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (j == 1 && !pr.two_rows) break;
          const uint8_t* ra = j == 0 ? sl[0] : sl[2];
          const uint8_t* rb = j == 0 ? sl[1] : sl[3];
          const float ay = j == 0 ? pr.s0.a : pr.s1.a;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int dx = g * 4 + q;
            if (dx < wd) {
              const AxisSample sx = axis_sample(dx, ws, scale_x);
#pragma unroll
              for (int c = 0; c < 3; ++c) {
                const int i0 = sx.i0 * 3 + c, i1 = sx.i1 * 3 + c;
                o[c][q] = round_u8(bilinear(u8_to_float(ra[i0]), u8_to_float(ra[i1]), u8_to_float(rb[i0]),
                                            u8_to_float(rb[i1]), sx.a, ay));
              }
            } else {
#pragma unroll
              for (int c = 0; c < 3; ++c) o[c][q] = 0;
            }
          }
          store_row(g, j, o);
        }
      }
    }
    __syncthreads();  // a later item's copies overwrite this buffer
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

static size_t row_smem(int ws) { return 2 * static_cast<size_t>((ws * 3 + 15) & ~15); }

template <bool TO_U8>
static cudaError_t launch_rows(const uint8_t* src, int n, int hs, int ws, long long pitch, void* out, int hd, int wd,
                               bool vec_out, cudaStream_t s) {
  if (n == 0 || hd == 0 || wd == 0) return cudaSuccess;
  const bool vec_in = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (pitch % 16 == 0);
  const size_t smem = row_smem(ws);
  if (smem > 48 * 1024) {
    const cudaError_t e = smem_attr_once<preprocess_row_kernel<TO_U8>>(smem);
    if (e != cudaSuccess) return e;
  }
  int threads = ((wd + 3) / 4 + 31) / 32 * 32;
  if (threads > 256) threads = 256;
  if (threads < 64) threads = 64;
  dim3 grid(hd, n);
  return launch_pdl(preprocess_row_kernel<TO_U8>, grid, dim3(threads), smem, s, src, hs, ws, pitch, out, hd, wd,
                    vec_in ? 1 : 0, vec_out ? 1 : 0);
}

cudaError_t launch_preprocess_fused(const uint8_t* src, int n, int hs, int ws, long long pitch, float* dst, int hd,
                                    int wd, int sms, cudaStream_t s) {
  if (n == 0 || hd == 0 || wd == 0) return cudaSuccess;
  const bool vec_out = (reinterpret_cast<uintptr_t>(dst) % 16 == 0) && (wd % 4 == 0);
  const bool vec_in = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (pitch % 16 == 0);
  const bool async_rows = vec_in && (ws * 3) % 16 == 0;
  const size_t smem = 4 * row_smem(ws);  // two buffers of four staged rows
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = smem_attr_once<preprocess_pair_kernel>(smem);
  if (e != cudaSuccess) return e;
  int threads = ((wd + 3) / 4 + 31) / 32 * 32;
  if (threads > 256) threads = 256;
  if (threads < 64) threads = 64;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, preprocess_pair_kernel, threads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const long long items = static_cast<long long>((hd + 1) / 2) * n;
  const long long cap = static_cast<long long>(sms) * per_sm;
  const unsigned grid = static_cast<unsigned>(items < cap ? items : cap);
  return launch_pdl(preprocess_pair_kernel, dim3(grid), dim3(threads), smem, s, src, n, hs, ws, pitch, dst, hd, wd,
                    async_rows ? 1 : 0, vec_in ? 1 : 0, vec_out ? 1 : 0);
}

cudaError_t launch_preprocess_resize(const uint8_t* src, int n, int hs, int ws, long long pitch, uint8_t* out,
                                     int hd, int wd, cudaStream_t s) {
  return launch_rows<true>(src, n, hs, ws, pitch, out, hd, wd, false, s);
}

// Pass 2: u8 -> fp32 / 255 (HWC kept).
__global__ void __launch_bounds__(256) normalize_kernel(const uint8_t* __restrict__ in, long long count,
                                                        float* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < count; i += stride)
    out[i] = __fdiv_rn(static_cast<float>(in[i]), 255.0f);
}

cudaError_t launch_preprocess_normalize(const uint8_t* in, long long count, float* out, cudaStream_t s) {
  if (count == 0) return cudaSuccess;
  long long blocks = (count + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  return launch_pdl(normalize_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, in, count, out);
}

// Pass 3: fp32 HWC [n, h, w, 3] -> fp32 CHW [n, 3, h, w].
__global__ void __launch_bounds__(256) layout_kernel(const float* __restrict__ in, int n, int h, int w,
                                                     float* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
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
  const cudaError_t e = launch_pdl(layout_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, in, n, h, w, out);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The sample coordinates every preprocess kernel uses along one axis of
// source extent S and destination extent D (one thread per destination
// index), for checks of the resize's indexing.
__global__ void __launch_bounds__(256) sample_coords_kernel(int S, int D, int* __restrict__ i0, int* __restrict__ i1,
                                                            float* __restrict__ a) {
  pdl_wait();
  pdl_launch_dependents();
  const float scale = __fdiv_rn(static_cast<float>(S), static_cast<float>(D));
  for (int d = blockIdx.x * blockDim.x + threadIdx.x; d < D; d += gridDim.x * blockDim.x) {
    const AxisSample s = axis_sample(d, S, scale);
    i0[d] = s.i0;
    i1[d] = s.i1;
    a[d] = s.a;
  }
}

cudaError_t launch_sample_coords(int S, int D, int* i0, int* i1, float* a, cudaStream_t s) {
  const int blocks = (D + 255) / 256 < 1024 ? (D + 255) / 256 : 1024;
  return launch_pdl(sample_coords_kernel, dim3(blocks), dim3(256), 0, s, S, D, i0, i1, a);
}

}  // namespace cb
