// Depthwise 3x3 convolution + folded BatchNorm + activation (+ residual), NHWC fp32.
//
// The computation is the one walked through for the Metal kernel on "How I
// sped up convolutions" (steps 1-5: window origin oh*s - pad, taps outside
// the image read as zero, BN and ReLU applied while the sum is still in a
// register, one store), laid out for a memory-bound GB300 kernel:
//
//  * dw_tma_kernel (the fast path): persistent CTAs.  A work item is one
//    image, one 32-channel chunk (128 bytes per pixel), one strip of output
//    rows and one tile of output columns.  A producer thread streams the
//    strip's input rows -- the full padded width of the tile, halo columns
//    included -- into a shared-memory ring with 4-D TMA tile copies; the
//    copy's out-of-range zero fill supplies the padding.  Each consumer
//    thread owns one (output column, 4 channels) pair, reads the three
//    columns of its window from each ring row once, and slides the 3x3
//    window down the strip in registers.
//  * dw_simple_kernel: one thread per (output pixel, 4 channels) or per
//    channel, direct global loads.  Used for views the TMA path cannot
//    describe (unaligned data, channel counts that are not multiples of 4).
#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace cb {

// --------------------------------------------------------------- simple path
template <bool VEC>
__global__ void __launch_bounds__(256) dw_simple_kernel(const DwArgs a) {
  constexpr int V = VEC ? 4 : 1;
  const int CV = a.C / V;
  const long long total = static_cast<long long>(a.N) * a.OH * a.OW * CV;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int cv = static_cast<int>(i % CV);
    const long long pix = i / CV;
    const int ow = static_cast<int>(pix % a.OW);
    const int oh = static_cast<int>((pix / a.OW) % a.OH);
    const int n = static_cast<int>(pix / (static_cast<long long>(a.OW) * a.OH));
    const int c = cv * V;
    float acc[V];
#pragma unroll
    for (int q = 0; q < V; ++q) acc[q] = 0.0f;
    for (int kh = 0; kh < 3; ++kh) {
      const int ih = oh * a.stride - a.pad + kh;
      if (ih < 0 || ih >= a.H) continue;
      for (int kw = 0; kw < 3; ++kw) {
        const int iw = ow * a.stride - a.pad + kw;
        if (iw < 0 || iw >= a.W) continue;
        const float* xp = a.x + n * a.xs_n + ih * a.xs_h + iw * a.xs_w + c;
        const float* wp = a.w + (kh * 3 + kw) * a.C + c;
        if (VEC) {
          const float4 xv = ldg4(xp), wv = ldg4(wp);
          acc[0] = fmaf(xv.x, wv.x, acc[0]);
          acc[V > 1 ? 1 : 0] = fmaf(xv.y, wv.y, acc[V > 1 ? 1 : 0]);
          acc[V > 2 ? 2 : 0] = fmaf(xv.z, wv.z, acc[V > 2 ? 2 : 0]);
          acc[V > 3 ? 3 : 0] = fmaf(xv.w, wv.w, acc[V > 3 ? 3 : 0]);
        } else {
          acc[0] = fmaf(__ldg(xp), __ldg(wp), acc[0]);
        }
      }
    }
    float* yp = a.out.y + n * a.out.ys_n + oh * a.out.ys_h + ow * a.out.ys_w + c;
    const float* rp = a.ep.r ? a.ep.r + n * a.ep.rs_n + oh * a.ep.rs_h + ow * a.ep.rs_w + c : nullptr;
#pragma unroll
    for (int q = 0; q < V; ++q) {
      const float r = a.ep.res_mode ? rp[q] : 0.0f;
      yp[q] = epi_apply(acc[q], __ldg(a.ep.scale + c + q), __ldg(a.ep.bias + c + q), r, a.ep.act, a.ep.res_mode);
    }
  }
}

cudaError_t launch_dw_simple(const DwArgs& a, bool vec4, cudaStream_t s) {
  const long long total = static_cast<long long>(a.N) * a.OH * a.OW * (vec4 ? a.C / 4 : a.C);
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  if (blocks > (1 << 20)) blocks = 1 << 20;
  if (vec4)
    dw_simple_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  else
    dw_simple_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ TMA path
struct DwTmaParams {
  DwArgs a;
  int rows_per_item, num_items, box_w, stages;
  int chunks, strips, wtiles, tile_w;
  int* err;
  uint64_t timeout_ns;
};

struct DwItem {
  int n, c0, oh0, oh1, ow0, ow1;
};

// Work items are numbered with the channel chunk fastest, so CTAs running at
// the same time read the same input rows (whole 1536-byte pixels of DRAM
// pages) rather than one 128-byte slice of many pixels.
__device__ __forceinline__ DwItem dw_decode(const DwTmaParams& p, int item) {
  DwItem it;
  const int ch = item % p.chunks;
  int rest = item / p.chunks;
  const int wt = rest % p.wtiles;
  rest /= p.wtiles;
  const int st = rest % p.strips;
  it.n = rest / p.strips;
  it.c0 = ch * 32;
  it.oh0 = st * p.rows_per_item;
  it.oh1 = min(it.oh0 + p.rows_per_item, p.a.OH);
  it.ow0 = wt * p.tile_w;
  it.ow1 = min(it.ow0 + p.tile_w, p.a.OW);
  return it;
}

template <int S>
__global__ void __launch_bounds__(512, 1) dw_tma_kernel(const __grid_constant__ CUtensorMap xmap,
                                                        const DwTmaParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int stage_bytes = p.box_w * 128;
  uint8_t* ring = smem_raw;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + p.stages * stage_bytes);
  uint64_t* empty = full + p.stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + p.stages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int consumer_warps = (blockDim.x >> 5) - 1;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], consumer_warps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const Watchdog wd{p.err, abort_flag, p.timeout_ns};
  const DwArgs& a = p.a;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&xmap);
      int slot = 0;
      uint32_t phase = 0, issued = 0, last_parity = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < p.num_items; item += gridDim.x) {
        const DwItem it = dw_decode(p, item);
        const int nrows = (it.oh1 - it.oh0 - 1) * S + 3;
        const int ih0 = it.oh0 * S - a.pad;
        const int iw0 = it.ow0 * S - a.pad;
        for (int j = 0; j < nrows; ++j) {
          if (!mbar_wait(&empty[slot], phase ^ 1u, wd)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(stage_bytes));
          tma_load_4d(ring + slot * stage_bytes, &xmap, &full[slot], it.c0, iw0, ih0 + j, it.n);
          issued |= 1u << slot;
          last_parity = (last_parity & ~(1u << slot)) | (phase << slot);
          if (++slot == p.stages) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      // Let every copy this thread issued land before the CTA can exit.
      for (int s = 0; s < p.stages; ++s)
        if (issued & (1u << s)) mbar_wait_drain(&full[s], (last_parity >> s) & 1u, 20000000ull);
    }
  } else {
    // ---------------------------------------------------------- consumers
    const int t = threadIdx.x - 32;
    const int owl = t >> 3, c4 = t & 7;
    int slot = 0;
    uint32_t phase = 0;
    bool ok = true;

    auto fetch = [&](float4(&dst)[3], bool read) {
      if (!ok) return;
      bool got = mbar_wait(&full[slot], phase, wd);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        ok = false;
        return;
      }
      if (read) {
        const float* row = reinterpret_cast<const float*>(ring + slot * stage_bytes) + c4 * 4;
#pragma unroll
        for (int kw = 0; kw < 3; ++kw) dst[kw] = *reinterpret_cast<const float4*>(row + (owl * S + kw) * 32);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (++slot == p.stages) {
        slot = 0;
        phase ^= 1u;
      }
    };

    for (int item = blockIdx.x; item < p.num_items; item += gridDim.x) {
      const DwItem it = dw_decode(p, item);
      const int ow = it.ow0 + owl;
      const int c = it.c0 + c4 * 4;
      const bool in_tile = ow < it.ow1;
      const bool active = in_tile && c < a.C;
      float4 wv[9];
      float4 sc = make_float4(0.f, 0.f, 0.f, 0.f), bi = sc;
      if (active) {
#pragma unroll
        for (int k = 0; k < 9; ++k) wv[k] = ldg4(a.w + k * a.C + c);
        sc = ldg4(a.ep.scale + c);
        bi = ldg4(a.ep.bias + c);
      } else {
#pragma unroll
        for (int k = 0; k < 9; ++k) wv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float4 ra[3], rb[3], rc[3];
      fetch(ra, in_tile);
      fetch(rb, in_tile);
      for (int oh = it.oh0; oh < it.oh1; ++oh) {
        fetch(rc, in_tile);
        if (ok && active) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int kw = 0; kw < 3; ++kw) {
            fma4(acc, ra[kw], wv[kw]);
            fma4(acc, rb[kw], wv[3 + kw]);
            fma4(acc, rc[kw], wv[6 + kw]);
          }
          float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
          if (a.ep.res_mode)
            r = *reinterpret_cast<const float4*>(a.ep.r + it.n * a.ep.rs_n + oh * a.ep.rs_h + ow * a.ep.rs_w + c);
          const float4 o = epi_apply4(acc, sc, bi, r, a.ep.act, a.ep.res_mode);
          *reinterpret_cast<float4*>(a.out.y + it.n * a.out.ys_n + oh * a.out.ys_h + ow * a.out.ys_w + c) = o;
        }
        if (S == 1) {
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            ra[k] = rb[k];
            rb[k] = rc[k];
          }
        } else if (oh + 1 < it.oh1) {
#pragma unroll
          for (int k = 0; k < 3; ++k) ra[k] = rc[k];
          fetch(rb, in_tile);
        }
      }
    }
  }
  __syncthreads();
}

cudaError_t launch_dw_tma(const CUtensorMap& xmap, const DwArgs& a, const DwTmaPlan& plan, int* err,
                          uint64_t timeout_ns, cudaStream_t s) {
  DwTmaParams p;
  p.a = a;
  p.rows_per_item = plan.rows_per_item;
  p.num_items = plan.num_items;
  p.box_w = plan.box_w;
  p.stages = plan.stages;
  p.chunks = (a.C + 31) / 32;
  p.strips = (a.OH + plan.rows_per_item - 1) / plan.rows_per_item;
  p.tile_w = (plan.box_w - 3) / a.stride + 1;
  p.wtiles = (a.OW + p.tile_w - 1) / p.tile_w;
  p.err = err;
  p.timeout_ns = timeout_ns;
  const int threads = 32 * (1 + plan.consumer_warps);
  if (a.stride == 1) {
    cudaFuncSetAttribute(dw_tma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(plan.smem_bytes));
    dw_tma_kernel<1><<<plan.grid, threads, plan.smem_bytes, s>>>(xmap, p);
  } else {
    cudaFuncSetAttribute(dw_tma_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(plan.smem_bytes));
    dw_tma_kernel<2><<<plan.grid, threads, plan.smem_bytes, s>>>(xmap, p);
  }
  return cudaGetLastError();
}

// Occupancy query used by the planner (registers decide how many CTAs fit).
int dw_tma_blocks_per_sm(int stride, int threads, size_t smem) {
  int n = 0;
  if (stride == 1) {
    cudaFuncSetAttribute(dw_tma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dw_tma_kernel<1>, threads, smem);
  } else {
    cudaFuncSetAttribute(dw_tma_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dw_tma_kernel<2>, threads, smem);
  }
  return n;
}

}  // namespace cb
