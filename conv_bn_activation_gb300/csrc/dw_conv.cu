// Depthwise 3x3 convolution + folded BatchNorm + activation (+ residual), NHWC fp32.
//
// The computation is the one walked through for the Metal kernel on "How I
// sped up convolutions" (steps 1-5: window origin oh*s - pad, taps outside
// the image read as zero, BN and ReLU applied while the sum is still in a
// register, one store), laid out for a memory-bound GB300 kernel:
//
//  * dw_tma_kernel (the fast path): persistent CTAs.  A work item is one
//    image, one 32-channel chunk (128 bytes per pixel), one strip of output
//    rows and one tile of output columns.  Four producer lanes (taking rows
//    in turn: one thread's copies complete one after another) stream the
//    strip's input rows -- the full padded width of the tile, halo columns
//    included -- into a shared-memory ring with 4-D TMA tile copies; the
//    copy's out-of-range zero fill supplies the padding.  Each consumer
//    thread owns one (output column, 4 channels) pair, reads the three
//    columns of its window from each ring row once, and slides the 3x3
//    window down the strip in registers.
//    With bf16 storage the same kernel moves 128-byte pixel chunks of 64
//    channels: values are widened to fp32 as they leave shared memory and
//    the fp32 result is rounded to bf16 (nearest even) at the store.
//  * dw_simple_kernel: one thread per (output pixel, 4 channels) or per
//    channel, direct global loads.  Used for views the TMA path cannot
//    describe (unaligned data, channel counts that are not multiples of 4).
#include "epilogue.cuh"
#include "launch_util.h"
#include "internal.h"
#include "ptx.cuh"

namespace cb {

// --------------------------------------------------------------- simple path
template <bool VEC>
__global__ void __launch_bounds__(256) dw_simple_kernel(const DwArgs a) {
  pdl_wait();
  pdl_launch_dependents();
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
    return launch_pdl(dw_simple_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, a);
  else
    return launch_pdl(dw_simple_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, a);
}

// ------------------------------------------------------------------ TMA path
struct DwTmaParams {
  DwArgs a;
  int rows_per_item, num_items, box_w, stages;
  int ch;      // channels per chunk: one 128-byte pixel row (32 fp32 or 64 bf16)
  int w_smem;  // bf16 at stride 1: the taps [9][C] staged in shared memory after the barriers
  int chunks, strips, wtiles, tile_w;
  int* err;
  uint64_t timeout_ns;
  int debug_skip_row;  // fault injection: CTA 0 withholds its first row copy (tests of the bounded waits)
};

struct DwItem {
  int n, c0, oh0, oh1, ow0, ow1;
};

// Work items are numbered with the channel chunk fastest, so CTAs running at
// the same time read the same input rows (whole pixels, i.e. whole DRAM
// pages) rather than one 128-byte slice of many pixels.
__device__ __forceinline__ DwItem dw_decode(const DwTmaParams& p, int item) {
  DwItem it;
  const int ch = item % p.chunks;
  int rest = item / p.chunks;
  const int wt = rest % p.wtiles;
  rest /= p.wtiles;
  const int st = rest % p.strips;
  it.n = rest / p.strips;
  it.c0 = ch * p.ch;
  it.oh0 = st * p.rows_per_item;
  it.oh1 = min(it.oh0 + p.rows_per_item, p.a.OH);
  it.ow0 = wt * p.tile_w;
  it.ow1 = min(it.ow0 + p.tile_w, p.a.OW);
  return it;
}

constexpr int kDwProducerLanes = 4;

// acc += a * b on four lanes as two packed fp32 FMAs (each lane rounded as
// one fmaf: the same bits as fma4, half the instructions).
__device__ __forceinline__ void fma4_packed(float4& acc, float4 a, float4 b) {
  const float2 lo = __ffma2_rn(make_float2(a.x, a.y), make_float2(b.x, b.y), make_float2(acc.x, acc.y));
  const float2 hi = __ffma2_rn(make_float2(a.z, a.w), make_float2(b.z, b.w), make_float2(acc.z, acc.w));
  acc = make_float4(lo.x, lo.y, hi.x, hi.y);
}

template <int ACT, int RES>
__device__ __forceinline__ float epi_c(float acc, float sc, float bi, float r) {
  float z = fmaf(acc, sc, bi);
  if (RES == 1) z += r;
  if (ACT == 1) z = fmaxf(z, 0.0f);
  if (ACT == 2) z = silu(z);
  if (RES == 2) z += r;
  return z;
}

// Output columns per consumer thread: 4 for bf16 at stride 1, else 2.  bf16
// carries twice the outputs per byte, so the per-row costs (barrier wait,
// loads, widening) must be shared by more of them.
template <typename T, int S>
__host__ __device__ constexpr int dw_cols() { return sizeof(T) == 2 && S == 1 ? 4 : 2; }

// Each consumer thread owns COLS adjacent output columns x 4 channels; its
// window needs NC = (COLS - 1) S + 3 input columns per row.  T: the storage
// type of x, y and the residual (float or bf16).
template <typename T, int S, int ACT, int RES>
__global__ void __launch_bounds__(512, 1) dw_tma_kernel(const __grid_constant__ CUtensorMap xmap,
                                                        const DwTmaParams p) {
  constexpr int COLS = dw_cols<T, S>();
  constexpr int NC = (COLS - 1) * S + 3;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // One ring slot: a row copy of box_w pixels of one chunk, 128 bytes each
  // (32 fp32 or 64 bf16 channels: an SM completes its copies one after
  // another, so a bf16 chunk is as wide as an fp32 one in bytes, not in
  // channels, and the layer takes half the copies).
  constexpr int CH = 128 / static_cast<int>(sizeof(T));  // channels per chunk
  constexpr bool kPacked = sizeof(T) == 2;                 // packed FMAs (bf16 storage)
  constexpr int TPP = CH / 4;                              // threads per column group
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
  pdl_launch_dependents();
  pdl_wait();
  const Watchdog wd{p.err, abort_flag, p.timeout_ns};
  const DwArgs& a = p.a;
  // Four-column threads read each tap once per input row for all four
  // columns: the taps come from shared memory (staged once per CTA) or, for
  // a layer too wide to stage, from L1.
  float* sw = reinterpret_cast<float*>(reinterpret_cast<uintptr_t>(abort_flag) + 16);  // 16-byte aligned
  const float* wsrc = a.w;
  if constexpr (COLS == 4) {
    if (p.w_smem) {
      for (int i = threadIdx.x; i < 9 * a.C / 4; i += blockDim.x)
        reinterpret_cast<float4*>(sw)[i] = ldg4(a.w + 4 * i);
      __syncthreads();
      wsrc = sw;
    }
  }

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    // Copies issued by one thread complete one after another, so
    // kDwProducerLanes lanes share the rows, each owning the ring slots s with
    // s % kDwProducerLanes == lane (one owner per slot keeps each lane's
    // barrier phases its own).
    if (lane < kDwProducerLanes) {
      if (lane == 0) tma_prefetch_desc(&xmap);
      int slot = 0;
      uint32_t phase = 0, issued = 0, last_parity = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < p.num_items; item += gridDim.x) {
        const DwItem it = dw_decode(p, item);
        const int nrows = (it.oh1 - it.oh0 - 1) * S + 3;
        const int ih0 = it.oh0 * S - a.pad;
        const int iw0 = it.ow0 * S - a.pad;
        for (int r = 0; r < nrows; ++r) {
          // fault injection: no copy and no arrive for CTA 0's first row, so
          // that row's barrier phase never completes and its waits run out
          const bool skip = p.debug_skip_row && blockIdx.x == 0 && item == 0 && r == 0;
          if (slot % kDwProducerLanes == lane && !skip) {
            if (!mbar_wait(&empty[slot], phase ^ 1u, wd)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(stage_bytes));
            tma_load_4d(ring + slot * stage_bytes, &xmap, &full[slot], it.c0, iw0, ih0 + r, it.n);
            issued |= 1u << slot;
            last_parity = (last_parity & ~(1u << slot)) | (phase << slot);
          }
          if (++slot == p.stages) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      // Let every copy this lane issued land before the CTA can exit.
      for (int s = 0; s < p.stages; ++s)
        if (issued & (1u << s)) mbar_wait_drain(&full[s], (last_parity >> s) & 1u, 20000000ull);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int t = threadIdx.x - 32;
  const int grp = t / TPP, c4 = t % TPP;
  int slot = 0;
  uint32_t phase = 0;
  bool ok = true;

  // Wait for the next ring row, copy this thread's NC window columns into
  // registers, release the slot.
  auto fetch = [&](float4(&dst)[NC], bool read) {
    if (!ok) return;
    bool got = mbar_wait(&full[slot], phase, wd);
    got = __all_sync(0xffffffffu, got);
    if (!got) {
      ok = false;
      return;
    }
    if (read) {
      const T* row = reinterpret_cast<const T*>(ring + slot * stage_bytes) + (COLS * grp * S) * CH + c4 * 4;
#pragma unroll
      for (int k = 0; k < NC; ++k) dst[k] = load4(row + k * CH);
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
    const int ow = it.ow0 + COLS * grp;
    const int c = it.c0 + c4 * 4;
    const bool in_tile = ow < it.ow1;            // the box covers every column of every group
    const bool active = in_tile && c < a.C;
    const bool second = active && ow + 1 < it.ow1;
    float4 wv[COLS == 2 ? 9 : 1];
    float4 sc = make_float4(0.f, 0.f, 0.f, 0.f), bi = sc;
    if (active) {
      if constexpr (COLS == 2) {
#pragma unroll
        for (int k = 0; k < 9; ++k) wv[k] = ldg4(a.w + k * a.C + c);
      }
      sc = ldg4(a.ep.scale + c);
      bi = ldg4(a.ep.bias + c);
    } else if constexpr (COLS == 2) {
#pragma unroll
      for (int k = 0; k < 9; ++k) wv[k] = sc;
    }
    T* yp = reinterpret_cast<T*>(a.out.y) + it.n * a.out.ys_n + it.oh0 * a.out.ys_h + ow * a.out.ys_w + c;
    const T* rp = RES ? reinterpret_cast<const T*>(a.ep.r) + it.n * a.ep.rs_n + it.oh0 * a.ep.rs_h + ow * a.ep.rs_w + c
                      : nullptr;

    // One output row from the window (top, mid, bottom); advances yp / rp.
    auto compute = [&](const float4(&top)[NC], const float4(&mid)[NC], const float4(&bot)[NC]) {
      if constexpr (COLS == 4) {
        if (ok && active) {
          // the same sum order as the two-column path: tap columns kw, and
          // within each the top, middle and bottom rows
          float4 acc[COLS];
#pragma unroll
          for (int j = 0; j < COLS; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int kw = 0; kw < 3; ++kw) {
            const float4 wt = *reinterpret_cast<const float4*>(wsrc + kw * a.C + c);
            const float4 wm = *reinterpret_cast<const float4*>(wsrc + (3 + kw) * a.C + c);
            const float4 wb = *reinterpret_cast<const float4*>(wsrc + (6 + kw) * a.C + c);
#pragma unroll
            for (int j = 0; j < COLS; ++j) {
              fma4_packed(acc[j], top[j * S + kw], wt);
              fma4_packed(acc[j], mid[j * S + kw], wm);
              fma4_packed(acc[j], bot[j * S + kw], wb);
            }
          }
#pragma unroll
          for (int j = 0; j < COLS; ++j) {
            if (ow + j < it.ow1) {
              float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
              if (RES) r = load4(rp + j * a.ep.rs_w);
              float4 o;
              o.x = epi_c<ACT, RES>(acc[j].x, sc.x, bi.x, r.x);
              o.y = epi_c<ACT, RES>(acc[j].y, sc.y, bi.y, r.y);
              o.z = epi_c<ACT, RES>(acc[j].z, sc.z, bi.z, r.z);
              o.w = epi_c<ACT, RES>(acc[j].w, sc.w, bi.w, r.w);
              store4(yp + j * a.out.ys_w, o);
            }
          }
        }
      } else if (ok && active) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int kw = 0; kw < 3; ++kw) {
            if constexpr (kPacked) {
              // bf16 storage moves half the bytes per output: the arithmetic
              // must keep up, so the FMAs go out packed
              fma4_packed(acc, top[j * S + kw], wv[kw]);
              fma4_packed(acc, mid[j * S + kw], wv[3 + kw]);
              fma4_packed(acc, bot[j * S + kw], wv[6 + kw]);
            } else {
              fma4(acc, top[j * S + kw], wv[kw]);
              fma4(acc, mid[j * S + kw], wv[3 + kw]);
              fma4(acc, bot[j * S + kw], wv[6 + kw]);
            }
          }
          if (j == 0 || second) {
            float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
            if (RES) r = load4(rp + j * a.ep.rs_w);
            float4 o;
            o.x = epi_c<ACT, RES>(acc.x, sc.x, bi.x, r.x);
            o.y = epi_c<ACT, RES>(acc.y, sc.y, bi.y, r.y);
            o.z = epi_c<ACT, RES>(acc.z, sc.z, bi.z, r.z);
            o.w = epi_c<ACT, RES>(acc.w, sc.w, bi.w, r.w);
            store4(yp + j * a.out.ys_w, o);
          }
        }
      }
      yp += a.out.ys_h;
      if (RES) rp += a.ep.rs_h;
    };

    float4 r0[NC], r1[NC], r2[NC];
    fetch(r0, in_tile);
    fetch(r1, in_tile);
    fetch(r2, in_tile);
    int oh = it.oh0;
    if (S == 1) {
      // window rows rotate r0,r1,r2 -> r1,r2,r0 -> r2,r0,r1: one new row per output row
      for (;;) {
        compute(r0, r1, r2);
        if (++oh == it.oh1) break;
        fetch(r0, in_tile);
        compute(r1, r2, r0);
        if (++oh == it.oh1) break;
        fetch(r1, in_tile);
        compute(r2, r0, r1);
        if (++oh == it.oh1) break;
        fetch(r2, in_tile);
      }
    } else {
      // stride 2: the bottom row is the next window's top; two new rows per output row
      for (;;) {
        compute(r0, r1, r2);
        if (++oh == it.oh1) break;
        fetch(r0, in_tile);
        fetch(r1, in_tile);
        compute(r2, r0, r1);
        if (++oh == it.oh1) break;
        fetch(r2, in_tile);
        fetch(r0, in_tile);
        compute(r1, r2, r0);
        if (++oh == it.oh1) break;
        fetch(r1, in_tile);
        fetch(r2, in_tile);
      }
    }
  }
}

template <typename T, int S, int ACT, int RES>
static void dw_tma_launch(const CUtensorMap& xmap, const DwTmaParams& p, int grid, int threads, size_t smem,
                          cudaStream_t s) {
  if (smem_attr_once<dw_tma_kernel<T, S, ACT, RES>>(smem) != cudaSuccess) return;
  launch_pdl(dw_tma_kernel<T, S, ACT, RES>, dim3(grid), dim3(threads), smem, s, xmap, p);
}

template <typename T, int S>
static void dw_tma_dispatch(const CUtensorMap& xmap, const DwTmaParams& p, int grid, int threads, size_t smem,
                            cudaStream_t s) {
  const int act = p.a.ep.act, res = p.a.ep.res_mode;
#define CB_DW_CASE(A, R) \
  if (act == A && res == R) return dw_tma_launch<T, S, A, R>(xmap, p, grid, threads, smem, s);
  CB_DW_CASE(0, 0) CB_DW_CASE(1, 0) CB_DW_CASE(2, 0)
  CB_DW_CASE(0, 1) CB_DW_CASE(1, 1) CB_DW_CASE(2, 1)
  CB_DW_CASE(0, 2) CB_DW_CASE(1, 2) CB_DW_CASE(2, 2)
#undef CB_DW_CASE
}

cudaError_t launch_dw_tma(const CUtensorMap& xmap, const DwArgs& a, const DwTmaPlan& plan, int* err,
                          uint64_t timeout_ns, int debug_skip_row, cudaStream_t s) {
  DwTmaParams p;
  p.a = a;
  p.rows_per_item = plan.rows_per_item;
  p.num_items = plan.num_items;
  p.box_w = plan.box_w;
  p.stages = plan.stages;
  p.ch = a.bf16 ? 64 : 32;
  p.w_smem = plan.w_smem;
  p.chunks = (a.C + p.ch - 1) / p.ch;
  p.strips = (a.OH + plan.rows_per_item - 1) / plan.rows_per_item;
  p.tile_w = plan.tile_w;
  p.wtiles = (a.OW + p.tile_w - 1) / p.tile_w;
  p.err = err;
  p.timeout_ns = timeout_ns;
  p.debug_skip_row = debug_skip_row;
  const int threads = 32 * (1 + plan.consumer_warps);
  if (a.bf16) {
    if (a.stride == 1)
      dw_tma_dispatch<__nv_bfloat16, 1>(xmap, p, plan.grid, threads, plan.smem_bytes, s);
    else
      dw_tma_dispatch<__nv_bfloat16, 2>(xmap, p, plan.grid, threads, plan.smem_bytes, s);
  } else if (a.stride == 1) {
    dw_tma_dispatch<float, 1>(xmap, p, plan.grid, threads, plan.smem_bytes, s);
  } else {
    dw_tma_dispatch<float, 2>(xmap, p, plan.grid, threads, plan.smem_bytes, s);
  }
  return cudaGetLastError();
}

template <typename T, int S>
static int dw_tma_occupancy(int threads, size_t smem) {
  int n = 0;
  smem_attr_once<dw_tma_kernel<T, S, 1, 0>>(smem);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dw_tma_kernel<T, S, 1, 0>, threads, smem);
  return n;
}

// Occupancy query used by the planner (registers decide how many CTAs fit).
// Cached per (stride, warps, shared-memory size in KB): occupancy is a
// function of the kernel and these alone.
int dw_tma_blocks_per_sm(int stride, int threads, size_t smem, bool bf16) {
  static std::atomic<int> cache[4][33][229];
  const int si = (stride == 1 ? 0 : 1) + (bf16 ? 2 : 0), wi = threads / 32, ki = static_cast<int>(smem / 1024);
  const bool cacheable = threads % 32 == 0 && wi <= 32 && smem % 1024 == 0 && ki <= 228;
  if (cacheable) {
    const int v = cache[si][wi][ki].load(std::memory_order_relaxed);
    if (v > 0) return v - 1;
  }
  int n = 0;
  if (bf16 && stride == 1) n = dw_tma_occupancy<__nv_bfloat16, 1>(threads, smem);
  else if (bf16) n = dw_tma_occupancy<__nv_bfloat16, 2>(threads, smem);
  else if (stride == 1) n = dw_tma_occupancy<float, 1>(threads, smem);
  else n = dw_tma_occupancy<float, 2>(threads, smem);
  if (cacheable) cache[si][wi][ki].store(n + 1, std::memory_order_relaxed);
  return n;
}

}  // namespace cb
