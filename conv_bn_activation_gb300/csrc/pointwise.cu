// 1x1 convolution + folded BN + activation (+ residual) for layers with at
// most 32 input and output channels, on the fp32 CUDA cores ("YOLO26N
// Inference Optimisation", the 1x1 C -> C/2 and C -> C convs of the stage
// blocks; "How I sped up convolutions", the pointwise conv).
//
// At these widths the layer is HBM-bound (16 -> 16 moves 128 bytes per
// pixel for 256 FMAs), and a tcgen05 MMA, whose issue costs at least ~111
// cycles for a 128 x N x 8 step, does less useful work per cycle than the
// CUDA cores.  So this kernel streams pixels (and their residual rows)
// through a shared-memory ring of 16 KB tiles (cp.async, every thread
// copying different bytes, several tiles in flight per CTA so that enough
// bytes are in flight to cover HBM latency); then each thread computes
// 4 pixels x 4 output channels from shared memory (register blocking: 64
// FMAs per 8 shared loads) and stores each pixel's four channels as one
// 16-byte store, so a warp's stores are whole pixel segments.  The residual
// is read straight into registers, issued before the FMAs that it then
// overlaps: staging it beside the input doubled the ring and held the
// residual layers to one CTA per SM.  The weights sit in shared memory as
// [ci][co/4] float4s.
#include "epilogue.cuh"
#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"

namespace cb {

namespace {

__device__ __forceinline__ float comp(const float4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Four output channels of one pixel; the activation is picked once per pixel
// (a uniform branch) so the four exponentials overlap.
__device__ __forceinline__ float4 pw_epilogue(float4 acc, float4 sc, float4 bi, float4 r, int act, int res_mode) {
  float z[4] = {fmaf(acc.x, sc.x, bi.x), fmaf(acc.y, sc.y, bi.y), fmaf(acc.z, sc.z, bi.z), fmaf(acc.w, sc.w, bi.w)};
  const float rr[4] = {r.x, r.y, r.z, r.w};
  if (res_mode == 1)
#pragma unroll
    for (int i = 0; i < 4; ++i) z[i] += rr[i];
  if (act == 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) z[i] = fmaxf(z[i], 0.0f);
  } else if (act == 2) {
#pragma unroll
    for (int i = 0; i < 4; ++i) z[i] = silu(z[i]);
  }
  if (res_mode == 2)
#pragma unroll
    for (int i = 0; i < 4; ++i) z[i] += rr[i];
  return make_float4(z[0], z[1], z[2], z[3]);
}

// 16-byte asynchronous global -> shared copy; src_bytes == 0 writes zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

constexpr int kPwThreads = 256;
constexpr int kPwU = 4;       // pixels per thread at most (register blocking)
constexpr int kPwStages = 3;  // tiles in flight per CTA (ring depth)

template <int CI, int CO, typename T>
struct PwShape {
  static constexpr int G = CO / 4;                                // channel groups of 4 outputs
  static constexpr int kEpp = 16 / static_cast<int>(sizeof(T));   // elements per 16-byte piece
  static constexpr int kVec = CI / kEpp;                          // 16-byte input pieces per pixel
  static constexpr int kPitch = kVec >= 4 ? kVec + 1 : kVec;      // staged input row, 16-byte units (padded)
  // pixels per tile: 16 KB of fp32 input (8 KB of bf16), or up to twice that
  // when narrow outputs would otherwise leave threads without 4 pixels' work
  // and the three-tile ring stays within 112 KB (two CTAs per SM; measured:
  // 32 -> 16 at 160x160 42.4 -> 37.5 us, while 16 -> 8, whose ring would
  // grow to 120 KB and one CTA per SM, went from 57.5 to 71.2 us)
  static constexpr int kTile0 = 4096 / CI;
  static constexpr int kTileBig = 1024 / G < 2 * kTile0 ? 1024 / G : 2 * kTile0;
  static constexpr int kTile =
      kTile0 < 1024 / G && kPwStages * kTileBig * kPitch * 16 <= 112 * 1024 ? kTileBig : kTile0;
  // pixels per thread: 4, fewer when a tile has too few (pixel group,
  // channel group) items to give every thread one (narrow outputs)
  static constexpr int kU = kTile * G / kPwThreads >= kPwU ? kPwU : (kTile * G / kPwThreads >= 2 ? 2 : 1);
  static constexpr int kGroups = kTile / kU;                      // pixel groups per tile
  static constexpr int kItems = kGroups * G;                      // (pixel group, channel group) items
  static constexpr int kXFloat4 = kTile * kPitch;
  // bf16 storage stages the residual in the ring too (16-byte copies): read
  // straight into registers, its 8-byte loads kept too few bytes in flight
  // to cover HBM latency (measured 120.5 us against 111 in fp32 for
  // 16 -> 16 + residual); a bf16 tile and its residual take as much shared
  // memory as an fp32 tile alone.
  static constexpr int kRVec = CO / kEpp;                          // 16-byte residual pieces per pixel
  static constexpr int kRPitch = kRVec >= 4 ? kRVec + 1 : kRVec;
  static constexpr bool kRStaged = sizeof(T) == 2 && kRVec >= 1 && (kTile * kRVec) % kPwThreads == 0;
  static constexpr int kRFloat4 = kRStaged ? kTile * kRPitch : 0;
  static size_t smem_bytes(bool res) {
    return 16 * (static_cast<size_t>(CI) * G + 2 * G +
                 static_cast<size_t>(kPwStages) * (kXFloat4 + (res ? kRFloat4 : 0)));
  }
};

// A ring of kPwStages tiles per CTA: a tile is kTile pixels whose CI inputs
// are 16 or 32 KB (half that in bf16), copied
// with 16-byte cp.async by all threads (different bytes per thread).  The
// staged rows of 64 bytes or more are padded by 16 bytes so that the
// pixel-strided reads below hit distinct bank groups.  Each thread computes
// 4 pixels x 4 output channels: per 4 input channels it reads 4 pixel
// float4s and 4 weight float4s and does 64 FMAs.  T: the storage type of x,
// y and the residual (float, or bf16 widened to fp32 as it leaves shared
// memory and rounded to nearest even at the store).
template <int CI, int CO, bool RES, typename T>
__global__ void __launch_bounds__(kPwThreads) pw_small_kernel(const DirectArgs a, int flat) {
  static_assert(CI % 4 == 0 && CO % 4 == 0 && CI <= 32 && CO <= 32, "channel counts");
  using Sh = PwShape<CI, CO, T>;
  constexpr int G = Sh::G, kVec = Sh::kVec, kPitch = Sh::kPitch, kEpp = Sh::kEpp;
  constexpr int kTile = Sh::kTile, kGroups = Sh::kGroups, kItems = Sh::kItems, kU = Sh::kU;
  constexpr int kPieces = kTile * kVec / kPwThreads;  // 16-byte copies per thread per tile
  static_assert(kVec >= 1 && kPieces * kPwThreads == kTile * kVec && kPwThreads % G == 0, "tile shape");
  constexpr bool kRStaged = RES && Sh::kRStaged;     // the residual staged beside the input (bf16)
  constexpr int kRVec = Sh::kRVec, kRPitch = Sh::kRPitch;
  constexpr int kRPieces = kRStaged ? kTile * kRVec / kPwThreads : 0;
  static_assert(!kRStaged || (kRVec >= 1 && kRPieces * kPwThreads == kTile * kRVec), "residual tile shape");
  extern __shared__ float4 pw_smem[];
  constexpr bool res = RES;  // a residual (its placement is a.ep.res_mode)
  float4* ws = pw_smem;             // [CI][G]
  float4* ssc = ws + CI * G;        // [G]
  float4* sbi = ssc + G;            // [G]
  float4* ring = sbi + G;           // kPwStages x tile
  constexpr int stage_f4 = Sh::kXFloat4 + (kRStaged ? Sh::kRFloat4 : 0);  // input tile, then its residual
  pdl_wait();
  pdl_launch_dependents();
  for (int i = threadIdx.x; i < CI * G; i += kPwThreads) {
    const int ci = i / G, g = i - (i / G) * G;
    const float* wp = a.w + (4 * g) * CI + ci;  // [co][ci]
    ws[i] = make_float4(__ldg(wp), __ldg(wp + CI), __ldg(wp + 2 * CI), __ldg(wp + 3 * CI));
  }
  for (int g = threadIdx.x; g < G; g += kPwThreads) {
    ssc[g] = ldg4(a.ep.scale + 4 * g);
    sbi[g] = ldg4(a.ep.bias + 4 * g);
  }

  const long long HW = static_cast<long long>(a.H) * a.W;
  const long long M = a.N * HW;
  const long long num_tiles = (M + kTile - 1) / kTile;
  auto pixel_off = [&](long long p, long long sn, long long sh, long long sw) -> long long {
    if (flat) return p * sw;
    const long long n = p / HW;
    const long long rem = p - n * HW;
    const long long h = rem / a.W;
    return n * sn + h * sh + (rem - h * a.W) * sw;
  };
  auto stage = [&](long long tile, int slot) {
    float4* xs = ring + slot * stage_f4;
#pragma unroll
    for (int k = 0; k < kPieces; ++k) {
      const int piece = threadIdx.x + k * kPwThreads;
      const int lp = piece / kVec, lj = piece - (piece / kVec) * kVec;
      const long long p = tile * kTile + lp;
      const bool in = p < M;
      const T* x = reinterpret_cast<const T*>(a.x);
      const T* src = in ? x + pixel_off(p, a.xs_n, a.xs_h, a.xs_w) + kEpp * lj : x;
      cp_async16(&xs[lp * kPitch + lj], src, in ? 16 : 0);
    }
    if constexpr (kRStaged) {
      float4* rs = xs + Sh::kXFloat4;
#pragma unroll
      for (int k = 0; k < kRPieces; ++k) {
        const int piece = threadIdx.x + k * kPwThreads;
        const int lp = piece / kRVec, lj = piece - (piece / kRVec) * kRVec;
        const long long p = tile * kTile + lp;
        const bool in = p < M;
        const T* r = reinterpret_cast<const T*>(a.ep.r);
        const T* src = in ? r + pixel_off(p, a.ep.rs_n, a.ep.rs_h, a.ep.rs_w) + kEpp * lj : r;
        cp_async16(&rs[lp * kRPitch + lj], src, in ? 16 : 0);
      }
    }
  };

  // prologue: the first kPwStages - 1 tiles of this CTA in flight
  long long tile = blockIdx.x;
#pragma unroll
  for (int k = 0; k < kPwStages - 1; ++k) {
    const long long t = tile + static_cast<long long>(k) * gridDim.x;
    if (t < num_tiles) stage(t, k);
    cp_async_commit();
  }
  __syncthreads();  // weights and constants visible
  for (int it = 0; tile < num_tiles; tile += gridDim.x, ++it) {
    const int slot = it % kPwStages;
    const long long ahead = tile + static_cast<long long>(kPwStages - 1) * gridDim.x;
    if (ahead < num_tiles) stage(ahead, (it + kPwStages - 1) % kPwStages);
    cp_async_commit();
    asm volatile("cp.async.wait_group %0;" ::"n"(kPwStages - 1) : "memory");  // this tile has landed
    __syncthreads();
    const float4* xs = ring + slot * stage_f4;
    // one item per thread at a time (bf16 tiles hold two per thread; their
    // loads hoisted together would double the live registers)
#pragma unroll 1
    for (int item = threadIdx.x; item < kItems; item += kPwThreads) {
      const int pg = item / G, g = item - (item / G) * G;  // pixels pg + u * kGroups
      // the residual's four pixels, in flight during the FMAs (a plain load:
      // the residual may be y itself, each element read before it is written)
      float4 rv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const long long p = tile * kTile + pg + u * kGroups;
        if constexpr (kRStaged) {
          rv[u] = load4(reinterpret_cast<const T*>(xs + Sh::kXFloat4 + (pg + u * kGroups) * kRPitch) + 4 * g);
        } else {
          rv[u] = (res && p < M) ? load4(reinterpret_cast<const T*>(a.ep.r) +
                                         pixel_off(p, a.ep.rs_n, a.ep.rs_h, a.ep.rs_w) + 4 * g)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float4 acc[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int c4 = 0; c4 < CI / 4; ++c4) {
        float4 xv[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u)
          xv[u] = load4(reinterpret_cast<const T*>(xs + (pg + u * kGroups) * kPitch) + 4 * c4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float4 w4 = ws[(4 * c4 + e) * G + g];
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            // channel pairs through packed FMAs (each lane one fmaf; measured
            // 2-30 % faster here, most with bf16 storage)
            const float xsv = comp(xv[u], e);
            const float2 xx = make_float2(xsv, xsv);
            const float2 lo = __ffma2_rn(xx, make_float2(w4.x, w4.y), make_float2(acc[u].x, acc[u].y));
            const float2 hi = __ffma2_rn(xx, make_float2(w4.z, w4.w), make_float2(acc[u].z, acc[u].w));
            acc[u] = make_float4(lo.x, lo.y, hi.x, hi.y);
          }
        }
      }
      const float4 sc = ssc[g], bi = sbi[g];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int lp = pg + u * kGroups;
        const long long p = tile * kTile + lp;
        if (p >= M) continue;
        store4(reinterpret_cast<T*>(a.out.y) + pixel_off(p, a.out.ys_n, a.out.ys_h, a.out.ys_w) + 4 * g,
               pw_epilogue(acc[u], sc, bi, rv[u], a.ep.act, a.ep.res_mode));
      }
    }
    __syncthreads();  // a later iteration's copies overwrite this slot
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

template <int CI, int CO, bool RES, typename T>
cudaError_t pw_launch_res(const DirectArgs& a, int flat, int sms, cudaStream_t s) {
  using Sh = PwShape<CI, CO, T>;
  const size_t smem = Sh::smem_bytes(RES);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = smem_attr_once<pw_small_kernel<CI, CO, RES, T>>(smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pw_small_kernel<CI, CO, RES, T>, kPwThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const long long M = static_cast<long long>(a.N) * a.H * a.W;
  const long long tiles = (M + Sh::kTile - 1) / Sh::kTile;
  const long long cap = static_cast<long long>(sms) * per_sm;
  const unsigned blocks = static_cast<unsigned>(tiles < cap ? tiles : cap);
  return launch_pdl(pw_small_kernel<CI, CO, RES, T>, dim3(blocks), dim3(kPwThreads), smem, s, a, flat);
}

template <int CI, int CO>
cudaError_t pw_launch(const DirectArgs& a, int flat, int sms, cudaStream_t s) {
  const bool res = a.ep.res_mode != 0;
  if (a.bf16) {
    if constexpr (CI >= 8) {
      return res ? pw_launch_res<CI, CO, true, __nv_bfloat16>(a, flat, sms, s)
                 : pw_launch_res<CI, CO, false, __nv_bfloat16>(a, flat, sms, s);
    }
    return cudaErrorInvalidValue;
  }
  return res ? pw_launch_res<CI, CO, true, float>(a, flat, sms, s) : pw_launch_res<CI, CO, false, float>(a, flat, sms, s);
}

template <int CI>
cudaError_t pw_launch_co(const DirectArgs& a, int flat, int sms, cudaStream_t s) {
  switch (a.Co) {
    case 4: return pw_launch<CI, 4>(a, flat, sms, s);
    case 8: return pw_launch<CI, 8>(a, flat, sms, s);
    case 16: return pw_launch<CI, 16>(a, flat, sms, s);
    case 32: return pw_launch<CI, 32>(a, flat, sms, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool pointwise_small_ok(int ci, int co, bool bf16) {
  return (ci == 8 || ci == 16 || ci == 32 || (ci == 4 && !bf16)) && (co == 4 || co == 8 || co == 16 || co == 32);
}

cudaError_t launch_pointwise_small(const DirectArgs& a, bool flat, int sms, cudaStream_t s) {
  if (static_cast<long long>(a.N) * a.H * a.W == 0) return cudaSuccess;
  const int f = flat ? 1 : 0;
  switch (a.Ci) {
    case 4: return pw_launch_co<4>(a, f, sms, s);
    case 8: return pw_launch_co<8>(a, f, sms, s);
    case 16: return pw_launch_co<16>(a, f, sms, s);
    case 32: return pw_launch_co<32>(a, f, sms, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cb
