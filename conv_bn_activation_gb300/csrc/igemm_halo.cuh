// Dense 3x3 stride-1 pad-1 convolution as an implicit GEMM on the
// 5th-generation tensor cores, with the A operand taken from one shared-memory
// halo tile per input-channel chunk instead of one im2col gather per filter
// tap.
//
// GEMM view ("YOLO26N Inference Optimisation", NHWC migration: implicit GEMM
// mapping): D[pixel, co] = sum over taps and Cin of x[shifted pixel, ci] *
// W[co, tap, ci].  Here the output pixels of an image are numbered over a
// padded width Wp = W + 2: q = oy * Wp + ox, ox in [0, Wp); the two columns
// ox = W, W + 1 are computed and discarded.  In that numbering the input
// pixel that tap (dy, dx) needs for output q sits at a constant offset
//     (q - y_lo * Wp) + dy * Wp + dx
// inside a halo tile holding input rows y_lo - 1 ... of the image, each
// padded by one zero column on both sides (y_lo = first output row of the
// tile).  So the nine taps of a 128-pixel tile are nine row offsets into ONE
// tile in shared memory: the copy engine fetches each input element about
// once per (tile, chunk) instead of nine times, and the tensor core reads
// the shifted rows straight from the swizzled tile (the 128-byte swizzle is
// a function of the shared-memory address, so a descriptor may start at any
// 128-byte row of a tile that TMA wrote).
//
// Tile: PX consecutive q of one image x CO output channels; K walks 32-channel
// chunks, and inside a chunk the nine taps (K = 32 each, four MMAs of K = 8).
// Two operand orders share this kernel:
//  * pixel-major (PX = 128, CO = BN in 32..256): the accumulator holds
//    pixels x channels, A = shifted halo rows, B = weights (M = 128, N = BN);
//  * channel-major (PX = 256 or 192, CO = 128): the accumulator holds
//    channels x pixels, A = weights, B = shifted halo rows (M = 128, N = PX).
//    On GB300 a kind::tf32 MMA costs about the same issue time for N = 64
//    and N = 128 and only a little more for N = 256 (111 / 111 / 128 cycles
//    per K = 8 step, measured), so a layer with 128 output channels runs its
//    tensor cores ~1.7x faster with 256 pixels as N than with its 128
//    channels as N.  The 192-pixel tile gives a layer of about 100 256-pixel
//    tiles (128 -> 128 channels at 40 x 40, batch 16) a tile for nearly
//    every SM instead of leaving a third of them idle.
//  * warp 0: TMA producer.  Lane 0 loads the halo tile of each (tile, chunk)
//    -- a 4-D tiled copy of R input rows x Wp columns x 32 channels starting
//    at (column -1, row y_lo - 1): rows and columns outside the image arrive
//    as zeros, which is the convolution's zero padding.  Lanes 1-3 load the
//    [CO x 32] weight slices, one per tap, each lane owning every third ring
//    stage (copies from different lanes overlap; one lane's complete one
//    after another).
//  * warp 1 (one thread): tcgen05.mma kind::tf32 (M = 128, N = CO or PX, K = 8)
//    into one of NACC TMEM accumulators; tcgen05.commit releases weight
//    stages, halo tiles and, at the end of a tile, the accumulator.
//  * warps 2-9: epilogue (two groups of four warps, one per TMEM lane
//    quarter), columns ox >= W and rows past the image masked.  Pixel-major
//    chunks are written back through TileStore (a transpose in shared memory
//    that makes the stores coalesced); a channel-major chunk already holds
//    32 consecutive channels of each pixel across a warp, so it is stored
//    straight from registers (cm_store).
// CTAs are persistent and stride over the (pixel tile, channel tile) pairs.
//
// Split K (split_k = 2, layers with fewer tiles than half the SMs): CTA
// pairs launched as clusters of two share each tile, CTA r taking half of
// the 32-channel chunks.  After its MMAs each CTA tells its partner that its
// operand buffers are free (a remote mbarrier arrive); each then stores the
// half of its accumulator that the partner finalises into the partner's
// shared memory (distributed shared memory, over the free buffers), arrives
// on the partner's data barrier, waits for the partner's half, adds it to
// its own (fp32, a + b in either CTA) and runs the epilogue on its half of
// the columns.  Every wait is bounded; a cluster barrier at exit keeps
// either CTA from leaving while its partner may still write to it.
#pragma once

#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"
#include "tc_store.cuh"
#include "trace.cuh"

#include <type_traits>

namespace cb {

constexpr int kHaloThreads = 320;
constexpr int kHaloKc = 32;              // input channels per K chunk (128-byte rows), or KC = 16 (64-byte rows)
constexpr int kHaloStagingBytes = 8 * TileStore<32>::kBufBytes;  // 8 epilogue warps x 4 KB

// TMEM accumulators per CTA (the epilogue of one tile overlaps the MMAs of
// the next ones) and the power-of-two column count they occupy, for an
// accumulator of acc_cols columns.  Narrow tiles keep eight, so that a tile
// of up to four 128-pixel sub-tiles (one halo copy for all of them) can run
// while the previous one is stored.
__host__ __device__ constexpr int halo_naccs(int acc_cols) { return acc_cols > 128 ? 2 : acc_cols <= 64 ? 8 : 4; }
__host__ __device__ constexpr int halo_tmem_cols(int acc_cols) {
  return halo_naccs(acc_cols) * acc_cols <= 128 ? 128 : halo_naccs(acc_cols) * acc_cols <= 256 ? 256 : 512;
}

// Channel-major write-back of one 32-pixel chunk.  Thread `lane` holds
// output channel c for the chunk's 32 pixels (v[p] = pixel p), so for each
// pixel the warp's lanes hold 32 consecutive channels and one store
// instruction writes a contiguous pixel segment: no transpose through shared
// memory.  yoff / roff are pixel `lane`'s element offsets (yoff < 0: a
// padding column or past the image), passed to every lane pixel by pixel.
template <int ACT, int RES, typename T>
__device__ __forceinline__ void cm_store_t(const uint32_t (&v)[32], long long yoff, long long roff, int c, bool cin,
                                           float sc, float bi, const OutView& out, const Epilogue& ep) {
  T* y = reinterpret_cast<T*>(out.y) + c;
  const T* rb = reinterpret_cast<const T*>(ep.r) + c;
#pragma unroll
  for (int g = 0; g < 32; g += 8) {
    long long yo[8];
    float r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      yo[i] = __shfl_sync(0xffffffffu, yoff, g + i);
      r[i] = 0.0f;
      if constexpr (RES != 0) {
        const long long ro = __shfl_sync(0xffffffffu, roff, g + i);
        if (yo[i] >= 0 && cin) r[i] = load1(rb + ro);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float z = tc_epi_post<ACT, RES, T>(fmaf(__uint_as_float(v[g + i]), sc, bi), r[i]);
      if (yo[i] >= 0 && cin) store1(y + yo[i], z);
    }
  }
}

template <typename T>
__device__ __forceinline__ void cm_store(const uint32_t (&v)[32], long long yoff, long long roff, int c, bool cin,
                                         float sc, float bi, const OutView& out, const Epilogue& ep) {
  switch (ep.act * 3 + ep.res_mode) {
    case 0: cm_store_t<0, 0, T>(v, yoff, roff, c, cin, sc, bi, out, ep); break;
    case 1: cm_store_t<0, 1, T>(v, yoff, roff, c, cin, sc, bi, out, ep); break;
    case 2: cm_store_t<0, 2, T>(v, yoff, roff, c, cin, sc, bi, out, ep); break;
    case 3: cm_store_t<1, 0, T>(v, yoff, roff, c, cin, sc, bi, out, ep); break;
    case 4: cm_store_t<1, 1, T>(v, yoff, roff, c, cin, sc, bi, out, ep); break;
    case 5: cm_store_t<1, 2, T>(v, yoff, roff, c, cin, sc, bi, out, ep); break;
    case 6: cm_store_t<2, 0, T>(v, yoff, roff, c, cin, sc, bi, out, ep); break;
    case 7: cm_store_t<2, 1, T>(v, yoff, roff, c, cin, sc, bi, out, ep); break;
    default: cm_store_t<2, 2, T>(v, yoff, roff, c, cin, sc, bi, out, ep); break;
  }
}

template <int PX, int CO, bool CM, int KC = kHaloKc, typename T = float>
__global__ void __launch_bounds__(kHaloThreads, 1) igemm_halo_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                     const __grid_constant__ CUtensorMap wmap,
                                                                     const HaloArgs a) {
  static_assert(KC == 32 || KC == 16 || KC == 8, "row bytes / 4 per chunk");
  // KC sizes a chunk in 4-byte units: one pixel's chunk is kRowBytes = 128,
  // 64 or 32 bytes (swizzled to match), i.e. KC fp32 or 2 KC bf16 channels.
  constexpr int kRowBytes = KC * 4;
  constexpr int kChan = kRowBytes / static_cast<int>(sizeof(T));  // channels per chunk
  static_assert(CM ? ((PX == 256 || PX == 192) && CO == 128)
                   : (PX == 128 && (CO == 32 || CO == 64 || CO == 128 || CO == 256)),
                "tile shape");
  const unsigned long long t_start = a.trace ? trace_globaltimer() : 0;
  constexpr int kAccCols = CM ? PX : CO;  // TMEM columns of one accumulator
  // column distance between accumulators: a wide one (two per CTA) starts on
  // a 256-column boundary
  constexpr int kAccStride = kAccCols > 128 ? 256 : kAccCols;
  // Sub-tiles: a tile of nsub x 128 consecutive pixels shares one halo copy;
  // each 128-pixel sub-tile has its own accumulator (pixel-major only).
  const int sub = CM ? 1 : a.sub;
  constexpr int NACC = halo_naccs(kAccCols);
  constexpr uint32_t kTmemCols = halo_tmem_cols(kAccCols);
  static_assert(NACC * kAccStride <= static_cast<int>(kTmemCols), "accumulators within the allocation");
  static_assert(kAccCols % 64 == 0 || kAccCols == 32, "split-K halves of whole 32-column chunks");
  constexpr int kTapBytes = CO * KC * 4;  // one tap's weight slice
  const int tps = a.taps_per_stage;            // taps per weight-ring stage: 1, 3 or 9 (one copy each)
  const int kBBytes = tps * kTapBytes;
  constexpr uint32_t kIdesc = CM ? idesc_for<T>(CO, PX) : idesc_for<T>(PX, CO);
  // Epilogue split of a tile between the two groups of four warps:
  // pixel-major tiles of 32 channels alternate between the groups, wider
  // ones are split into column halves; channel-major tiles give the groups
  // alternate 32-pixel chunks.  Either way in 32-column chunks.  Channel-major
  // chunks are stored straight from registers (cm_store), pixel-major ones
  // through the warp's staging buffer (TileStore).
  constexpr bool kSplitTiles = !CM && CO == 32;
  constexpr int kWidth = CM ? PX / 2 : (kSplitTiles ? CO : CO / 2);
  constexpr int kChunks = kWidth / 32;
  constexpr int kEpiArrivals = kSplitTiles ? 4 : 8;
  constexpr int kBLanes = 3;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sHalo = smem;                                  // 2 x halo_bytes
  uint8_t* sB = sHalo + 2 * a.halo_bytes;                 // nb x kBBytes
  uint8_t* sStage = sB + a.nb_stages * kBBytes;           // epilogue staging
  uint64_t* hfull = reinterpret_cast<uint64_t*>(sStage + kHaloStagingBytes);
  uint64_t* hempty = hfull + 2;
  uint64_t* bfull = hempty + 2;
  uint64_t* bempty = bfull + a.nb_stages;
  uint64_t* tfull = bempty + a.nb_stages;
  uint64_t* tempty = tfull + NACC;
  uint64_t* xfree = tempty + NACC;  // split K: the partner's operand buffers are free
  uint64_t* xdata = xfree + 1;      // split K: the partner's half accumulator has landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xdata + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int h = 0; h < 2; ++h) {
      mbar_init(&hfull[h], 1);
      mbar_init(&hempty[h], 1);
    }
    for (int s = 0; s < a.nb_stages; ++s) {
      mbar_init(&bfull[s], 1);
      mbar_init(&bempty[s], 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiArrivals);
    }
    mbar_init(xfree, 1);
    mbar_init(xdata, 256);  // every epilogue thread of the partner
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const int split = kSplitTiles ? 1 : a.split_k;  // 1, or 2: a cluster of two CTAs per tile
  if (split == 2) cluster_sync();  // both CTAs' barriers are initialised before any remote arrive
  const uint32_t rank = split == 2 ? cluster_ctarank() : 0u;
  const int kc_begin = rank ? a.num_kc / 2 : 0;
  const int kc_end = (split == 2 && rank == 0) ? a.num_kc / 2 : a.num_kc;
  const int tile0 = static_cast<int>(blockIdx.x) / split, tile_step = static_cast<int>(gridDim.x) / split;
  // This CTA holds its TMEM: the next kernel may launch (its CTAs cannot
  // take TMEM this one still needs); then wait for the previous kernel.
  pdl_launch_dependents();
  pdl_wait();
  const uint32_t tmem_base = *tmem_slot;
  const Watchdog wd{a.err, abort_flag, a.timeout_ns};
  const int num_tiles = a.m_tiles * a.n_tiles;
  const uint32_t halo_tx = static_cast<uint32_t>(kRowBytes * a.Wp * a.rows * (a.stride == 2 ? 4 : 1));
  // resident weights: the layer's whole weight tensor is one stage of nine
  // taps (one channel chunk, one channel tile), copied once per CTA
  const bool resident = a.w_resident != 0;
  const bool tr_cta = a.trace && blockIdx.x == a.trace_cta;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane <= kBLanes) {
      if (lane == 0) {
        tma_prefetch_desc(&xmap);
        tma_prefetch_desc(&wmap);
      }
      int h = 0, s = 0;
      uint32_t hphase = 0, bphase = 0, issued = 0, last_parity = 0;
      bool ok = true;
      TraceBuf tr;
      for (int tile = tile0; ok && tile < num_tiles; tile += tile_step) {
        const int m_tile = tile / a.n_tiles, n_tile = tile % a.n_tiles;
        const int n_img = m_tile / a.tiles_per_img;
        const int rem = m_tile - n_img * a.tiles_per_img;
        const int blk = rem / a.tiles_per_blk;
        const int q0 = (rem - blk * a.tiles_per_blk) * PX * sub;
        const int y_lo = q0 / a.Wp;
        const int x0 = blk * a.blk_w - 1;  // first column of the tile (phase column at stride 2)
        for (int kc = kc_begin; ok && kc < kc_end; ++kc) {
          if (lane == 0) {
            if (!mbar_wait(&hempty[h], hphase ^ 1u, wd)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&hfull[h], halo_tx);
            if (a.stride == 1) {
              tma_load_4d(sHalo + h * a.halo_bytes, &xmap, &hfull[h], kc * kChan, x0, y_lo - 1, n_img);
            } else {
              // four phase tiles: input rows 2i + py, columns 2j + px (element strides 2)
              for (int ph = 0; ph < 4; ++ph)
                tma_load_4d(sHalo + h * a.halo_bytes + ph * a.phase_bytes, &xmap, &hfull[h], kc * kChan,
                            2 * x0 + (ph & 1), 2 * (y_lo - 1) + (ph >> 1), n_img);
            }
            issued |= 1u << h;
            last_parity = (last_parity & ~(1u << h)) | (hphase << h);
          }
          if (++h == 2) {
            h = 0;
            hphase ^= 1u;
          }
          for (int tap = 0; tap < 9; tap += tps) {
            if (resident) {
              // one chunk, one channel tile: every tile takes the same nine
              // taps, loaded once into the single stage and kept
              if (lane == 1 && tile == tile0) {
                mbar_arrive_expect_tx(&bfull[0], static_cast<uint32_t>(kBBytes));
                tma_load_3d(sB, &wmap, &bfull[0], kc * kChan, n_tile * CO, 0);
                issued |= 1u;
              }
              continue;
            }
            if (lane != 0 && s % kBLanes == lane - 1) {
              if (!mbar_wait(&bempty[s], bphase ^ 1u, wd)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&bfull[s], static_cast<uint32_t>(kBBytes));
              // weights viewed as (Ci, Co, tap): one box of tps taps lands as tps [CO x 32] slices
              tma_load_3d(sB + s * kBBytes, &wmap, &bfull[s], kc * kChan, n_tile * CO, tap);
              tr.add(tr_cta && lane == 1);
              issued |= 1u << s;
              last_parity = (last_parity & ~(1u << s)) | (bphase << s);
            }
            if (++s == a.nb_stages) {
              s = 0;
              bphase ^= 1u;
            }
          }
        }
      }
      // Let every copy this lane issued land before the CTA can exit.
      if (lane == 0) {
        for (int hh = 0; hh < 2; ++hh)
          if (issued & (1u << hh)) mbar_wait_drain(&hfull[hh], (last_parity >> hh) & 1u, 20000000ull);
      } else {
        for (int ss = 0; ss < a.nb_stages; ++ss)
          if (issued & (1u << ss)) mbar_wait_drain(&bfull[ss], (last_parity >> ss) & 1u, 20000000ull);
      }
      tr.flush(tr_cta && lane == 1, 0);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int h = 0, s = 0;
      uint32_t hphase = 0, bphase = 0;
      uint32_t bcommitted = 0, bparity = 0, hcommitted = 0, hparity = 0, tcommitted = 0, tparity = 0;
      bool ok = true;
      int local = 0;
      TraceBuf tr;
      // The issue rate of this thread bounds the narrow tiles, so the chunk
      // loop below is specialised on (taps per stage, sub-tiles) and fully
      // unrolled: each MMA takes one add to its descriptors' address field
      // (16-byte units).  tap_off[t] places tap t inside a halo buffer.
      constexpr uint32_t kRowOff = kRowBytes >> 4;
      constexpr uint32_t kSubOff = (PX * kRowBytes) >> 4;
      constexpr uint32_t kTapOff = kTapBytes >> 4;
      uint32_t tap_off[9];
#pragma unroll
      for (int t = 0; t < 9; ++t) {
        const int dy = t / 3, dx = t % 3;
        const uint32_t wp_off = static_cast<uint32_t>(a.Wp) * kRowOff;
        // stride 2: input row 2 oy + dy - 1 is phase row (dy != 1) at oy - 1 + (dy != 0); columns alike
        tap_off[t] = a.stride == 1 ? dy * wp_off + dx * kRowOff
                                   : ((dy != 1 ? 2u : 0u) + (dx != 1 ? 1u : 0u)) * (static_cast<uint32_t>(a.phase_bytes) >> 4) +
                                         (dy != 0 ? wp_off : 0u) + (dx != 0 ? kRowOff : 0u);
      }
      // every descriptor shares its high word (stride, swizzle mode)
      const uint32_t desc_hi = static_cast<uint32_t>(kmajor_swizzled_desc(0u, kRowBytes) >> 32);
      auto desc_lo = [](uint32_t saddr) { return static_cast<uint32_t>(kmajor_swizzled_desc(saddr, kRowBytes)); };
      auto make_desc = [&](uint32_t lo) { return (static_cast<uint64_t>(desc_hi) << 32) | lo; };
      // One K chunk of a tile: 9 taps x NSUB sub-tiles x KC / 8 MMAs, weight
      // stages of TPS taps.  Returns false when a wait timed out.
      bool w_ready = false;  // resident weights: landed (waited for once)
      auto issue_chunk = [&](auto tps_c, auto nsub_c, uint32_t x_lo, const uint32_t (&d_tmem)[kHaloMaxSub],
                             bool first) -> bool {
        constexpr int TPS = decltype(tps_c)::value, NSUB = decltype(nsub_c)::value;
        uint32_t w_lo = 0;
#pragma unroll
        for (int tap = 0; tap < 9; ++tap) {
          if (tap % TPS == 0) {
            if (!w_ready) {
              if (!mbar_wait(&bfull[s], bphase, wd)) return false;
              tr.add(tr_cta);
              tc_fence_after_sync();
              w_ready = resident;
            }
            w_lo = desc_lo(smem_u32(sB + s * kBBytes));
          }
          const uint32_t xt = x_lo + tap_off[tap], wt = w_lo + (tap % TPS) * kTapOff;
#pragma unroll
          for (int i = 0; i < NSUB; ++i) {
#pragma unroll
            for (int kk = 0; kk < KC / 8; ++kk) {
              const uint64_t xd = make_desc(xt + i * kSubOff + 2 * kk), wdsc = make_desc(wt + 2 * kk);
              mma_op<T>(d_tmem[i], CM ? wdsc : xd, CM ? xd : wdsc, kIdesc, (tap == 0 && kk == 0 && first) ? 0u : 1u);
            }
          }
          if (tap % TPS == TPS - 1 && !resident) {
            mma_commit(&bempty[s]);
            tr.add(tr_cta);
            const uint32_t bit = 1u << s;
            bparity = (bcommitted & bit) ? (bparity ^ bit) : (bparity & ~bit);
            bcommitted |= bit;
            if (++s == a.nb_stages) {
              s = 0;
              bphase ^= 1u;
            }
          }
        }
        return true;
      };
      using I1 = std::integral_constant<int, 1>;
      using I2 = std::integral_constant<int, 2>;
      using I3 = std::integral_constant<int, 3>;
      using I4 = std::integral_constant<int, 4>;
      using I9 = std::integral_constant<int, 9>;
      auto issue_tps = [&](auto nsub_c, uint32_t x_lo, const uint32_t (&d_tmem)[kHaloMaxSub], bool first) -> bool {
        return tps == 9 ? issue_chunk(I9{}, nsub_c, x_lo, d_tmem, first)
             : tps == 3 ? issue_chunk(I3{}, nsub_c, x_lo, d_tmem, first)
                        : issue_chunk(I1{}, nsub_c, x_lo, d_tmem, first);
      };
      for (int tile = tile0; ok && tile < num_tiles; tile += tile_step) {
        const int m_tile = tile / a.n_tiles;
        const int n_img = m_tile / a.tiles_per_img;
        const int rem = m_tile - n_img * a.tiles_per_img;
        const int gi = rem - (rem / a.tiles_per_blk) * a.tiles_per_blk;
        const int q0 = gi * PX * sub;
        const int nsub = min(sub, a.px_tiles_per_blk - gi * sub);
        const int base_row = q0 - (q0 / a.Wp) * a.Wp;
        // the accumulators of this tile's sub-tiles
        uint32_t d_tmem[kHaloMaxSub];
#pragma unroll
        for (int i = 0; i < kHaloMaxSub; ++i)
          d_tmem[i] = tmem_base + static_cast<uint32_t>(((local + i) & (NACC - 1)) * kAccStride);
        for (int i = 0; ok && i < nsub; ++i) {
          const int acc = (local + i) & (NACC - 1);
          if (!mbar_wait(&tempty[acc], (((local + i) / NACC) & 1) ^ 1u, wd)) ok = false;
        }
        if (!ok) break;
        tc_fence_after_sync();
        for (int kc = kc_begin; ok && kc < kc_end; ++kc) {
          if (!mbar_wait(&hfull[h], hphase, wd)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t x_lo = desc_lo(smem_u32(sHalo + h * a.halo_bytes) + static_cast<uint32_t>(base_row * kRowBytes));
          const bool first = kc == kc_begin;
          if (CM || CO > 64 || nsub == 1) ok = issue_tps(I1{}, x_lo, d_tmem, first);
          else if (nsub == 2) ok = issue_tps(I2{}, x_lo, d_tmem, first);
          else if (nsub == 3) ok = issue_tps(I3{}, x_lo, d_tmem, first);
          else ok = issue_tps(I4{}, x_lo, d_tmem, first);
          if (!ok) break;
          mma_commit(&hempty[h]);
          const uint32_t hbit = 1u << h;
          hparity = (hcommitted & hbit) ? (hparity ^ hbit) : (hparity & ~hbit);
          hcommitted |= hbit;
          if (++h == 2) {
            h = 0;
            hphase ^= 1u;
          }
        }
        if (!ok) break;
        for (int i = 0; i < nsub; ++i) {
          const int acc = (local + i) & (NACC - 1);
          mma_commit(&tfull[acc]);
          const uint32_t tbit = 1u << acc;
          tparity = (tcommitted & tbit) ? (tparity ^ tbit) : (tparity & ~tbit);
          tcommitted |= tbit;
        }
        local += nsub;
      }
      // Let every MMA this thread issued finish before TMEM is released.
      for (int ss = 0; ss < a.nb_stages; ++ss)
        if (bcommitted & (1u << ss)) mbar_wait_drain(&bempty[ss], (bparity >> ss) & 1u, 20000000ull);
      for (int hh = 0; hh < 2; ++hh)
        if (hcommitted & (1u << hh)) mbar_wait_drain(&hempty[hh], (hparity >> hh) & 1u, 20000000ull);
      for (int b = 0; b < NACC; ++b)
        if (tcommitted & (1u << b)) mbar_wait_drain(&tfull[b], (tparity >> b) & 1u, 20000000ull);
      tr.flush(tr_cta, 1);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int group = (warp - 2) >> 2;
    const int col0 = (CM || kSplitTiles) ? 0 : group * kWidth;
    uint8_t* stage_buf = sStage + (warp - 2) * TileStore<32>::kBufBytes;
    const bool res = a.ep.res_mode != 0;
    const bool vec = a.vec_store != 0;
    int local = 0;
    TraceBuf tr;
    const bool tr_on = tr_cta && warp == 2 && lane == 0;
    for (int tile = tile0, si = 0, nsub = 0; tile < num_tiles; ++local) {
      // walk the sub-tiles of each tile in turn
      if (si == nsub) {
        if (nsub) {
          tile += tile_step;
          if (tile >= num_tiles) break;
        }
        const int mt = tile / a.n_tiles, rm = mt - (mt / a.tiles_per_img) * a.tiles_per_img;
        const int g = rm - (rm / a.tiles_per_blk) * a.tiles_per_blk;
        nsub = min(sub, a.px_tiles_per_blk - g * sub);
        si = 0;
      }
      const int sub_i = si++;
      if (kSplitTiles && (local & 1) != group) continue;
      const int acc = local % NACC;
      const uint32_t acc_phase = (local / NACC) & 1;
      const int m_tile = tile / a.n_tiles, n_tile = tile % a.n_tiles;
      const int n_img = m_tile / a.tiles_per_img;
      const int rem = m_tile - n_img * a.tiles_per_img;
      const int blk = rem / a.tiles_per_blk;
      const int q0 = ((rem - blk * a.tiles_per_blk) * sub + sub_i) * PX;
      // Element offsets of output pixel q (-1: a padding column or past the image).
      auto pixel_offsets = [&](int qq, long long& yoff, long long& roff) {
        const int oy = qq / a.Wp, oxl = qq - (qq / a.Wp) * a.Wp;
        const int ox = blk * a.blk_w + oxl;
        const bool valid = oy < a.OH && oxl < a.blk_w && ox < a.OW;
        yoff = valid ? n_img * a.out.ys_n + oy * a.out.ys_h + static_cast<long long>(ox) * a.out.ys_w : -1;
        roff = (valid && res) ? n_img * a.ep.rs_n + oy * a.ep.rs_h + static_cast<long long>(ox) * a.ep.rs_w : 0;
      };

      // channel-major: this thread's output channel and its folded-BN scale / bias, the same in every chunk (in flight
      // while the accumulator is waited for)
      const int cm_c = n_tile * CO + q * 32 + lane;
      const bool cm_cin = CM && cm_c < a.Cout;
      const float cm_sc = cm_cin ? __ldg(a.ep.scale + cm_c) : 0.0f, cm_bi = cm_cin ? __ldg(a.ep.bias + cm_c) : 0.0f;
      bool got = mbar_wait(&tfull[acc], acc_phase, wd);
      got = __all_sync(0xffffffffu, got);
      if (!got) break;
      tc_fence_after_sync();
      tr.add(tr_on);
      const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kAccStride);
      if (!kSplitTiles && split == 2) {
        // One tile per cluster (the host guarantees it): exchange halves.
        constexpr int kHalf = kAccCols / 2, kHalfChunks = kHalf / 32;
        // [kHalf / 4 column quads][128 lanes][4], over the halo / weight
        // buffers: each 16-byte store or load of a warp covers 512
        // contiguous bytes
        float* recv = reinterpret_cast<float*>(smem);
        const uint32_t partner = rank ^ 1u;
        const int own0 = static_cast<int>(rank) * kHalf, exp0 = kHalf - own0;
        // every MMA of this CTA is done (tfull): its operand buffers are free
        if (warp == 2 && lane == 0) mbar_arrive_remote(map_shared_rank(smem_u32(xfree), partner));
        bool ready = mbar_wait_cluster(xfree, 0, wd);
        ready = __all_sync(0xffffffffu, ready);
        tr.add(tr_on);
        if (ready) {
          const uint32_t rrecv = map_shared_rank(smem_u32(recv), partner);
          for (int i = group; i < kHalfChunks; i += 2) {
            uint32_t v[32];
            tmem_ld_cols<32>(lane_base + exp0 + i * 32, v);
            tmem_wait_regs(v);
            const uint32_t dst = rrecv + static_cast<uint32_t>((i * 8 * 128 + q * 32 + lane) * 16);
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              st_cluster_v4(dst + static_cast<uint32_t>(j / 4 * 128 * 16), v[j], v[j + 1], v[j + 2], v[j + 3]);
          }
          mbar_arrive_remote(map_shared_rank(smem_u32(xdata), partner));
        }
        tr.add(tr_on);
        bool have = mbar_wait_cluster(xdata, 0, wd);
        have = __all_sync(0xffffffffu, have);
        tr.add(tr_on);
        if (!have) break;
        for (int i = group; i < kHalfChunks; i += 2) {
          uint32_t v[32];
          tmem_ld_cols<32>(lane_base + own0 + i * 32, v);
          tmem_wait_regs(v);
          const float4* rp = reinterpret_cast<const float4*>(recv) + i * 8 * 128 + q * 32 + lane;
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 r4 = rp[j / 4 * 128];
            v[j] = __float_as_uint(__uint_as_float(v[j]) + r4.x);
            v[j + 1] = __float_as_uint(__uint_as_float(v[j + 1]) + r4.y);
            v[j + 2] = __float_as_uint(__uint_as_float(v[j + 2]) + r4.z);
            v[j + 3] = __float_as_uint(__uint_as_float(v[j + 3]) + r4.w);
          }
          long long yoff, roff;
          __syncwarp();
          if constexpr (!CM) {
            pixel_offsets(q0 + q * 32 + lane, yoff, roff);
            const TileStore<32>::Consts k =
                TileStore<32>::consts(lane, n_tile * CO + own0 + i * 32, a.Cout, vec, a.ep);
            TileStore<32>::stage(stage_buf, lane, v);
            __syncwarp();
            TileStore<32>::template write<T>(stage_buf, lane, yoff, roff, k, a.Cout, a.out, a.ep);
          } else {
            pixel_offsets(q0 + own0 + i * 32 + lane, yoff, roff);
            cm_store<T>(v, yoff, roff, cm_c, cm_cin, cm_sc, cm_bi, a.out, a.ep);
          }
          tr.add(tr_on);
        }
        continue;
      }
      if constexpr (!CM) {
        // thread = pixel row q0 + 32q + lane; chunks of 32 channels
        // The scale / bias of chunk k + 1 are in flight while chunk k is
        // staged and stored.
        long long yoff, roff;
        pixel_offsets(q0 + q * 32 + lane, yoff, roff);
        const int cbase = n_tile * CO + col0;
        TileStore<32>::Consts k = TileStore<32>::consts(lane, cbase, a.Cout, vec, a.ep);
#pragma unroll 1
        for (int cidx = 0; cidx < kChunks; ++cidx) {
          uint32_t v[32];
          tmem_ld_cols<32>(lane_base + col0 + cidx * 32, v);
          tmem_wait_regs(v);
          TileStore<32>::Consts kn = k;
          if (cidx + 1 < kChunks) {
            kn = TileStore<32>::consts(lane, cbase + (cidx + 1) * 32, a.Cout, vec, a.ep);
          } else {
            // every column of this warp's quarter is in registers: release the accumulator
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
          }
          __syncwarp();  // the previous chunk's readers are done with the staging buffer
          TileStore<32>::stage(stage_buf, lane, v);
          __syncwarp();
          TileStore<32>::template write<T>(stage_buf, lane, yoff, roff, k, a.Cout, a.out, a.ep);
          k = kn;
        }
      } else {
        // thread = output channel cm_c; chunks of 32 pixels, group g taking
        // chunks g, g + 2, ...
#pragma unroll 1
        for (int cidx = group; cidx < PX / 32; cidx += 2) {
          uint32_t v[32];
          tmem_ld_cols<32>(lane_base + cidx * 32, v);
          tmem_wait_regs(v);
          if (cidx + 2 >= PX / 32) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
          }
          tr.add(tr_on);
          long long yoff, roff;
          pixel_offsets(q0 + cidx * 32 + lane, yoff, roff);
          cm_store<T>(v, yoff, roff, cm_c, cm_cin, cm_sc, cm_bi, a.out, a.ep);
          tr.add(tr_on);
        }
      }
      tr.add(tr_on);
    }
    tr.flush(tr_on, 2);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (split == 2) cluster_sync();  // the partner no longer touches this CTA's shared memory
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0) {
    trace_cta_span(a.trace, 0, t_start);
    trace_cta_span(a.trace, 1, trace_globaltimer());
  }
}

// Launch of one instantiation (clusters of two CTAs for split K), and how
// many such clusters the device runs at once (0 if none).
template <int PX, int CO, bool CM, int KC = kHaloKc, typename T = float>
cudaError_t halo_launch(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int grid, size_t smem,
                        cudaStream_t s) {
  cudaError_t e = smem_attr_once<igemm_halo_kernel<PX, CO, CM, KC, T>>(smem);
  if (e != cudaSuccess) return e;
  if (a.split_k == 2)
    return launch_pdl_cluster(igemm_halo_kernel<PX, CO, CM, KC, T>, dim3(grid), dim3(kHaloThreads), smem, s, 2, xmap,
                              wmap, a);
  return launch_pdl(igemm_halo_kernel<PX, CO, CM, KC, T>, dim3(grid), dim3(kHaloThreads), smem, s, xmap, wmap, a);
}

template <int PX, int CO, bool CM>
int halo_pairs(size_t smem) {
  if (smem_attr_once<igemm_halo_kernel<PX, CO, CM>>(smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kHaloThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, igemm_halo_kernel<PX, CO, CM>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace cb
