// Dense convolution (kh x kw = 1x1 or 3x3, stride 1 or 2, groups 1) as an
// implicit GEMM on the 5th-generation tensor cores, with the folded-BN /
// residual / activation epilogue fused.
//
// GEMM view ("YOLO26N Inference Optimisation", NHWC migration: implicit GEMM
// mapping): A = im2col(x) [M = N*OH*OW, K = kh*kw*Cin], B = W [Cout, K],
// D = A * B^T [M, Cout] -- which is the NHWC output.  NHWC keeps Cin
// contiguous, so every K step is a dense row per output pixel.
//
// Tile: 128 output pixels (consecutive in (n, oh, ow) order, wrapping across
// rows and images) x BN output channels.  K is walked tap by tap, KC input
// channels at a time: KC = 32 (128-byte rows, 128-byte swizzle) in general,
// KC = 16 or 8 (64- / 32-byte rows and swizzles) for layers with 16 or 8
// input channels, so that the copy engine moves no padding channels.
//  * warp 0 (four lanes taking K steps in turn): TMA producer.  For tiles of
//    blk_h x blk_w output pixels of one image (blk_w != 0) the A tile of a
//    (tap, chunk) is one tiled copy: a box of KC channels x (stride * blk_w)
//    x (stride * blk_h) input elements traversed with element strides equal
//    to the conv stride, started at the tap's offset (the copy engine takes
//    about one 128-byte row per clock this way, against several per row in
//    im2col mode; zero fill outside the image is the padding).  Otherwise:
//    The A tile comes from an im2col-mode
//    tensor copy: the map's bounding box enumerates exactly the output pixel
//    positions (lower corner -pad, upper corner pad - (k - 1), traversal
//    stride = conv stride) and the per-copy offsets select the filter tap,
//    so padding and the OW / OH / batch tails are handled by the copy engine
//    (out-of-image pixels and channels >= Cin arrive as zeros).  The B tile
//    is a 3-D tiled copy of the [Cout][tap][Cin] weights.
//  * warp 1 (one thread): issues tcgen05.mma kind::tf32 (M=128, N=BN, K=8;
//    KC/8 per step) into a TMEM accumulator; tcgen05.commit releases each
//    smem stage and, at the end of a tile, the accumulator.
//  * warps 2-9: epilogue, two groups of four warps (one per TMEM lane
//    quarter = 32 output pixels).  Narrow tiles go to the groups in turn;
//    wide tiles are split by columns between them.  Each warp reads its
//    lanes with tcgen05.ld and writes them back through TileStore: staged in
//    shared memory, then scale/bias, residual, activation and TF32 rounding
//    applied pixel-major with coalesced stores.  Rows past M and channels
//    past Cout are masked, so nothing is written outside the logical output
//    (padded output rows stay untouched -- "YOLO26N Inference Optimisation",
//    Bug fixed: TMA overflow).
// Two to four TMEM accumulators let the epilogues of earlier tiles overlap
// the MMAs of later ones.  CTAs are persistent (one per SM) and stride over
// the tiles.
#pragma once

#include "epilogue.cuh"
#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"
#include "tc_store.cuh"
#include "trace.cuh"

namespace cb {

constexpr int kTileM = 128;
constexpr int kEpiWarps = 8;
constexpr int kProducerLanes = 4;
constexpr int kIgemmThreads = 64 + 32 * kEpiWarps;

constexpr int kIgemmStagingBytes = kEpiWarps * TileStore<16>::kBufBytes;  // chunks of at most 16 columns
__host__ __device__ constexpr int igemm_a_bytes(int kc) { return kTileM * kc * 4; }
__host__ __device__ constexpr int igemm_b_bytes(int bn, int kc) { return ((bn * kc * 4) + 1023) / 1024 * 1024; }
// TMEM accumulators per CTA: narrow tiles keep four in flight so the MMAs can
// run ahead of the epilogue; wide tiles two.
__host__ __device__ constexpr int igemm_naccs(int bn) { return bn <= 64 ? 4 : 2; }
__host__ __device__ constexpr int tmem_cols_for(int cols) {
  return cols <= 32 ? 32 : cols <= 64 ? 64 : cols <= 128 ? 128 : cols <= 256 ? 256 : 512;
}

template <int BN, int KC, typename T = float>
__global__ void __launch_bounds__(kIgemmThreads, 1) igemm_tf32_kernel(const __grid_constant__ CUtensorMap amap,
                                                                      const __grid_constant__ CUtensorMap bmap,
                                                                      const IgemmArgs a) {
  constexpr int kABytes = igemm_a_bytes(KC);
  constexpr int kBBytes = igemm_b_bytes(BN, KC);
  // KC sizes a K step in 4-byte units: rows of KC * 4 bytes, KC fp32 or 2 KC bf16 channels
  constexpr int kRowBytes = KC * 4;
  constexpr int kChan = kRowBytes / static_cast<int>(sizeof(T));
  constexpr uint32_t kIdesc = idesc_for<T>(kTileM, BN);
  constexpr int NACC = igemm_naccs(BN);
  constexpr uint32_t kTmemCols = tmem_cols_for(NACC * BN);
  // Epilogue split: for narrow tiles the two 4-warp groups take alternate
  // tiles (each warp all BN columns of its 32 rows); for wide tiles both
  // groups take every tile and split its columns in halves.
  constexpr bool kSplitTiles = BN < 64;
  constexpr int kWidth = kSplitTiles ? BN : BN / 2;
  constexpr int CH = (kWidth % 16 == 0) ? 16 : 8;
  constexpr int kChunks = kWidth / CH;
  constexpr int kEpiArrivals = kSplitTiles ? 4 : 8;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + a.stages * kABytes;
  uint8_t* sStage = sB + a.stages * kBBytes;  // epilogue staging, one buffer per epilogue warp
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + kIgemmStagingBytes);
  uint64_t* empty = full + a.stages;
  uint64_t* tfull = empty + a.stages;
  uint64_t* tempty = tfull + NACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + NACC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiArrivals);
    }
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
  // This CTA holds its TMEM: the next kernel may launch (its CTAs cannot
  // take TMEM this one still needs); then wait for the previous kernel.
  pdl_launch_dependents();
  pdl_wait();
  const uint32_t tmem_base = *tmem_slot;
  const Watchdog wd{a.err, abort_flag, a.timeout_ns};
  const int num_tiles = a.m_tiles * a.n_tiles;
  const bool tr_cta = a.trace && blockIdx.x == a.trace_cta;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Copies issued by one thread complete one after another (~400-500
    // cycles each, measured on GB300), while copies from different lanes
    // overlap; so kProducerLanes lanes share the work, each owning the ring
    // stages s with s % kProducerLanes == lane.  Every lane walks the whole
    // (tile, tap, chunk) sequence and issues the steps that land in its
    // stages; one owner per stage keeps each lane's barrier phases its own.
    if (lane < kProducerLanes) {
      if (lane == 0) {
        tma_prefetch_desc(&amap);
        tma_prefetch_desc(&bmap);
      }
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_parity = 0;
      bool ok = true;
      TraceBuf tr;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int m_tile = tile / a.n_tiles, n_tile = tile % a.n_tiles;
        int n_img, w0, h0;
        if (a.blk_w) {
          const int per_img = a.blocks_x * a.blocks_y;
          n_img = m_tile / per_img;
          const int rem = m_tile - n_img * per_img;
          const int by = rem / a.blocks_x, bx = rem - by * a.blocks_x;
          w0 = bx * a.blk_w * a.stride - a.pad;
          h0 = by * a.blk_h * a.stride - a.pad;
        } else {
          const int m0 = m_tile * kTileM;
          n_img = m0 / a.OHW;
          const int rem = m0 - n_img * a.OHW;
          const int oh = rem / a.OW, ow = rem - (rem / a.OW) * a.OW;
          w0 = ow * a.stride - a.pad;
          h0 = oh * a.stride - a.pad;
        }
        for (int tap = 0; ok && tap < a.taps; ++tap) {
          const uint16_t off_h = static_cast<uint16_t>(tap / a.kw);
          const uint16_t off_w = static_cast<uint16_t>(tap % a.kw);
          for (int kc = 0; kc < a.num_kc; ++kc) {
            if (stage % kProducerLanes == lane) {
              if (!mbar_wait(&empty[stage], phase ^ 1u, wd)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(kABytes + BN * KC * 4));
              if (a.blk_w)
                tma_load_4d(sA + stage * kABytes, &amap, &full[stage], kc * kChan, w0 + off_w, h0 + off_h, n_img);
              else
                tma_load_im2col_4d(sA + stage * kABytes, &amap, &full[stage], kc * kChan, w0, h0, n_img, off_w,
                                   off_h);
              tma_load_3d(sB + stage * kBBytes, &bmap, &full[stage], kc * kChan, tap, n_tile * BN);
              tr.add(tr_cta && lane == 0);
              issued |= 1u << stage;
              last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
            }
            if (++stage == a.stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Let every copy this lane issued land before the CTA can exit.
      for (int s = 0; s < a.stages; ++s)
        if (issued & (1u << s)) mbar_wait_drain(&full[s], (last_parity >> s) & 1u, 20000000ull);
      tr.flush(tr_cta && lane == 0, 0);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t committed = 0, commit_parity = 0;  // per smem stage: last commit's phase parity
      uint32_t tcommitted = 0, tcommit_parity = 0;
      bool ok = true;
      int local = 0;
      TraceBuf tr;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++local) {
        const int acc = local % NACC;
        const uint32_t acc_phase = (local / NACC) & 1;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, wd)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int k = 0; k < a.k_iters; ++k) {
          if (!mbar_wait(&full[stage], phase, wd)) {
            ok = false;
            break;
          }
          tr.add(tr_cta);
          tc_fence_after_sync();
          const uint64_t adesc = kmajor_swizzled_desc(smem_u32(sA + stage * kABytes), kRowBytes);
          const uint64_t bdesc = kmajor_swizzled_desc(smem_u32(sB + stage * kBBytes), kRowBytes);
#pragma unroll
          for (int kk = 0; kk < KC / 8; ++kk) {
            // advance 32 bytes (8 tf32 or 16 bf16) along K inside the swizzled row
            mma_op<T>(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, kIdesc, (k | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          tr.add(tr_cta);
          // the commit completes the barrier phase the producer waits on next
          const uint32_t bit = 1u << stage;
          commit_parity = (committed & bit) ? (commit_parity ^ bit) : (commit_parity & ~bit);
          committed |= bit;
          if (++stage == a.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        const uint32_t tbit = 1u << acc;
        tcommit_parity = (tcommitted & tbit) ? (tcommit_parity ^ tbit) : (tcommit_parity & ~tbit);
        tcommitted |= tbit;
      }
      // Let every MMA this thread issued finish before TMEM is released.
      for (int s = 0; s < a.stages; ++s)
        if (committed & (1u << s)) mbar_wait_drain(&empty[s], (commit_parity >> s) & 1u, 20000000ull);
      for (int b = 0; b < NACC; ++b)
        if (tcommitted & (1u << b)) mbar_wait_drain(&tfull[b], (tcommit_parity >> b) & 1u, 20000000ull);
      tr.flush(tr_cta, 1);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int group = (warp - 2) >> 2;
    const int col0 = kSplitTiles ? 0 : group * kWidth;
    const int row = q * 32 + lane;          // tile row = output pixel within the tile
    uint8_t* stage_buf = sStage + (warp - 2) * TileStore<CH>::kBufBytes;
    const bool res = a.ep.res_mode != 0;
    const bool vec = a.vec_store != 0;
    int local = 0;
    TraceBuf tr;
    const bool tr_on = tr_cta && warp == 2 && lane == 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
      if (kSplitTiles && (local & 1) != group) continue;
      const int acc = local % NACC;
      const uint32_t acc_phase = (local / NACC) & 1;
      const int m_tile = tile / a.n_tiles, n_tile = tile % a.n_tiles;
      long long yoff = -1, roff = 0;
      int n_img = 0, oh = 0, ow = 0;
      bool valid;
      if (a.blk_w) {
        const int per_img = a.blocks_x * a.blocks_y;
        n_img = m_tile / per_img;
        const int rem = m_tile - n_img * per_img;
        const int by = rem / a.blocks_x, bx = rem - by * a.blocks_x;
        oh = by * a.blk_h + row / a.blk_w;
        ow = bx * a.blk_w + row % a.blk_w;
        valid = oh < a.OHW / a.OW && ow < a.OW;
      } else {
        const int m = m_tile * kTileM + row;
        valid = m < a.M;
        if (valid) {
          n_img = m / a.OHW;
          const int rem = m - n_img * a.OHW;
          oh = rem / a.OW;
          ow = rem - (rem / a.OW) * a.OW;
        }
      }
      if (valid) {
        yoff = n_img * a.out.ys_n + oh * a.out.ys_h + static_cast<long long>(ow) * a.out.ys_w;
        if (res) roff = n_img * a.ep.rs_n + oh * a.ep.rs_h + static_cast<long long>(ow) * a.ep.rs_w;
      }
      const int cbase = n_tile * BN + col0;

      bool got = mbar_wait(&tfull[acc], acc_phase, wd);
      got = __all_sync(0xffffffffu, got);
      if (!got) break;
      tc_fence_after_sync();
      tr.add(tr_on);
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN + col0);
      // The scale / bias of chunk k + 1 are in flight while chunk k is
      // staged and stored.
      typename TileStore<CH>::Consts k = TileStore<CH>::consts(lane, cbase, a.Cout, vec, a.ep);
#pragma unroll 1
      for (int cidx = 0; cidx < kChunks; ++cidx) {
        uint32_t v[CH];
        tmem_ld_cols<CH>(taddr + cidx * CH, v);
        tmem_wait_regs(v);
        typename TileStore<CH>::Consts kn = k;
        if (cidx + 1 < kChunks) {
          kn = TileStore<CH>::consts(lane, cbase + (cidx + 1) * CH, a.Cout, vec, a.ep);
        } else {
          // every column of this warp's quarter is in registers: release the accumulator
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
        }
        __syncwarp();  // the previous chunk's readers are done with the staging buffer
        TileStore<CH>::stage(stage_buf, lane, v);
        __syncwarp();
        TileStore<CH>::template write<T>(stage_buf, lane, yoff, roff, k, a.Cout, a.out, a.ep);
        k = kn;
      }
      tr.add(tr_on);
    }
    tr.flush(tr_on, 2);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int BN, int KC, typename T>
cudaError_t igemm_launch_bn(const CUtensorMap& amap, const CUtensorMap& bmap, const IgemmArgs& a, int grid,
                            size_t smem, cudaStream_t s) {
  cudaError_t e = smem_attr_once<igemm_tf32_kernel<BN, KC, T>>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(igemm_tf32_kernel<BN, KC, T>, dim3(grid), dim3(kIgemmThreads), smem, s, amap, bmap, a);
}

template <int KC, typename T = float>
cudaError_t igemm_launch_kc(const CUtensorMap& amap, const CUtensorMap& bmap, const IgemmArgs& a, int bn, int grid,
                            size_t smem, cudaStream_t s) {
  switch (bn) {
    case 16: return igemm_launch_bn<16, KC, T>(amap, bmap, a, grid, smem, s);
    case 32: return igemm_launch_bn<32, KC, T>(amap, bmap, a, grid, smem, s);
    case 48: return igemm_launch_bn<48, KC, T>(amap, bmap, a, grid, smem, s);
    case 64: return igemm_launch_bn<64, KC, T>(amap, bmap, a, grid, smem, s);
    case 96: return igemm_launch_bn<96, KC, T>(amap, bmap, a, grid, smem, s);
    case 128: return igemm_launch_bn<128, KC, T>(amap, bmap, a, grid, smem, s);
    case 192: return igemm_launch_bn<192, KC, T>(amap, bmap, a, grid, smem, s);
    case 256: return igemm_launch_bn<256, KC, T>(amap, bmap, a, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cb
