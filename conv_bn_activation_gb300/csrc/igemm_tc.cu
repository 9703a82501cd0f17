// Dense convolution (kh x kw = 1x1 or 3x3, stride 1 or 2, groups 1) as an
// implicit GEMM on the 5th-generation tensor cores, with the folded-BN /
// residual / activation epilogue fused.
//
// GEMM view ("YOLO26N Inference Optimisation", NHWC migration: implicit GEMM
// mapping): A = im2col(x) [M = N*OH*OW, K = kh*kw*Cin], B = W [Cout, K],
// D = A * B^T [M, Cout] -- which is the NHWC output.  NHWC keeps Cin
// contiguous, so every K step is a dense 128-byte row per output pixel.
//
// Tile: 128 output pixels (consecutive in (n, oh, ow) order, wrapping across
// rows and images) x BN output channels.  K is walked tap by tap, 32 input
// channels (128 bytes of fp32) at a time.
//  * warp 0 (one thread): TMA producer.  The A tile comes from an im2col-mode
//    tensor copy: the map's bounding box enumerates exactly the output pixel
//    positions (lower corner -pad, upper corner pad - (k - 1), traversal
//    stride = conv stride) and the per-copy offsets select the filter tap,
//    so padding and the OW / OH / batch tails are handled by the copy engine
//    (out-of-image pixels and channels >= Cin arrive as zeros).  The B tile
//    is a 3-D tiled copy of the [Cout][tap][Cin] weights.  Both use the
//    128-byte swizzle.
//  * warp 1 (one thread): issues tcgen05.mma kind::tf32 (M=128, N=BN, K=8;
//    four per 32-channel step) into a TMEM accumulator; tcgen05.commit
//    releases each smem stage and, at the end of a tile, the accumulator.
//  * warps 2-5: epilogue.  Each warp reads its 32 TMEM lanes (= 32 output
//    pixels) with tcgen05.ld, applies scale/bias, residual and activation,
//    rounds to the nearest TF32 value and stores the row segment.  (The MMA
//    truncates its fp32 operands to TF32, which biases every product toward
//    zero; storing round-to-nearest TF32 activations lets the next
//    tensor-core layer read them exactly, so the bias does not compound
//    along a chain.)  Rows past M and channels past Cout are
//    masked, so nothing is written outside the logical output (padded
//    output rows stay untouched -- "YOLO26N Inference Optimisation", Bug
//    fixed: TMA overflow).
// Two TMEM accumulators let the epilogue of tile i overlap the MMAs of tile
// i+1.  CTAs are persistent (one per SM) and stride over the tiles.
#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace cb {

constexpr int kTileM = 128;
constexpr int kKChunk = 32;                       // fp32 elements per 128-byte row
constexpr int kABytes = kTileM * kKChunk * 4;     // 16 KB per stage
constexpr int kThreads = 192;

__host__ __device__ constexpr int tmem_cols_for(int bn) {
  return (2 * bn <= 32) ? 32 : (2 * bn <= 64) ? 64 : (2 * bn <= 128) ? 128 : (2 * bn <= 256) ? 256 : 512;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) igemm_tf32_kernel(const __grid_constant__ CUtensorMap amap,
                                                                 const __grid_constant__ CUtensorMap bmap,
                                                                 const IgemmArgs a) {
  constexpr int kBBytes = BN * kKChunk * 4;
  constexpr uint32_t kIdesc = idesc_tf32(kTileM, BN);
  constexpr uint32_t kTmemCols = tmem_cols_for(BN);

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + a.stages * kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + a.stages * kBBytes);
  uint64_t* empty = full + a.stages;
  uint64_t* tfull = empty + a.stages;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
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
  const uint32_t tmem_base = *tmem_slot;
  const Watchdog wd{a.err, abort_flag, a.timeout_ns};
  const int num_tiles = a.m_tiles * a.n_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&amap);
      tma_prefetch_desc(&bmap);
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_parity = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int m_tile = tile / a.n_tiles, n_tile = tile % a.n_tiles;
        const int m0 = m_tile * kTileM;
        const int n_img = m0 / a.OHW;
        const int rem = m0 - n_img * a.OHW;
        const int oh = rem / a.OW, ow = rem - (rem / a.OW) * a.OW;
        const int w0 = ow * a.stride - a.pad, h0 = oh * a.stride - a.pad;
        for (int tap = 0; ok && tap < a.taps; ++tap) {
          const uint16_t off_h = static_cast<uint16_t>(tap / a.kw);
          const uint16_t off_w = static_cast<uint16_t>(tap % a.kw);
          for (int kc = 0; kc < a.num_kc; ++kc) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, wd)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(kABytes + kBBytes));
            tma_load_im2col_4d(sA + stage * kABytes, &amap, &full[stage], kc * kKChunk, w0, h0, n_img, off_w,
                               off_h);
            tma_load_3d(sB + stage * kBBytes, &bmap, &full[stage], kc * kKChunk, tap, n_tile * BN);
            issued |= 1u << stage;
            last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == a.stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      for (int s = 0; s < a.stages; ++s)
        if (issued & (1u << s)) mbar_wait_drain(&full[s], (last_parity >> s) & 1u, 20000000ull);
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
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, wd)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int k = 0; k < a.k_iters; ++k) {
          if (!mbar_wait(&full[stage], phase, wd)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + stage * kABytes));
          const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sB + stage * kBBytes));
#pragma unroll
          for (int kk = 0; kk < kKChunk / 8; ++kk) {
            // advance 8 tf32 (32 bytes) along K inside the swizzled 128-byte row
            mma_tf32(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, kIdesc, (k | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
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
      for (int b = 0; b < 2; ++b)
        if (tcommitted & (1u << b)) mbar_wait_drain(&tfull[b], (tcommit_parity >> b) & 1u, 20000000ull);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;     // tile row = output pixel within the tile
    int local = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      bool got = mbar_wait(&tfull[acc], acc_phase, wd);
      got = __all_sync(0xffffffffu, got);
      if (!got) break;
      tc_fence_after_sync();
      const int m_tile = tile / a.n_tiles, n_tile = tile % a.n_tiles;
      const int m = m_tile * kTileM + row;
      const bool valid = m < a.M;
      int n_img = 0, oh = 0, ow = 0;
      if (valid) {
        n_img = m / a.OHW;
        const int rem = m - n_img * a.OHW;
        oh = rem / a.OW;
        ow = rem - oh * a.OW;
      }
      float* yrow = a.out.y + n_img * a.out.ys_n + oh * a.out.ys_h + ow * a.out.ys_w;
      const float* rrow =
          a.ep.res_mode ? a.ep.r + n_img * a.ep.rs_n + oh * a.ep.rs_h + ow * a.ep.rs_w : nullptr;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
      for (int j0 = 0; j0 < BN; j0 += 16) {
        uint32_t v[16];
        tmem_ld_x16(taddr + j0, v);
        tmem_ld_wait();
        const int c0 = n_tile * BN + j0;
        if (valid) {
          if (a.vec_store && c0 + 16 <= a.Cout) {
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
              const float4 sc = ldg4(a.ep.scale + c0 + j), bi = ldg4(a.ep.bias + c0 + j);
              float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
              if (a.ep.res_mode) r = *reinterpret_cast<const float4*>(rrow + c0 + j);
              const float4 accv = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                              __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
              float4 o = epi_apply4(accv, sc, bi, r, a.ep.act, a.ep.res_mode);
              o = make_float4(round_tf32(o.x), round_tf32(o.y), round_tf32(o.z), round_tf32(o.w));
              *reinterpret_cast<float4*>(yrow + c0 + j) = o;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int c = c0 + j;
              if (c < a.Cout) {
                const float r = a.ep.res_mode ? rrow[c] : 0.0f;
                yrow[c] = round_tf32(epi_apply(__uint_as_float(v[j]), __ldg(a.ep.scale + c), __ldg(a.ep.bias + c), r,
                                               a.ep.act, a.ep.res_mode));
              }
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

int igemm_stages(int bn) {
  const int per = kABytes + bn * kKChunk * 4;
  int s = (200 * 1024) / per;
  if (s > 12) s = 12;
  if (s < 2) s = 2;
  return s;
}

size_t igemm_smem_bytes(int bn, int stages) {
  return 1024 /*alignment slack*/ + static_cast<size_t>(stages) * (kABytes + bn * kKChunk * 4) +
         (2 * stages + 4) * sizeof(uint64_t) + 16;
}

template <int BN>
static cudaError_t launch_bn(const CUtensorMap& amap, const CUtensorMap& bmap, const IgemmArgs& a, int grid,
                             size_t smem, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(igemm_tf32_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  igemm_tf32_kernel<BN><<<grid, kThreads, smem, s>>>(amap, bmap, a);
  return cudaGetLastError();
}

cudaError_t launch_igemm(const CUtensorMap& amap, const CUtensorMap& bmap, const IgemmArgs& a, int bn, int grid,
                         size_t smem, cudaStream_t s) {
  switch (bn) {
    case 16: return launch_bn<16>(amap, bmap, a, grid, smem, s);
    case 32: return launch_bn<32>(amap, bmap, a, grid, smem, s);
    case 48: return launch_bn<48>(amap, bmap, a, grid, smem, s);
    case 64: return launch_bn<64>(amap, bmap, a, grid, smem, s);
    case 96: return launch_bn<96>(amap, bmap, a, grid, smem, s);
    case 128: return launch_bn<128>(amap, bmap, a, grid, smem, s);
    case 192: return launch_bn<192>(amap, bmap, a, grid, smem, s);
    case 256: return launch_bn<256>(amap, bmap, a, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cb
