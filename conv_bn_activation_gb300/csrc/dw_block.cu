// One DepthwiseSeparableConv block in one kernel ("How I sped up
// convolutions": the block listing; the fusion the article's summary points
// to): depthwise 3x3 + BN + ReLU, pointwise 1x1 + BN, the skip (identity, or
// 1x1 conv + BN) and the final ReLU, with the depthwise output never leaving
// the SM.
//
// GEMM view: for 128 output pixels (the MMA's M) the block output is
//     y = relu(s2 * (T * Wpwᵀ) + b2 + skip),
//     T = relu(s1 * dw3x3(x) + b1)                          [128 x Ci]
//     skip = x                                              (identity)
//          = s_sk * (Xs * Wskᵀ) + b_sk                       (1x1 conv, stride s)
// where Xs holds the block input at the strided output positions.  K walks
// 32-channel chunks: first the chunks of T into TMEM accumulator 0, then (a
// conv skip) the chunks of Xs into accumulator 1.
//  * warps 2-9 (256 threads) build each A chunk [128 pixels x 32 channels] in
//    shared memory, in the 128-byte swizzled K-major layout the tensor core
//    reads (the 16-byte group g of row r at position g ^ (r % 8)): the
//    depthwise taps on CUDA cores from the block input (L2-resident at these
//    sizes), BN and ReLU applied, rounded to TF32; or the strided input
//    pixels for the skip.  A proxy fence makes the stores visible to the
//    tensor core, then they arrive on the chunk's barrier;
//  * warp 0 lane 0 loads the matching B chunk [Co x 32] of the pointwise or
//    skip weights with TMA;
//  * warp 1 lane 0 issues the four K = 8 MMAs per chunk (M = 128, N = Co)
//    and commits each stage back to both producers;
//  * then warps 2-9 read the accumulators (two warps per TMEM lane quarter,
//    half the channels each) and write the block output: scale/bias, the
//    skip, ReLU, rounded to TF32 like every tensor-core layer's output.
// Two stages of A and B let the builders fill one chunk while the MMAs read
// the other.  One tile per CTA (the blocks have at most a few hundred tiles).
// Every wait is bounded; a timeout is reported through the device error word.
#include "epilogue.cuh"
#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"
#include "tc_store.cuh"
#include "trace.cuh"

namespace cb {

namespace {

constexpr int kThreads = 320;
constexpr int kWorkers = 256;
constexpr int kABytes = 128 * 128;  // 128 rows x 32 fp32

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float4 tf32x4(float4 v) {
  return make_float4(round_tf32(v.x), round_tf32(v.y), round_tf32(v.z), round_tf32(v.w));
}

__global__ void __launch_bounds__(kThreads, 1) dw_block_kernel(const __grid_constant__ CUtensorMap pw_map,
                                                               const __grid_constant__ CUtensorMap sk_map,
                                                               const DwBlockArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int Ci = a.Ci, Co = a.Co;
  const int b_bytes = Co * 128;
  uint8_t* sA = smem;                    // 2 x 16 KB
  uint8_t* sB = sA + 2 * kABytes;        // 2 x Co x 128 B
  float* sW = reinterpret_cast<float*>(sB + 2 * b_bytes);  // depthwise weights [9][Ci]
  float* s1 = sW + 9 * Ci;               // depthwise scale / bias [Ci]
  float* b1 = s1 + Ci;
  float* s2 = b1 + Ci;                   // pointwise scale / bias [Co]
  float* b2 = s2 + Co;
  float* ssk = b2 + Co;                  // skip scale / bias [Co]
  float* bsk = ssk + Co;
  uint64_t* bars = reinterpret_cast<uint64_t*>(bsk + Co + ((11 * Ci + 4 * Co) & 1));  // 8-byte aligned
  uint64_t* a_full = bars;               // [2], 256 builder arrivals
  uint64_t* b_full = bars + 2;           // [2], TMA bytes
  uint64_t* empty = bars + 4;            // [2], MMA commit
  uint64_t* tfull = bars + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 7);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&a_full[s], kWorkers);
      mbar_init(&b_full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  const uint32_t tmem_cols = a.tmem_cols;
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  pdl_launch_dependents();
  pdl_wait();
  // parameters into shared memory (after the previous kernel's writes are visible)
  for (int i = threadIdx.x; i < 9 * Ci; i += kThreads) sW[i] = __ldg(a.dw_w + i);
  for (int i = threadIdx.x; i < Ci; i += kThreads) {
    s1[i] = __ldg(a.dw_scale + i);
    b1[i] = __ldg(a.dw_bias + i);
  }
  for (int i = threadIdx.x; i < Co; i += kThreads) {
    s2[i] = __ldg(a.pw_scale + i);
    b2[i] = __ldg(a.pw_bias + i);
    ssk[i] = a.skip_conv ? __ldg(a.sk_scale + i) : 0.0f;
    bsk[i] = a.skip_conv ? __ldg(a.sk_bias + i) : 0.0f;
  }
  __syncthreads();
  const uint32_t tmem_base = *tmem_slot;
  const Watchdog wd{a.err, abort_flag, a.timeout_ns};
  const int steps = a.num_kc * (a.skip_conv ? 2 : 1);
  const int m0 = blockIdx.x * 128;
  const bool tr_cta = a.trace && static_cast<int>(blockIdx.x) == a.trace_cta;
  TraceBuf tr;
  tr.add(tr_cta && (threadIdx.x == 0 || threadIdx.x == 32 || threadIdx.x == 64));

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&pw_map);
      if (a.skip_conv) tma_prefetch_desc(&sk_map);
      uint32_t issued = 0, last_parity = 0;
      for (int step = 0; step < steps; ++step) {
        const int s = step & 1, round = step >> 1;
        if (round > 0 && !mbar_wait(&empty[s], static_cast<uint32_t>(round - 1) & 1u, wd)) break;
        mbar_arrive_expect_tx(&b_full[s], static_cast<uint32_t>(b_bytes));
        const bool pw = step < a.num_kc;
        const int kc = pw ? step : step - a.num_kc;
        tma_load_3d(sB + s * b_bytes, pw ? &pw_map : &sk_map, &b_full[s], kc * 32, 0, 0);
        tr.add(tr_cta);
        issued |= 1u << s;
        last_parity = (last_parity & ~(1u << s)) | ((static_cast<uint32_t>(round) & 1u) << s);
      }
      for (int s = 0; s < 2; ++s)
        if (issued & (1u << s)) mbar_wait_drain(&b_full[s], (last_parity >> s) & 1u, 20000000ull);
      tr.flush(tr_cta, 0);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_tf32(128, Co);
      uint32_t committed = 0, parity = 0;
      bool ok = true;
      for (int step = 0; step < steps; ++step) {
        const int s = step & 1, round = step >> 1;
        const uint32_t ph = static_cast<uint32_t>(round) & 1u;
        const bool got_a = mbar_wait(&a_full[s], ph, wd);
        tr.add(tr_cta);
        if (!got_a || !mbar_wait(&b_full[s], ph, wd)) {
          ok = false;
          break;
        }
        tr.add(tr_cta);
        tc_fence_after_sync();
        const bool pw = step < a.num_kc;
        const uint32_t d = tmem_base + (pw ? 0u : static_cast<uint32_t>(Co));
        const bool first = step == 0 || step == a.num_kc;
        const uint64_t adesc = kmajor_swizzled_desc(smem_u32(sA + s * kABytes), 128);
        const uint64_t bdesc = kmajor_swizzled_desc(smem_u32(sB + s * b_bytes), 128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_tf32(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, (!first || kk) ? 1u : 0u);
        mma_commit(&empty[s]);
        const uint32_t bit = 1u << s;
        parity = (committed & bit) ? (parity ^ bit) : (parity & ~bit);
        committed |= bit;
      }
      if (ok) mma_commit(tfull);
      tr.flush(tr_cta, 1);
      // let every MMA finish before TMEM is released
      for (int s = 0; s < 2; ++s)
        if (committed & (1u << s)) mbar_wait_drain(&empty[s], (parity >> s) & 1u, 20000000ull);
    }
  } else {
    // ------------------------------------------------- A builders, epilogue
    const int wt = threadIdx.x - 64;
    // This thread's items: rows wt / 8 + 32 k (k = 0..3) of the tile, channel quad wt % 8.
    const int qd = wt & 7;
    bool ok = true;
    for (int step = 0; step < steps; ++step) {
      const int s = step & 1, round = step >> 1;
      if (round > 0) {
        bool w = mbar_wait(&empty[s], static_cast<uint32_t>(round - 1) & 1u, wd);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
      }
      tr.add(tr_cta && threadIdx.x == 64);
      const bool dw = step < a.num_kc;
      const int c = (dw ? step : step - a.num_kc) * 32 + qd * 4;
      uint8_t* dst = sA + s * kABytes;
      // One item at a time (not unrolled: registers), its nine input loads
      // issued before any is used (out-of-image taps load the tensor's first
      // pixel and are masked).
#pragma unroll 1
      for (int k = 0; k < 4; ++k) {
        const int r = (wt >> 3) + 32 * k;
        const int m = m0 + r;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m < a.M && c < Ci) {
          const int n = m / (a.OH * a.OW), rem = m - n * (a.OH * a.OW);
          const int oh = rem / a.OW, ow = rem - (rem / a.OW) * a.OW;
          const float* xn = a.x + n * a.xs_n;
          if (dw) {
            const int ih0 = oh * a.stride - 1, iw0 = ow * a.stride - 1;
            float4 xv[9];
            bool in[9];
#pragma unroll
            for (int t = 0; t < 9; ++t) {
              const int ih = ih0 + t / 3, iw = iw0 + t % 3;
              in[t] = ih >= 0 && ih < a.H && iw >= 0 && iw < a.W;
              const float* src = in[t] ? xn + ih * a.xs_h + static_cast<long long>(iw) * a.xs_w + c : a.x;
              xv[t] = __ldg(reinterpret_cast<const float4*>(src));
            }
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int t = 0; t < 9; ++t) {
              if (!in[t]) continue;
              const float4 wv = *reinterpret_cast<const float4*>(sW + t * Ci + c);
              acc.x = fmaf(xv[t].x, wv.x, acc.x);
              acc.y = fmaf(xv[t].y, wv.y, acc.y);
              acc.z = fmaf(xv[t].z, wv.z, acc.z);
              acc.w = fmaf(xv[t].w, wv.w, acc.w);
            }
            const float4 sc = *reinterpret_cast<const float4*>(s1 + c), bi = *reinterpret_cast<const float4*>(b1 + c);
            v = make_float4(fmaxf(fmaf(acc.x, sc.x, bi.x), 0.f), fmaxf(fmaf(acc.y, sc.y, bi.y), 0.f),
                            fmaxf(fmaf(acc.z, sc.z, bi.z), 0.f), fmaxf(fmaf(acc.w, sc.w, bi.w), 0.f));
          } else {
            v = __ldg(reinterpret_cast<const float4*>(xn + oh * a.stride * a.xs_h +
                                                      static_cast<long long>(ow * a.stride) * a.xs_w + c));
          }
          v = tf32x4(v);
        }
        *reinterpret_cast<float4*>(dst + r * 128 + ((qd ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();  // the tensor core reads these stores through the async proxy
      mbar_arrive(&a_full[s]);
      tr.add(tr_cta && threadIdx.x == 64);
    }

    // --------------------------------------------------------- epilogue
    bool got = ok && mbar_wait(tfull, 0, wd);
    got = __all_sync(0xffffffffu, got);
    tr.add(tr_cta && threadIdx.x == 64);
    if (got) {
      tc_fence_after_sync();
      const int q = warp & 3, group = (warp - 2) >> 2;
      const int row = q * 32 + lane;
      const int m = m0 + row;
      const bool valid = m < a.M;
      const int mm = valid ? m : 0;
      const int n = mm / (a.OH * a.OW), rem = mm - n * (a.OH * a.OW);
      const int oh = rem / a.OW, ow = rem - (rem / a.OW) * a.OW;
      float* yp = a.out.y + n * a.out.ys_n + oh * a.out.ys_h + static_cast<long long>(ow) * a.out.ys_w;
      // identity skip: stride 1, the input pixel at the output position
      const float* xp = a.x + n * a.xs_n + oh * a.xs_h + static_cast<long long>(ow) * a.xs_w;
      const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int half = Co / 2;
      // 16-column chunks; a chunk's residual loads (identity skip) are issued
      // before its TMEM loads are waited for.
#pragma unroll 1
      for (int col = group * half; col < (group + 1) * half; col += 16) {
        uint32_t v1[16], v2[16];
        float4 rx[4];
        tmem_ld_cols<16>(lane_base + col, v1);
        if (a.skip_conv) tmem_ld_cols<16>(lane_base + Co + col, v2);
        if (!a.skip_conv) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            rx[j] = valid ? __ldg(reinterpret_cast<const float4*>(xp + col + 4 * j)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        tmem_wait_regs(v1);
        if (a.skip_conv) tmem_wait_regs(v2);
        if (valid) {
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            const int cc = col + j;
            const float4 sc = *reinterpret_cast<const float4*>(s2 + cc), bi = *reinterpret_cast<const float4*>(b2 + cc);
            float4 r;
            if (a.skip_conv) {
              const float4 ss = *reinterpret_cast<const float4*>(ssk + cc),
                           sb = *reinterpret_cast<const float4*>(bsk + cc);
              r = make_float4(fmaf(__uint_as_float(v2[j]), ss.x, sb.x), fmaf(__uint_as_float(v2[j + 1]), ss.y, sb.y),
                              fmaf(__uint_as_float(v2[j + 2]), ss.z, sb.z),
                              fmaf(__uint_as_float(v2[j + 3]), ss.w, sb.w));
            } else {
              r = rx[j / 4];
            }
            const float4 o = make_float4(
                round_tf32(fmaxf(fmaf(__uint_as_float(v1[j]), sc.x, bi.x) + r.x, 0.f)),
                round_tf32(fmaxf(fmaf(__uint_as_float(v1[j + 1]), sc.y, bi.y) + r.y, 0.f)),
                round_tf32(fmaxf(fmaf(__uint_as_float(v1[j + 2]), sc.z, bi.z) + r.z, 0.f)),
                round_tf32(fmaxf(fmaf(__uint_as_float(v1[j + 3]), sc.w, bi.w) + r.w, 0.f)));
            *reinterpret_cast<float4*>(yp + cc) = o;
          }
        }
      }
    }
  }

  if (warp >= 2) {
    tr.add(tr_cta && threadIdx.x == 64);
    tr.flush(tr_cta && threadIdx.x == 64, 2);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

}  // namespace

int dw_block_read_trace(unsigned long long* out, int max_records) { return igemm_read_trace_tu(out, max_records); }

size_t dw_block_smem_bytes(int ci, int co) {
  return 1024 + 2 * static_cast<size_t>(kABytes) + 2 * static_cast<size_t>(co) * 128 +
         (11 * static_cast<size_t>(ci) + 4 * co + 1) * sizeof(float) + 8 * sizeof(uint64_t) + 16;
}

cudaError_t launch_dw_block(const CUtensorMap& pw_map, const CUtensorMap& sk_map, const DwBlockArgs& a,
                            cudaStream_t s) {
  if (a.M == 0) return cudaSuccess;
  const size_t smem = dw_block_smem_bytes(a.Ci, a.Co);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  const cudaError_t e = smem_attr_once<dw_block_kernel>(227 * 1024);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>((a.M + 127) / 128);
  return launch_pdl(dw_block_kernel, dim3(grid), dim3(kThreads), smem, s, pw_map, sk_map, a);
}

}  // namespace cb
