// The body of a YOLO-style stage with C = 32 channels in one kernel, on the
// tensor cores ("YOLO26N Inference Optimisation": the conv2d_bn_silu layers
// hold most of the GPU time; the stage is the chain's unit).  For the
// stage's stride-2 output x1 (32 channels):
//     a   = act(s1 * conv1x1(x1) + b1)                  32 -> 16
//     b   = act(s2 * conv3x3(a) + b2)                   16 -> 16, pad 1
//     out = act(s3 * conv1x1([a | b]) + b3) + x1        32 -> 32, residual after the activation
// At 3,840 multiply-adds per output pixel the body is a contraction: the
// three convolutions run as tcgen05 MMAs with fp32 accumulators in TMEM, at
// the precision of the library's other tensor-core layers.  fp32 storage:
// kind::tf32 on TF32 operands (weights rounded to the nearest TF32 once; a,
// b and out rounded to the nearest TF32 when formed).  bf16 storage (the same
// kernel, T = bf16): kind::f16 on bf16 operands; a and b stored as bf16 as
// the layers store them, the 3x3's weights bf16 as the bf16 tensor-core
// layer multiplies them, the 1x1 layers' weights split into a bf16 head and
// tail (two MMAs each) so that they act with fp32 accuracy as in the 1x1
// layer kernels.  a and b never leave the SM; the kernel reads x1 once (plus
// its tiles' halos, mostly from L2) and writes out once, where the three
// layer launches move a, b and the concat through HBM and read x1 twice.
//
// Work: tiles of 4 x 32 output pixels (the MMA's M = 128).
//  * One CTA per SM (a kernel that allocates TMEM is placed one per SM)
//    made of independent 128-thread warpgroups (three for fp32, six for
//    bf16), each with its own shared memory, TMEM columns, mbarriers and
//    named barrier, walking its own tiles: while one waits for its MMAs, the
//    others form operands.
//  * x1 over the tile and its 1-pixel halo (6 x 34 pixels x 32 channels)
//    arrives by one TMA copy (zero outside the image), swizzled K-major rows
//    (128 bytes fp32, 64 bf16): the A operand of the 1x1 16 <- 32 over two
//    M = 128 row blocks (rows past the 204 haloed pixels are never used).
//  * a is written three times into shared memory, copy dx holding haloed
//    column c + dx at column c (6 rows x 32 columns each, swizzled rows of 64
//    bytes fp32, 32 bf16).  Tap (dy, dx) of the 3x3 then reads, for output
//    pixel p = 32 r + c, row p + 32 dy of copy dx: a constant offset, so each
//    tap is one descriptor start address and no output column is wasted.
//    Outside the image a is zero (the 3x3's padding, not act(b1)).
//  * b (the 3x3's MMAs) overwrites copy 0, which no MMA reads any more; the
//    last 1x1 reads [a | b] as two K halves: the centre of copy 1 (rows
//    32-159) and b.
//  * out = act(bn(.)) + x1 (x1 from global memory, where its tile was just
//    read: L2; loaded while the 3x3's MMAs run) is staged in shared memory
//    over the copies of a and leaves by one TMA tensor store, which clips the
//    tile at the image's edges.
//  * Two threads of each warpgroup issue and wait (bounded waits); the others
//    wait in the warpgroup's named barrier.  One issues the 3x3's and the
//    last 1x1's MMAs and the output store; the other the x1 copies and the
//    first 1x1's MMAs: it loads the next tile's x1 as soon as this tile's
//    first MMAs have read it, and issues the next tile's 1x1 while this
//    tile's 3x3 runs, so that the next tile starts at its first epilogue.
//  * The epilogues compute every value unconditionally and mask the ones
//    outside the image afterwards: a select around each value made the
//    compiler branch around its exponential, one value after another.
#include "epilogue.cuh"
#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"
#include "tc_store.cuh"

#include <cuda_bf16.h>

namespace cb {

namespace {

constexpr int kTW = 32, kTH = 4;                // output tile
constexpr int kM = kTW * kTH;                   // 128: the MMA's M, a warpgroup's threads
constexpr int kHW = kTW + 2, kHH = kTH + 2;     // the haloed tile
constexpr int kHPx = kHW * kHH;                 // 204 haloed pixels
constexpr int kCopyRows = kHH * kTW;            // 192 rows per copy of a
constexpr int kBarsPerWG = 5;                   // per warpgroup: 3x3 / last 1x1, x1, first 1x1, two drains

// Storage type T: fp32 (kind::tf32 MMAs, K = 8 per instruction) or bf16
// (kind::f16 with bf16 operands, K = 16); either way an MMA consumes 32
// bytes of each K-major row.  Rows: x1 32 channels, a and b 16, out 32.
template <typename T>
struct Cfg;
// bf16: the two 1x1 layers' weights are split into a bf16 head and tail
// (w1 = h + l at kW1 and kW1L, w3 likewise), two MMAs each, so that they act
// with fp32 accuracy as in the fp32-weight layer kernels; the 3x3 multiplies
// bf16 weights like the bf16 tensor-core layers, and a and b are bf16 as in
// the layers' bf16 storage.
template <>
struct Cfg<float> {
  static constexpr int kWG = 3;                              // warpgroups per CTA
  static constexpr int kXRow = 128, kARow = 64, kOutRow = 128;  // bytes; swizzle = row bytes
  static constexpr bool kSplitW = false;
  static constexpr int kW1 = 0, kW1L = 0, kW2 = 2048, kTap = 1024, kW3 = 11264, kW3L = 0, kWBytes = 15360;
  static constexpr int kTmemCols = 256;
};
template <>
struct Cfg<__nv_bfloat16> {
  static constexpr int kWG = 6;  // (4: 52.6 us, 5: 50.3, 6: 48.6 at 160 x 160 batch 32; 80 registers)
  static constexpr int kXRow = 64, kARow = 32, kOutRow = 64;
  static constexpr bool kSplitW = true;
  static constexpr int kW1 = 0, kW1L = 1024, kW2 = 2048, kTap = 512, kW3 = 7168, kW3L = 9216, kWBytes = 11264;
  static constexpr int kTmemCols = 512;
};

template <typename T>
struct Lay {
  using C = Cfg<T>;
  static constexpr int kWG = C::kWG;
  static constexpr int kThreads = kWG * kM;
  static constexpr int kKX = C::kXRow / 32, kKA = C::kARow / 32;  // MMA K steps over an x1 row / an a row
  static constexpr int kXBytes = 2 * kM * C::kXRow;               // the 1x1's two row blocks (rows past 204 never used)
  static constexpr int kCopyBytes = kCopyRows * C::kARow;
  static constexpr int kWGBytes = kXBytes + 3 * kCopyBytes;
  static constexpr int kBar = C::kWBytes + kWG * kWGBytes;
  static constexpr int kSmemEnd = kBar + 8 * kBarsPerWG * kWG + 8;
  static constexpr int kWGCols = 80;                              // D1 (2 x 16), D2 (16), D3 (32)
  static_assert((C::kSplitW ? C::kW3L : C::kW3) + 32 * C::kXRow == C::kWBytes && C::kWBytes <= kStageTcWImgWords * 4,
                "weight image");
  static_assert(kXBytes % 1024 == 0 && kCopyBytes % 1024 == 0 && C::kWBytes % 1024 == 0, "1024-byte swizzle atoms");
  static_assert(2 * kCopyBytes >= kM * C::kOutRow, "the output tile fits over copies 0 and 1");
  static_assert(kWG * kWGCols <= C::kTmemCols, "TMEM split");
};

template <typename T>
constexpr size_t smem_bytes() {
  return 1024 + Lay<T>::kSmemEnd;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier `id` over one warpgroup's 128 threads; the _and form also
// returns whether `v` holds in all of them.
__device__ __forceinline__ void group_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }
__device__ __forceinline__ bool group_sync_and(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id)
      : "memory");
  return r != 0;
}

// Tiled tensor store shared -> global, completing in this thread's bulk
// group; elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The stores committed so far have read their shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// The stores committed so far are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// The nearest TF32 value (ties away from zero, as cvt.rna) of x, by integer
// operations: half a unit of the 10-bit mantissa's last place added to the
// magnitude, the 13 bits below it cleared (infinities stay; a NaN is
// returned as it is, since the addition could carry out of its mantissa).
// Off the conversion pipe, which the epilogues' exponentials and
// reciprocals share.
__device__ __forceinline__ float tf32_rna(float x) {
  return x == x ? __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u) : x;
}

template <int ACT>
__device__ __forceinline__ float act_t(float z) {
  if constexpr (ACT == 1) return fmaxf(z, 0.0f);
  if constexpr (ACT == 2) return silu(z);
  return z;
}

// tcgen05.wait::ld naming both halves of two x16 loads as its operands, so
// that no use of them is scheduled above the wait.
__device__ __forceinline__ void tmem_wait_regs32(uint32_t (&r)[2][16]) {
  tmem_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&r[0][0]));
}

// A row of a or b (16 channels) in the copies' layout: fp32 as a 64-byte row
// of a 64-byte-swizzled operand (16-byte piece q of row r at q ^ (r / 2 % 4)),
// bf16 (nearest even) as a 32-byte row of a 32-byte-swizzled one (q ^ (r / 4 % 2)).
__device__ __forceinline__ void store_arow(uint8_t* base, int r, const float (&v)[16], float) {
  uint8_t* row = base + r * 64;
  const int s = (r >> 1) & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<float4*>(row + ((q ^ s) << 4)) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ void store_arow(uint8_t* base, int r, const float (&v)[16], __nv_bfloat16) {
  uint8_t* row = base + r * 32;
  const int s = (r >> 2) & 1;
#pragma unroll
  for (int q = 0; q < 2; ++q)
    *reinterpret_cast<uint4*>(row + ((q ^ s) << 4)) =
        make_uint4(bf16x2_rn(v[8 * q], v[8 * q + 1]), bf16x2_rn(v[8 * q + 2], v[8 * q + 3]),
                   bf16x2_rn(v[8 * q + 4], v[8 * q + 5]), bf16x2_rn(v[8 * q + 6], v[8 * q + 7]));
}

// The value an operand holds: TF32 (nearest, ties away) for fp32 storage; for
// bf16 storage the rounding happens when the row is stored.
__device__ __forceinline__ float operand_value(float x, float) { return tf32_rna(x); }
__device__ __forceinline__ float operand_value(float x, __nv_bfloat16) { return x; }

// The residual pixel as 16-byte pieces (fp32: 8 of 4 channels, bf16: 4 of 8),
// unpacked in the last epilogue.
template <typename T>
struct Res {
  using V = float4;
  static constexpr int kN = 8;
  __device__ static V zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
};
template <>
struct Res<__nv_bfloat16> {
  using V = uint4;
  static constexpr int kN = 4;
  __device__ static V zero() { return make_uint4(0u, 0u, 0u, 0u); }
};

template <int ACT, typename T>
__global__ void __launch_bounds__(Lay<T>::kThreads, 1)
    stage_body_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap ymap,
                         const __grid_constant__ StageBodyTcArgs a, int tiles_x, int tiles_y) {
  using C = Cfg<T>;
  using L = Lay<T>;
  constexpr int kWG = L::kWG;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* const smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int g = threadIdx.x / kM;  // warpgroup
  const int t = threadIdx.x % kM;  // its thread: output pixel t of the tile, TMEM lane t
  const int warp = threadIdx.x >> 5;
  uint8_t* const xs = smem + C::kWBytes + g * L::kWGBytes;  // haloed x1
  uint8_t* const cp0 = xs + L::kXBytes;                      // copies of a (dx = 0, 1, 2); b over copy 0
  uint64_t* const bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* const mbar = bars + kBarsPerWG * g;  // this warpgroup's 3x3 and last 1x1 completions
  uint64_t* const xfull = mbar + 1;              // its x1 copies
  uint64_t* const d1bar = mbar + 2;              // its first 1x1 completions
  uint64_t* const drain = mbar + 3;              // [2]: the two issuing threads' MMAs, on the way out
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(bars + kBarsPerWG * kWG);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int bar_id = 1 + g;  // named barrier of the warpgroup (0 is __syncthreads)
  // Two threads of the warpgroup issue and wait, from warps that have one
  // haloed pixel per thread in the first epilogue (warps 0-1 have two):
  // the leader (warp 3) the 3x3's and the last 1x1's MMAs and the output
  // store; the x1 thread (warp 2) the x1 copies and the first 1x1's MMAs,
  // which it issues for the next tile while the leader issues this tile's
  // 3x3 and the rest of the warpgroup waits.
  const bool leader = t == 96, xthr = t == 64;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kBarsPerWG * kWG; ++i) mbar_init(&bars[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&xmap);
    tma_prefetch_desc(&ymap);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  // the weights' image (TF32 or bf16, swizzled on the host) from the parameter block
  for (int i = threadIdx.x; i < C::kWBytes / 16; i += L::kThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(a.wimg[4 * i], a.wimg[4 * i + 1], a.wimg[4 * i + 2], a.wimg[4 * i + 3]);
  fence_proxy_async_smem();  // read by the tensor core
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  pdl_launch_dependents();
  pdl_wait();

  const uint32_t tmem = *tmem_slot + static_cast<uint32_t>(g * L::kWGCols);
  const uint32_t tlane = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const Watchdog wd{a.err, abort_flag, a.timeout_ns};
  const uint64_t dx1[2] = {kmajor_swizzled_desc(smem_u32(xs), C::kXRow),
                           kmajor_swizzled_desc(smem_u32(xs + kM * C::kXRow), C::kXRow)};
  const uint64_t dw1 = kmajor_swizzled_desc(smem_u32(smem + C::kW1), C::kXRow);
  const uint64_t dw1l = kmajor_swizzled_desc(smem_u32(smem + C::kW1L), C::kXRow);  // (bf16: the tails)
  const uint64_t dw3l = kmajor_swizzled_desc(smem_u32(smem + C::kW3L), C::kXRow);
  const uint64_t dw2 = kmajor_swizzled_desc(smem_u32(smem + C::kW2), C::kARow);
  const uint64_t dw3 = kmajor_swizzled_desc(smem_u32(smem + C::kW3), C::kXRow);
  const uint64_t dcp = kmajor_swizzled_desc(smem_u32(cp0), C::kARow);
  constexpr uint32_t kCopyStep = L::kCopyBytes >> 4, kDyStep = (kTW * C::kARow) >> 4, kTapStep = C::kTap >> 4;
  constexpr uint32_t id16 = idesc_for<T>(kM, 16), id32 = idesc_for<T>(kM, 32);
  constexpr int kKX = L::kKX, kKA = L::kKA;

  const int num_tiles = a.N * tiles_y * tiles_x;
  const int workers = static_cast<int>(gridDim.x) * kWG;
  const int first = g * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
  auto issue_x = [&](int tile) {  // the x1 thread: tile's haloed x1
    const int tx = tile % tiles_x, rest = tile / tiles_x, ty = rest % tiles_y, n = rest / tiles_y;
    mbar_arrive_expect_tx(xfull, static_cast<uint32_t>(kHPx * C::kXRow));
    tma_load_4d(xs, &xmap, xfull, 0, tx * kTW - 1, ty * kTH - 1, n);
  };
  // bookkeeping of the two issuing threads: copies issued / waited for (x1
  // thread), MMA groups waited for (leader), whether either issued MMAs
  int x_issued = 0, x_done = 0, mma_done = 0, d1_done = 0;
  bool issued_mma = false;
  bool stores = false;  // the leader: a tensor store whose source the next tile overwrites
  auto mma_wait = [&]() {  // the leader: commit the MMAs issued, wait for them
    mma_commit(mbar);
    const bool ok = mbar_wait(mbar, static_cast<uint32_t>(mma_done) & 1u, wd);
    if (ok) ++mma_done;
    return ok;
  };
  // the x1 thread: wait for the x1 of the tile to run next, issue its 1x1
  // into D1, committed to d1bar (the leader waits for it before the epilogue
  // that reads D1)
  auto cv1 = [&]() {
    if (!mbar_wait(xfull, static_cast<uint32_t>(x_done) & 1u, wd)) return false;
    ++x_done;
    tc_fence_after_sync();
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int j = 0; j < kKX; ++j) {
        if constexpr (C::kSplitW) mma_op<T>(tmem + 16 * m, dx1[m] + 2 * j, dw1l + 2 * j, id16, j > 0 ? 1u : 0u);
        mma_op<T>(tmem + 16 * m, dx1[m] + 2 * j, dw1 + 2 * j, id16, (C::kSplitW || j > 0) ? 1u : 0u);
      }
    mma_commit(d1bar);
    issued_mma = true;
    return true;
  };
  bool xok = true;  // the x1 thread: the 1x1 of the tile about to run was issued
  if (xthr && first < num_tiles) {
    if (!a.debug_skip_x) {  // (fault injection: nothing issued, the first wait runs out)
      issue_x(first);
      ++x_issued;
    }
    xok = cv1();
  }

  for (int tile = first; tile < num_tiles; tile += workers) {
    const int tx = tile % tiles_x, rest = tile / tiles_x, ty = rest % tiles_y, n = rest / tiles_y;
    const bool more = tile + workers < num_tiles;
    // ---------------------------------------- a = 1x1 over the haloed tile (issued ahead)
    bool ok = true;
    if (xthr) ok = xok;
    if (leader) {
      ok = mbar_wait(d1bar, static_cast<uint32_t>(d1_done) & 1u, wd);
      if (ok) ++d1_done;
      if (ok && stores) {  // the previous tile's output has left the copies of a
        bulk_wait_read_all();
        stores = false;
      }
    }
    __syncwarp();
    if (!group_sync_and(bar_id, ok)) break;
    if (xthr && more) {  // x1 has been read: the next tile's
      issue_x(tile + workers);
      ++x_issued;
    }
    tc_fence_after_sync();
    {
      uint32_t v2[2][16];  // both row blocks loaded, one wait
      tmem_ld_x16(tmem + tlane, v2[0]);
      tmem_ld_x16(tmem + tlane + 16, v2[1]);
      tmem_wait_regs32(v2);
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const uint32_t (&v)[16] = v2[m];
      const int hp = m * kM + t;
      if (hp < kHPx) {
        const int hy = hp / kHW, hx = hp - hy * kHW;
        const int ih = ty * kTH - 1 + hy, iw = tx * kTW - 1 + hx;
        // outside the image a is +0: every value computed, then masked (a select
        // would branch around each value's exponential and serialise them)
        const uint32_t keep = ih >= 0 && ih < a.H && iw >= 0 && iw < a.W ? 0xFFFFFFFFu : 0u;
        float o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          o[i] = __uint_as_float(
              __float_as_uint(operand_value(act_t<ACT>(fmaf(__uint_as_float(v[i]), a.sb[i], a.sb[16 + i])), T{})) &
              keep);
#pragma unroll
        for (int dx = 0; dx < 3; ++dx) {
          const int c = hx - dx;
          if (c >= 0 && c < kTW) store_arow(cp0 + dx * L::kCopyBytes, hy * kTW + c, o, T{});
        }
      }
    }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    group_sync(bar_id);

    // ---------------------------------------- b = 3x3 over a (nine taps)
    // the residual x1 of this thread's output pixel for the last epilogue (L2:
    // the tile was just read), loaded while the nine taps' MMAs run: the
    // barrier after them waits for the loads too
    const int oh = ty * kTH + t / kTW, ow = tx * kTW + t % kTW;
    const bool in = oh < a.H && ow < a.W;
    using RV = typename Res<T>::V;
    RV r[Res<T>::kN];
    {
      const RV* rp = reinterpret_cast<const RV*>(static_cast<const T*>(a.x) + n * a.xs_n + (in ? oh : 0) * a.xs_h +
                                                 (in ? ow : 0) * a.xs_w);
#pragma unroll
      for (int q = 0; q < Res<T>::kN; ++q) r[q] = in ? rp[q] : Res<T>::zero();
    }
    if (leader) {
      tc_fence_after_sync();
#pragma unroll
      for (int dy = 0; dy < 3; ++dy)
#pragma unroll
        for (int dx = 0; dx < 3; ++dx)
#pragma unroll
          for (int j = 0; j < kKA; ++j)
            mma_op<T>(tmem + 32, dcp + dx * kCopyStep + dy * kDyStep + 2 * j, dw2 + (dy * 3 + dx) * kTapStep + 2 * j,
                      id16, (dy | dx | j) != 0 ? 1u : 0u);
      issued_mma = true;
      ok = mma_wait();
    }
    if (xthr && more) {  // the next tile's 1x1 meanwhile: D1 and the x1 buffer are free
      xok = cv1();
      ok = xok;
    }
    __syncwarp();
    if (!group_sync_and(bar_id, ok)) break;
    tc_fence_after_sync();
    {
      uint32_t v[16];
      tmem_ld_x16(tmem + tlane + 32, v);
      tmem_wait_regs(v);
      float o[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        o[i] = operand_value(act_t<ACT>(fmaf(__uint_as_float(v[i]), a.sb[32 + i], a.sb[48 + i])), T{});
      store_arow(cp0, t, o, T{});  // b over copy 0
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    group_sync(bar_id);

    // ---------------------------------------- out = 1x1 over [a | b]
    if (leader) {
      tc_fence_after_sync();
#pragma unroll
      for (int j = 0; j < kKA; ++j) {  // a: the centre of copy 1 (haloed row hy = r + 1, column c + 1)
        if constexpr (C::kSplitW) mma_op<T>(tmem + 48, dcp + kCopyStep + kDyStep + 2 * j, dw3l + 2 * j, id32, j > 0 ? 1u : 0u);
        mma_op<T>(tmem + 48, dcp + kCopyStep + kDyStep + 2 * j, dw3 + 2 * j, id32, (C::kSplitW || j > 0) ? 1u : 0u);
      }
#pragma unroll
      for (int j = 0; j < kKA; ++j) {  // b
        if constexpr (C::kSplitW) mma_op<T>(tmem + 48, dcp + 2 * j, dw3l + 2 * kKA + 2 * j, id32, 1u);
        mma_op<T>(tmem + 48, dcp + 2 * j, dw3 + 2 * kKA + 2 * j, id32, 1u);
      }
      ok = mma_wait();
    }
    __syncwarp();
    if (!group_sync_and(bar_id, ok)) break;
    tc_fence_after_sync();
    {
      uint32_t v2[2][16];
      tmem_ld_x16(tmem + tlane + 48, v2[0]);
      tmem_ld_x16(tmem + tlane + 64, v2[1]);
      tmem_wait_regs32(v2);
      // the output tile, in the tensor store's box over copies 0 and 1: fp32
      // 128-byte rows with the 128-byte swizzle (piece q of row t at q ^ (t % 8)),
      // bf16 64-byte rows with the 64-byte swizzle (q ^ (t / 2 % 4))
      if constexpr (sizeof(T) == 4) {
        uint8_t* const row = cp0 + t * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) {  // channels 4q .. 4q + 3
          const float rr[4] = {r[q].x, r[q].y, r[q].z, r[q].w};
          float o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = 4 * q + i;
            o[i] = tf32_rna(act_t<ACT>(fmaf(__uint_as_float(v2[q >> 2][c & 15]), a.sb[64 + c], a.sb[96 + c])) + rr[i]);
          }
          *reinterpret_cast<float4*>(row + ((q ^ (t & 7)) << 4)) = make_float4(o[0], o[1], o[2], o[3]);
        }
      } else {
        uint8_t* const row = cp0 + t * 64;
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // channels 8q .. 8q + 7
          const uint32_t w[4] = {r[q].x, r[q].y, r[q].z, r[q].w};
          float o[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c = 8 * q + i;
            const float rr = __uint_as_float((i & 1) ? (w[i >> 1] & 0xFFFF0000u) : (w[i >> 1] << 16));
            o[i] = act_t<ACT>(fmaf(__uint_as_float(v2[c >> 4][c & 15]), a.sb[64 + c], a.sb[96 + c])) + rr;
          }
          *reinterpret_cast<uint4*>(row + ((q ^ ((t >> 1) & 3)) << 4)) =
              make_uint4(bf16x2_rn(o[0], o[1]), bf16x2_rn(o[2], o[3]), bf16x2_rn(o[4], o[5]), bf16x2_rn(o[6], o[7]));
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    group_sync(bar_id);
    if (leader) {
      tma_store_4d(&ymap, cp0, 0, tx * kTW, ty * kTH, n);
      bulk_commit_group();
      stores = true;
    }
  }
  // on the way out (also after a timeout): the copy and the MMA group still
  // in flight land, the stores complete, before the shared memory and TMEM
  // are released
  if (xthr && x_issued > x_done) mbar_wait_drain(xfull, static_cast<uint32_t>(x_done) & 1u, 20000000ull);
  if ((leader || xthr) && issued_mma) {  // a commit with nothing after it: all this thread's MMAs are done
    uint64_t* const d = drain + (leader ? 0 : 1);
    mma_commit(d);
    mbar_wait_drain(d, 0u, 20000000ull);
  }
  if (leader) bulk_wait_all();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(*tmem_slot, C::kTmemCols);
  }
}

template <int ACT, typename T>
cudaError_t launch_t(const CUtensorMap& xmap, const CUtensorMap& ymap, const StageBodyTcArgs& a, int sms,
                     cudaStream_t s) {
  constexpr size_t smem = smem_bytes<T>();
  constexpr int kWG = Lay<T>::kWG;
  cudaError_t e = smem_attr_once<stage_body_tc_kernel<ACT, T>>(smem);
  if (e != cudaSuccess) return e;
  const int tiles_x = (a.W + kTW - 1) / kTW, tiles_y = (a.H + kTH - 1) / kTH;
  const long long tiles = static_cast<long long>(a.N) * tiles_x * tiles_y;
  if (tiles >= (1LL << 31) - static_cast<long long>(sms) * kWG) return cudaErrorInvalidValue;
  const long long ctas = (tiles + kWG - 1) / kWG;
  const unsigned grid = static_cast<unsigned>(ctas < sms ? ctas : sms);
  return launch_pdl(stage_body_tc_kernel<ACT, T>, dim3(grid), dim3(Lay<T>::kThreads), smem, s, xmap, ymap, a, tiles_x,
                    tiles_y);
}

template <typename T>
cudaError_t launch_type(const CUtensorMap& xmap, const CUtensorMap& ymap, const StageBodyTcArgs& a, int sms,
                        cudaStream_t s) {
  if (a.act == 0) return launch_t<0, T>(xmap, ymap, a, sms, s);
  if (a.act == 1) return launch_t<1, T>(xmap, ymap, a, sms, s);
  return launch_t<2, T>(xmap, ymap, a, sms, s);
}

}  // namespace

void stage_body_tc_boxes(int* x_box_w, int* x_box_h, int* y_box_w, int* y_box_h) {
  *x_box_w = kHW;
  *x_box_h = kHH;
  *y_box_w = kTW;
  *y_box_h = kTH;
}

cudaError_t launch_stage_body_tc(const CUtensorMap& xmap, const CUtensorMap& ymap, const StageBodyTcArgs& a, int sms,
                                 cudaStream_t s) {
  if (a.N == 0 || a.H == 0 || a.W == 0) return cudaSuccess;
  return a.bf16 ? launch_type<__nv_bfloat16>(xmap, ymap, a, sms, s) : launch_type<float>(xmap, ymap, a, sms, s);
}

}  // namespace cb
