// Stem convolution 3 -> 16 channels, 3x3, stride 2, pad 1, with the folded-BN
// / activation (/ residual) epilogue, on the tensor cores at fp32 accuracy,
// for packed NHWC input (fp32, or bf16 storage).
//
// GEMM view ("YOLO26N Inference Optimisation": the 640x640x3 stem, the
// conv2d_bn_silu layer): 128 output pixels (M) x 16 output channels (N) x
// 27 products (K = kh, kw, ci, padded to 32).  The layer is bound by HBM
// (the input read once, the 16-channel output written once); what the
// tensor core takes over is the 432 FMAs per pixel that kept the CUDA-core
// stem's issue slots busy.
//
// fp32 accuracy from TF32 operands (the split-operand scheme of Markidis et
// al. 2018 and Ootomo & Yokota 2022): each fp32 value v is split into a TF32
// head and tail, v = h + l; the products of two TF32 values are exact in the
// fp32 accumulator, and a_h*w_h + a_l*w_h + a_h*w_l misses a*w only by the
// dropped a_l*w_l and what the tails lose.  Weights: h = tf32(w) (nearest),
// l = tf32(w - h), so |w - h - l| <= 2^-22 |w|.  Activations (per pixel, so
// kept cheap): the MMA reads an fp32 operand as TF32 by ignoring its low 13
// bits, so h is v itself (read as v truncated to TF32) and l = v - trunc(v)
// (exact; one mask, one subtraction), which the MMA truncates in turn:
// |v - h - l| < 2^-20 |v|.  Each product is then within about 2^-20 |a w|.
// bf16 inputs are TF32 values already (a_l = 0).  The result is held to the
// fp32 CUDA-core bar, not the TF32 one.
//
// Layout of the work:
//  * one persistent CTA per SM (a kernel that allocates TMEM is placed one
//    CTA per SM), made of independent 128-thread warpgroups (6 for fp32, 8
//    for bf16), each with its own staging ring, TMEM columns and mbarrier,
//    synchronised by its own named barrier: while one warpgroup waits for
//    its MMAs or its copies, the others build or store;
//  * a warpgroup walks tiles of 2 output rows x 64 columns; a tile's input
//    (5 rows x 132 pixels, from input column 2*ow0 - 4; bf16: 136 pixels
//    from 2*ow0 - 8, so that copies start on 16-byte boundaries) is staged
//    raw into a ring of kStages buffers, kStages - 1 tiles ahead of the one
//    computed: one bulk copy (cp.async.bulk) per input row for the part
//    inside the image, completing on the slot's mbarrier, and zeros (the
//    padding) stored by the warpgroup's first warp outside it;
//  * thread t of a warpgroup gathers the A row of its output pixel (three
//    runs of 9 consecutive staged values, one per filter row: 3 columns x 3
//    channels), splits it into head and tail in registers and stores both
//    into TMEM (tcgen05.st, lane t, 32 columns each): the MMAs read A from
//    TMEM, so A costs no shared-memory bandwidth;
//  * B is w_h (rows 0-15) and w_l (rows 16-31), 128-byte swizzled K-major
//    rows in shared memory, built once per CTA; the warpgroup's thread 0
//    issues, per tile, A_l x w_h, A_h x w_l and A_h x w_h (four MMAs each,
//    M = 128, N = 16, K = 8; the small terms first) into one 16-column
//    accumulator D, committed to the warpgroup's mbarrier; thread 0 alone
//    waits for that commit and for the next tile's rows (bounded waits),
//    while the others sleep in the warpgroup's named barrier: two barriers
//    per tile, tile coordinates walked by additions;
//  * each warp reads its 32 TMEM lanes of D (thread t: pixel t), applies
//    scale / bias / residual / activation and writes the pixel's 64 bytes
//    (bf16: 32).
#include "epilogue.cuh"
#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"
#include "tc_store.cuh"

#include <cuda_bf16.h>

namespace cb {

namespace {

constexpr int kTH = 2;               // output rows per tile
constexpr int kTW = 64;              // output columns per tile
constexpr int kM = kTH * kTW;        // 128 output pixels: the MMA's M
constexpr int kWGThreads = kM;       // a warpgroup; its thread t: A row t, TMEM lane t
constexpr int kRows = 2 * kTH + 1;   // staged input rows
constexpr int kStages = 4;           // staged tiles per warpgroup
constexpr int kBRow = 128;           // bytes per B row (32 TF32 K entries)
constexpr int kBBytes = 32 * kBRow;  // B = w_h (rows 0-15), w_l (rows 16-31)
constexpr int kTmemCols = 512;       // allocated whole (one CTA per SM); kWG x kWGCols of it used

// Staging of one input row: groups of pixels that make 48 bytes (three
// 16-byte copies), starting kFirst pixels left of input column 2 * ow0.
// TMEM columns of a warpgroup: A head at 0, A tail at 32 (fp32), D after A.
template <typename T>
struct Staging;
template <>
struct Staging<float> {
  static constexpr int kFirst = 4, kGroupPx = 4, kGroups = 33;  // 132 pixels
  static constexpr bool kSplit = true;                           // head and tail A operands
  static constexpr int kWG = 6;                                  // warpgroups per CTA
  static constexpr int kWGCols = 80, kDCol = 64;                 // A 0-63, D 64-79
};
template <>
struct Staging<__nv_bfloat16> {
  static constexpr int kFirst = 8, kGroupPx = 8, kGroups = 17;  // 136 pixels
  static constexpr bool kSplit = false;                          // bf16 values are TF32 values
  static constexpr int kWG = 8;
  static constexpr int kWGCols = 48, kDCol = 32;                 // A 0-31, D 32-47
};

// Shared memory: B, the warpgroups' staging rings, scale / bias, the
// warpgroups' mbarriers (MMA completion, staged slots), the TMEM slot and the
// abort flag.
template <typename T>
struct Layout {
  static constexpr int kWG = Staging<T>::kWG;
  static constexpr int kRowBytes = Staging<T>::kGroups * 48;  // staged bytes per input row
  static constexpr int kRawBytes = kRows * kRowBytes;         // one staged tile
  static constexpr int kB = 0;
  static constexpr int kRaw = kB + kBBytes;
  static constexpr int kSB = kRaw + kWG * kStages * kRawBytes;
  static constexpr int kBar = kSB + 32 * 4;             // MMA barriers [kWG], staging barriers [kWG][kStages]
  static constexpr int kEnd = kBar + 8 * kWG * (1 + kStages) + 8;
  static_assert(kRaw % 16 == 0 && kRawBytes % 16 == 0 && kBar % 8 == 0, "alignment");
  static_assert(kWG * Staging<T>::kWGCols <= kTmemCols, "TMEM split");
};

template <typename T>
constexpr size_t smem_bytes() {
  return 1024 + Layout<T>::kEnd;  // + alignment of the base to the 1024-byte swizzle atom
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global to shared memory, completing as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier `id` over the 128 threads of one warpgroup; the _and form
// also returns whether `v` holds in all of them.
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

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::tf32, one CTA: A (M x K) read from
// tensor memory, lane = row, one 32-bit column per K entry.
__device__ __forceinline__ void mma_tf32_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 bits, 32 consecutive columns per thread, registers -> TMEM.
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  __syncwarp();
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  __syncwarp();
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// The nearest TF32 value to x (ties away from zero), as fp32 bits: half a
// unit of the 10-bit mantissa's last place added to the magnitude, the 13
// bits below it cleared (finite x below the largest TF32 value).  Integer
// operations only, off the conversion pipe.
__device__ __forceinline__ uint32_t tf32_bits(float x) { return (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u; }

// x minus x truncated to TF32 (the low 13 mantissa bits cleared): exact.
__device__ __forceinline__ uint32_t tf32_tail_bits(float x) {
  return __float_as_uint(x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u));
}

struct Tile {
  int n, oh0, ow0;
};

// The tiles first, first + step, first + 2 step, ... (tile index
// ((n * tiles_y) + ty) * tiles_x + tx) walked without divisions: the step's
// own quotient and remainders are taken once, each advance adds them with
// carries.
struct TileWalk {
  int tx, ty, n, dtx, dty, dn;
  __device__ __forceinline__ void init(int first, int step, int tiles_x, int tiles_y) {
    tx = first % tiles_x;
    const int r = first / tiles_x;
    ty = r % tiles_y;
    n = r / tiles_y;
    dtx = step % tiles_x;
    const int dr = step / tiles_x;
    dty = dr % tiles_y;
    dn = dr / tiles_y;
  }
  __device__ __forceinline__ Tile tile() const { return Tile{n, ty * kTH, tx * kTW}; }
  __device__ __forceinline__ void next(int tiles_x, int tiles_y) {
    tx += dtx;
    int c = tx >= tiles_x ? 1 : 0;
    tx -= c * tiles_x;
    ty += dty + c;
    c = ty >= tiles_y ? 1 : 0;
    ty -= c * tiles_y;
    n += dn + c;
  }
};

// Stages one tile's input rows into `raw` (run by one whole warp): lane 0
// arms `full` with the byte count and issues one bulk copy per input row
// for the columns inside the image; the lanes store zeros everywhere else
// (rows above or below the image, columns left or right of it).  Staged
// pixel c holds input column c0 + c; the in-image span [lo, hi) starts and
// ends on whole 48-byte pixel groups (W is a multiple of the group).
template <typename T>
__device__ __forceinline__ void stage_tile(const StemArgs& a, const Tile& p, uint8_t* raw, uint64_t* full, int lane) {
  using S = Staging<T>;
  constexpr int kPx = S::kGroups * S::kGroupPx;  // staged pixels per row
  constexpr int kPxBytes = 3 * sizeof(T);
  constexpr int kUnits = Layout<T>::kRowBytes / 16;
  const int c0 = 2 * p.ow0 - S::kFirst;  // input column of staged pixel 0
  const int ih0 = 2 * p.oh0 - 1;
  const int lo = max(c0, 0), hi = min(c0 + kPx, a.W);
  const uint32_t off = static_cast<uint32_t>((lo - c0) * kPxBytes), span = static_cast<uint32_t>((hi - lo) * kPxBytes);
  const int r_lo = max(-ih0, 0), r_hi = min(a.H - ih0, kRows);  // staged rows inside the image
  if (lane == 0) {
    mbar_arrive_expect_tx(full, span * static_cast<uint32_t>(r_hi - r_lo));
    const T* src = static_cast<const T*>(a.src) + p.n * a.xs_n + 3LL * lo;
    for (int r = r_lo; r < r_hi; ++r) bulk_g2s(raw + r * Layout<T>::kRowBytes + off, src + (ih0 + r) * a.xs_h, span, full);
  }
  if (r_lo > 0 || r_hi < kRows || off > 0 || off + span < static_cast<uint32_t>(Layout<T>::kRowBytes)) {
    for (int i = lane; i < kRows * kUnits; i += 32) {
      const int r = i / kUnits;
      const uint32_t b = static_cast<uint32_t>(i - r * kUnits) * 16;
      if (r < r_lo || r >= r_hi || b < off || b >= off + span)
        *reinterpret_cast<uint4*>(raw + r * Layout<T>::kRowBytes + b) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  __syncwarp();
}

// The 10 staged values of one input row from which this thread's pixel
// takes its 9 (columns 2*ow - 1 .. 2*ow + 1, channels 0..2): v[1..9].
__device__ __forceinline__ void row_values(const uint8_t* row, int lx, float (&v)[10], float) {
  const float2* p = reinterpret_cast<const float2*>(row + 4 * (6 * lx + 8));
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    const float2 f = p[i];
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void row_values(const uint8_t* row, int lx, float (&v)[10], __nv_bfloat16) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(row + 2 * (6 * lx + 20));
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    const uint32_t u = p[i];
    v[2 * i] = __uint_as_float(u << 16);
    v[2 * i + 1] = __uint_as_float(u & 0xFFFF0000u);
  }
}

template <typename T, int ACT, bool RES>
__global__ void __launch_bounds__(Staging<T>::kWG * kWGThreads, 1) stem_tc_kernel(const StemArgs a) {
  using S = Staging<T>;
  using L = Layout<T>;
  constexpr int kWG = L::kWG;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int g = threadIdx.x / kWGThreads;  // warpgroup
  const int t = threadIdx.x % kWGThreads;  // its thread: A row t, TMEM lane t
  const int warp = threadIdx.x >> 5;
  uint8_t* const sB = smem + L::kB;
  uint8_t* const ring = smem + L::kRaw + g * kStages * L::kRawBytes;
  float* const sc = reinterpret_cast<float*>(smem + L::kSB);
  float* const bi = sc + 16;
  uint64_t* const bars = reinterpret_cast<uint64_t*>(smem + L::kBar);  // [kWG]
  uint64_t* const full = bars + kWG + g * kStages;                      // this warpgroup's [kStages]
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(bars + kWG * (1 + kStages));
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* const bar = bars + g;
  const int bar_id = 1 + g;  // named barrier of the warpgroup (0 is __syncthreads)

  if (threadIdx.x == 0) {
    for (int i = 0; i < kWG * (1 + kStages); ++i) mbar_init(&bars[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  pdl_launch_dependents();
  pdl_wait();
  // B: rows 0-15 the heads, rows 16-31 the tails of the weights OHWI
  // [16][27], K = (kh * 3 + kw) * 3 + ci (the A row order); 128-byte
  // swizzled K-major rows (16-byte group q of row r at q ^ (r % 8));
  // thread i < 256: row i / 8, group i % 8
  if (threadIdx.x < 256) {
    const int row = threadIdx.x >> 3, q = threadIdx.x & 7, co = row & 15;
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = 4 * q + i;
      const float w = k < 27 ? __ldg(a.w + co * 27 + k) : 0.0f;
      const uint32_t h = tf32_bits(w);
      u[i] = row < 16 ? h : tf32_bits(w - __uint_as_float(h));
    }
    *reinterpret_cast<uint4*>(sB + row * kBRow + ((q ^ (row & 7)) << 4)) = make_uint4(u[0], u[1], u[2], u[3]);
  }
  if (threadIdx.x < 16) {
    sc[threadIdx.x] = __ldg(a.ep.scale + threadIdx.x);
    bi[threadIdx.x] = __ldg(a.ep.bias + threadIdx.x);
  }
  fence_proxy_async_smem();  // B is read by the tensor core
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t tcol = tmem_base + static_cast<uint32_t>(g * S::kWGCols);     // this warpgroup's columns
  const uint32_t tlane = static_cast<uint32_t>((warp & 3) * 32) << 16;         // this warp's lanes
  const Watchdog wd{a.err, abort_flag, a.timeout_ns};
  const uint64_t b_desc = kmajor_swizzled_desc(smem_u32(sB), kBRow);

  const int ly = t / kTW, lx = t % kTW;
  const int num_tiles = a.N * a.tiles_y * a.tiles_x;
  const int workers = static_cast<int>(gridDim.x) * kWG;
  const int first = g * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
  bool pending = false;    // thread 0: an MMA group whose completion nobody has seen
  int it = 0, staged = 0;  // tiles consumed / staged by this warpgroup (its tile q sits in slot q % kStages)
  const bool stager = t < 32;  // the warpgroup's first warp stages
  TileWalk cur, ahead;
  cur.init(first, workers, a.tiles_x, a.tiles_y);
  ahead = cur;
  for (; staged < kStages - 1 && first + staged * workers < num_tiles; ++staged) {
    if (stager) stage_tile<T>(a, ahead.tile(), ring + staged * L::kRawBytes, &full[staged], t);
    ahead.next(a.tiles_x, a.tiles_y);
  }
  // Two named barriers per tile: after A is in TMEM (then thread 0 issues the
  // MMAs), and after thread 0 has seen the MMAs complete and the next tile's
  // rows arrive (its waits; the others sleep in the barrier, which also
  // carries thread 0's wait result).
  bool in = true;
  if (t == 0 && first < num_tiles) in = mbar_wait(&full[0], 0u, wd);
  __syncwarp();  // warp 0 converged again before the aligned barrier
  bool ok = group_sync_and(bar_id, in);
  for (int tile = first; ok && tile < num_tiles; tile += workers, ++it) {
    const Tile p = cur.tile();
    cur.next(a.tiles_x, a.tiles_y);
    // the slot kStages - 1 tiles ahead was last read by the previous tile's
    // A gather, which every thread of the warpgroup finished before that
    // tile's MMA barrier
    if (first + staged * workers < num_tiles) {
      const int q = staged % kStages;
      if (stager) stage_tile<T>(a, ahead.tile(), ring + q * L::kRawBytes, &full[q], t);
      ahead.next(a.tiles_x, a.tiles_y);
      ++staged;
    }

    // ------------------------------------------------ A row t into TMEM
    {
      const uint8_t* raw = ring + (it % kStages) * L::kRawBytes;
      float v[3][10];
#pragma unroll
      for (int kh = 0; kh < 3; ++kh) row_values(raw + (2 * ly + kh) * L::kRowBytes, lx, v[kh], T{});
      // K entry k = kh * 9 + j is v[kh][1 + j]; entries 27..31 are zero
      uint32_t h[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) h[k] = k < 27 ? __float_as_uint(v[k / 9][1 + k % 9]) : 0u;
      tmem_st_x32(tcol + tlane, h);
      if constexpr (S::kSplit) {
        uint32_t l[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) l[k] = k < 27 ? tf32_tail_bits(v[k / 9][1 + k % 9]) : 0u;
        tmem_st_x32(tcol + tlane + 32, l);
      }
      tmem_st_wait();
    }
    tc_fence_before_sync();  // the TMEM stores (and the previous tile's TMEM loads) are done
    group_sync(bar_id);

    // ------------------------------------------ MMAs, and the wait for them
    bool got = true;
    if (t == 0) {
      tc_fence_after_sync();
      const uint32_t d = tcol + S::kDCol;
      constexpr uint32_t idesc = idesc_tf32(kM, 16);
      const uint64_t b_tail = b_desc + ((16 * kBRow) >> 4);  // rows 16-31 (whole swizzle atoms)
      uint32_t accumulate = 0;
      if constexpr (S::kSplit) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk, accumulate = 1)
          mma_tf32_tmem_a(d, tcol + 32 + 8 * kk, b_desc + 2 * kk, idesc, accumulate);
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk, accumulate = 1) mma_tf32_tmem_a(d, tcol + 8 * kk, b_tail + 2 * kk, idesc, accumulate);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) mma_tf32_tmem_a(d, tcol + 8 * kk, b_desc + 2 * kk, idesc, 1u);
      mma_commit(bar);
      pending = true;
      got = mbar_wait(bar, static_cast<uint32_t>(it) & 1u, wd);
      // the next tile's rows: the bulk copies (its slot's barrier) and the
      // zeros (stored before an earlier barrier of the warpgroup)
      if (got && tile + workers < num_tiles)
        got = mbar_wait(&full[(it + 1) % kStages], static_cast<uint32_t>((it + 1) / kStages) & 1u, wd);
    }
    __syncwarp();
    ok = group_sync_and(bar_id, got);
    if (!ok) break;
    pending = false;
    tc_fence_after_sync();

    // ---------------------------------------------------------- epilogue
    uint32_t acc[16];
    tmem_ld_x16(tcol + tlane + S::kDCol, acc);
    tmem_wait_regs(acc);
    const int oh = p.oh0 + ly, ow = p.ow0 + lx;
    if (oh < a.OH && ow < a.OW) {
      T* yp = reinterpret_cast<T*>(a.out.y) + p.n * a.out.ys_n + oh * a.out.ys_h + ow * a.out.ys_w;
      const T* rp =
          RES ? reinterpret_cast<const T*>(a.ep.r) + p.n * a.ep.rs_n + oh * a.ep.rs_h + ow * a.ep.rs_w : nullptr;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 s4 = reinterpret_cast<const float4*>(sc)[j], b4 = reinterpret_cast<const float4*>(bi)[j];
        float z[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) z[i] = __uint_as_float(acc[4 * j + i]);
        float4 o;
        if (!RES) {
          o = make_float4(epi_t<ACT, 0>(z[0], s4.x, b4.x, 0.0f), epi_t<ACT, 0>(z[1], s4.y, b4.y, 0.0f),
                          epi_t<ACT, 0>(z[2], s4.z, b4.z, 0.0f), epi_t<ACT, 0>(z[3], s4.w, b4.w, 0.0f));
        } else {
          const float4 rv = load4(rp + 4 * j);
          if (a.ep.res_mode == 1)
            o = make_float4(epi_t<ACT, 1>(z[0], s4.x, b4.x, rv.x), epi_t<ACT, 1>(z[1], s4.y, b4.y, rv.y),
                            epi_t<ACT, 1>(z[2], s4.z, b4.z, rv.z), epi_t<ACT, 1>(z[3], s4.w, b4.w, rv.w));
          else
            o = make_float4(epi_t<ACT, 2>(z[0], s4.x, b4.x, rv.x), epi_t<ACT, 2>(z[1], s4.y, b4.y, rv.y),
                            epi_t<ACT, 2>(z[2], s4.z, b4.z, rv.z), epi_t<ACT, 2>(z[3], s4.w, b4.w, rv.w));
        }
        store4(yp + 4 * j, o);
      }
    }
  }
  // after a timeout: let the copies and the MMA group still in flight finish
  // before the shared memory and TMEM are released
  if (t == 0)
    for (int q = it; q < staged; ++q)
      mbar_wait_drain(&full[q % kStages], static_cast<uint32_t>(q / kStages) & 1u, 20000000ull);
  if (pending) mbar_wait_drain(bar, static_cast<uint32_t>(it) & 1u, 20000000ull);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <typename T, int ACT, bool RES>
cudaError_t launch_t(const StemArgs& a, int sms, cudaStream_t s) {
  constexpr size_t smem = smem_bytes<T>();
  constexpr int kWG = Staging<T>::kWG;
  const cudaError_t e = smem_attr_once<stem_tc_kernel<T, ACT, RES>>(smem);
  if (e != cudaSuccess) return e;
  // one CTA per SM, each of kWG warpgroups taking every (grid * kWG)-th tile
  const long long tiles = static_cast<long long>(a.N) * a.tiles_y * a.tiles_x;
  const long long need = (tiles + kWG - 1) / kWG;
  const unsigned grid = static_cast<unsigned>(need < sms ? need : sms);
  return launch_pdl(stem_tc_kernel<T, ACT, RES>, dim3(grid), dim3(kWG * kWGThreads), smem, s, a);
}

template <typename T, bool RES>
cudaError_t launch_res(const StemArgs& a, int sms, cudaStream_t s) {
  if (a.ep.act == 0) return launch_t<T, 0, RES>(a, sms, s);
  if (a.ep.act == 1) return launch_t<T, 1, RES>(a, sms, s);
  return launch_t<T, 2, RES>(a, sms, s);
}

template <typename T>
cudaError_t launch_type(const StemArgs& a, int sms, cudaStream_t s) {
  return a.ep.res_mode ? launch_res<T, true>(a, sms, s) : launch_res<T, false>(a, sms, s);
}

}  // namespace

bool stem_tc_ok(const StemArgs& a) {
  const long long tiles = static_cast<long long>(a.N) * ((a.OH + kTH - 1) / kTH) * ((a.OW + kTW - 1) / kTW);
  return tiles < (1LL << 31) - static_cast<long long>(kStages) * 152 * 8;  // tile + kStages * workers fits an int
}

cudaError_t launch_stem_tc(const StemArgs& args, bool bf16, int sms, cudaStream_t s) {
  StemArgs a = args;
  a.tiles_y = (a.OH + kTH - 1) / kTH;
  a.tiles_x = (a.OW + kTW - 1) / kTW;
  if (static_cast<long long>(a.N) * a.tiles_y * a.tiles_x == 0) return cudaSuccess;
  if (!stem_tc_ok(a) || sms > 152 * 8) return cudaErrorInvalidValue;
  return bf16 ? launch_type<__nv_bfloat16>(a, sms, s) : launch_type<float>(a, sms, s);
}

}  // namespace cb
