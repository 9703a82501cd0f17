// Write-back of a tensor-core accumulator tile with the fused BN / residual /
// activation epilogue ("YOLO26N Inference Optimisation", kernel fusion:
// conv + BN + SiLU in one kernel; the per-channel scale/bias is the folded
// BatchNorm).
//
// The accumulator sits in TMEM as 128 rows (output pixels) x BN fp32
// columns (output channels).  An epilogue warp may only read its own
// 32-lane quarter, and tcgen05.ld hands thread t row t.  Stored straight
// from there, a warp instruction touches 32 different pixels, 16 bytes
// each: 32 partial-sector writes per instruction, and the store path, not
// the math, sets the epilogue's length.  So each CH-column chunk goes
// through shared memory:
//   1. stage(): thread = row writes its CH values, 16-byte groups
//      XOR-swizzled by row (conflict-free for 8 consecutive rows);
//   2. write(): CH/4 lanes per pixel, each one 16-byte channel group, read
//      the staged values back pixel by pixel (also conflict-free), apply
//      scale/bias, residual and activation, round to TF32 and store: a warp
//      instruction now writes 32 / (CH/4) whole pixel segments.
#pragma once

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace cb {

// SiLU on the tensor-core path is epilogue.cuh's (relative error a few
// 1e-7, far inside this path's TF32 tolerance).  The
// result is rounded to the nearest TF32 value: the MMA truncates its fp32
// operands to TF32, which biases every product toward zero; storing
// round-to-nearest TF32 activations lets the next tensor-core layer read
// them exactly, so the bias does not compound along a chain.
__device__ __forceinline__ float tc_epi(float acc, float sc, float bi, float r, int act, int res_mode) {
  float z = fmaf(acc, sc, bi);
  if (res_mode == 1) z += r;
  if (act == 1) z = fmaxf(z, 0.0f);
  if (act == 2) z = silu(z);
  if (res_mode == 2) z += r;
  return round_tf32(z);
}

// The same with the activation and residual placement fixed at compile
// time: no branch between the elements of a chunk, so their exponentials
// and divisions interleave.
template <int ACT, int RES>
__device__ __forceinline__ float tc_epi_t(float acc, float sc, float bi, float r) {
  float z = fmaf(acc, sc, bi);
  if constexpr (RES == 1) z += r;
  if constexpr (ACT == 1) z = fmaxf(z, 0.0f);
  if constexpr (ACT == 2) z = silu(z);
  if constexpr (RES == 2) z += r;
  return round_tf32(z);
}

// The epilogue after the folded BN (scale and bias applied by the caller,
// two channels per packed FMA).  fp32 outputs (T = float) are rounded to the
// nearest TF32 value; bf16 outputs are rounded to bf16 when stored.
template <int ACT, int RES, typename T = float>
__device__ __forceinline__ float tc_epi_post(float z, float r) {
  if constexpr (RES == 1) z += r;
  if constexpr (ACT == 1) z = fmaxf(z, 0.0f);
  if constexpr (ACT == 2) z = silu(z);
  if constexpr (RES == 2) z += r;
  if constexpr (sizeof(T) == 4) return round_tf32(z);
  return z;
}

// One element of type T widened to fp32, and stored from fp32 (bf16: nearest even).
__device__ __forceinline__ float load1(const float* p) { return *p; }
__device__ __forceinline__ float load1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store1(float* p, float v) { *p = v; }
__device__ __forceinline__ void store1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// 32 lanes x 32 bits, 32 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
  __syncwarp();
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// tcgen05.wait::ld that names the destination registers of the loads it
// waits for, so that no use of them can be scheduled above it.
__device__ __forceinline__ void tmem_wait_regs(uint32_t (&r)[32]) {
  __syncwarp();
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_wait_regs(uint32_t (&r)[16]) {
  __syncwarp();
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_wait_regs(uint32_t (&r)[8]) {
  __syncwarp();
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
               :
               : "memory");
}

template <int CH>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&v)[CH]) {
  static_assert(CH == 8 || CH == 16 || CH == 32, "chunk width");
  if constexpr (CH == 32)
    tmem_ld_x32(taddr, v);
  else if constexpr (CH == 16)
    tmem_ld_x16(taddr, v);
  else
    tmem_ld_x8(taddr, v);
}

template <int CH>
struct TileStore {
  static constexpr int kLpp = CH / 4;     // lanes per pixel in the store phase
  static constexpr int kPpi = 32 / kLpp;  // pixels per store instruction
  static constexpr int kRowBytes = CH * 4;
  static constexpr int kBufBytes = 32 * kRowBytes;  // one warp's staging buffer

  // XOR applied to the 16-byte group index of row `row`: 8 consecutive rows
  // then cover all 8 bank groups both when a thread writes its row and when
  // kLpp lanes read one pixel.
  __device__ static __forceinline__ int swz(int row) {
    if constexpr (CH == 32) return row & 7;
    if constexpr (CH == 16) return (row >> 1) & 3;
    return (row >> 2) & 1;
  }

  __device__ static __forceinline__ void stage(uint8_t* buf, int lane, const uint32_t (&v)[CH]) {
    uint8_t* rowp = buf + lane * kRowBytes;
    const int s = swz(lane);
#pragma unroll
    for (int j = 0; j < CH / 4; ++j)
      *reinterpret_cast<uint4*>(rowp + ((j ^ s) << 4)) = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  }

  // Per-lane epilogue constants of one chunk: the lane's 16-byte channel
  // group c .. c + 3 (c = c0 + 4 * (lane % kLpp)) and its folded-BN scale
  // and bias.  Loaded once per chunk position, ahead of the chunk they
  // serve.
  struct Consts {
    float sc[4], bi[4];
    int c;
    bool cvec, cin;
  };
  __device__ static __forceinline__ Consts consts(int lane, int c0, int Cout, bool vec, const Epilogue& ep) {
    Consts k;
    k.c = c0 + 4 * (lane % kLpp);
    k.cvec = vec && k.c + 4 <= Cout;
    k.cin = k.c < Cout;
    if (k.cvec) {
      const float4 s4 = __ldg(reinterpret_cast<const float4*>(ep.scale + k.c));
      const float4 b4 = __ldg(reinterpret_cast<const float4*>(ep.bias + k.c));
      k.sc[0] = s4.x, k.sc[1] = s4.y, k.sc[2] = s4.z, k.sc[3] = s4.w;
      k.bi[0] = b4.x, k.bi[1] = b4.y, k.bi[2] = b4.z, k.bi[3] = b4.w;
    } else {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        k.sc[jj] = k.c + jj < Cout ? __ldg(ep.scale + k.c + jj) : 0.0f;
        k.bi[jj] = k.c + jj < Cout ? __ldg(ep.bias + k.c + jj) : 0.0f;
      }
    }
    return k;
  }

  // yoff / roff: this lane's row's element offsets into y / r (yoff < 0:
  // row masked).  One uniform branch per chunk picks the compile-time
  // epilogue.  T: the element type of y and r (the views' storage type).
  template <typename T = float>
  __device__ static __forceinline__ void write(const uint8_t* buf, int lane, long long yoff, long long roff,
                                               const Consts& k, int Cout, const OutView& out, const Epilogue& ep) {
    switch (ep.act * 3 + ep.res_mode) {
      case 0: write_t<0, 0, T>(buf, lane, yoff, roff, k, Cout, out, ep); break;
      case 1: write_t<0, 1, T>(buf, lane, yoff, roff, k, Cout, out, ep); break;
      case 2: write_t<0, 2, T>(buf, lane, yoff, roff, k, Cout, out, ep); break;
      case 3: write_t<1, 0, T>(buf, lane, yoff, roff, k, Cout, out, ep); break;
      case 4: write_t<1, 1, T>(buf, lane, yoff, roff, k, Cout, out, ep); break;
      case 5: write_t<1, 2, T>(buf, lane, yoff, roff, k, Cout, out, ep); break;
      case 6: write_t<2, 0, T>(buf, lane, yoff, roff, k, Cout, out, ep); break;
      case 7: write_t<2, 1, T>(buf, lane, yoff, roff, k, Cout, out, ep); break;
      default: write_t<2, 2, T>(buf, lane, yoff, roff, k, Cout, out, ep); break;
    }
  }

  // Straight-line over the kLpp passes: all loads first, then all the math,
  // then the (predicated) stores, so that the exponentials and reciprocals of
  // different pixels overlap instead of each pass waiting on the last.
  template <int ACT, int RES, typename T>
  __device__ static __forceinline__ void write_t(const uint8_t* buf, int lane, long long yoff, long long roff,
                                                 const Consts& k, int Cout, const OutView& out,
                                                 const Epilogue& ep) {
    const int j = lane % kLpp;
    const int c = k.c;
    long long yo[kLpp], ro[kLpp];
    float z[kLpp][4];
#pragma unroll
    for (int pass = 0; pass < kLpp; ++pass) {
      const int p = pass * kPpi + lane / kLpp;
      yo[pass] = __shfl_sync(0xffffffffu, yoff, p);
      ro[pass] = RES != 0 ? __shfl_sync(0xffffffffu, roff, p) : 0;
      const uint4 u = *reinterpret_cast<const uint4*>(buf + p * kRowBytes + ((j ^ swz(p)) << 4));
      z[pass][0] = __uint_as_float(u.x), z[pass][1] = __uint_as_float(u.y);
      z[pass][2] = __uint_as_float(u.z), z[pass][3] = __uint_as_float(u.w);
    }
    float r[kLpp][4];
#pragma unroll
    for (int pass = 0; pass < kLpp; ++pass) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) r[pass][jj] = 0.0f;
      if constexpr (RES != 0) {
        if (yo[pass] >= 0 && k.cin) {
          const T* rp = reinterpret_cast<const T*>(ep.r) + ro[pass] + c;
          if (k.cvec) {
            const float4 t = load4(rp);
            r[pass][0] = t.x, r[pass][1] = t.y, r[pass][2] = t.z, r[pass][3] = t.w;
          } else {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
              if (c + jj < Cout) r[pass][jj] = load1(rp + jj);
          }
        }
      }
    }
#pragma unroll
    for (int pass = 0; pass < kLpp; ++pass)
#pragma unroll
      for (int jj = 0; jj < 4; jj += 2) {
        // scale and bias of two channels in one packed FMA (each lane one fmaf)
        const float2 a = __ffma2_rn(make_float2(z[pass][jj], z[pass][jj + 1]), make_float2(k.sc[jj], k.sc[jj + 1]),
                                    make_float2(k.bi[jj], k.bi[jj + 1]));
        z[pass][jj] = tc_epi_post<ACT, RES, T>(a.x, r[pass][jj]);
        z[pass][jj + 1] = tc_epi_post<ACT, RES, T>(a.y, r[pass][jj + 1]);
      }
#pragma unroll
    for (int pass = 0; pass < kLpp; ++pass) {
      if (yo[pass] < 0 || !k.cin) continue;
      T* yp = reinterpret_cast<T*>(out.y) + yo[pass] + c;
      if (k.cvec) {
        store4(yp, make_float4(z[pass][0], z[pass][1], z[pass][2], z[pass][3]));
      } else {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
          if (c + jj < Cout) store1(yp + jj, z[pass][jj]);
      }
    }
  }
};

}  // namespace cb
