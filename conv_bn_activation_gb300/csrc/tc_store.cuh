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

#include "internal.h"
#include "ptx.cuh"

namespace cb {

// SiLU on the tensor-core path uses the fast exponential and division
// (relative error ~1e-6, far inside this path's TF32 tolerance).  The
// result is rounded to the nearest TF32 value: the MMA truncates its fp32
// operands to TF32, which biases every product toward zero; storing
// round-to-nearest TF32 activations lets the next tensor-core layer read
// them exactly, so the bias does not compound along a chain.
__device__ __forceinline__ float tc_epi(float acc, float sc, float bi, float r, int act, int res_mode) {
  float z = fmaf(acc, sc, bi);
  if (res_mode == 1) z += r;
  if (act == 1) z = fmaxf(z, 0.0f);
  if (act == 2) z = __fdividef(z, 1.0f + __expf(-z));
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
  if constexpr (ACT == 2) z = __fdividef(z, 1.0f + __expf(-z));
  if constexpr (RES == 2) z += r;
  return round_tf32(z);
}

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

  // yoff / roff: this lane's row's element offsets into y / r (yoff < 0:
  // row masked).  c0: first output channel of the chunk.  One uniform
  // branch per chunk picks the compile-time epilogue.
  __device__ static __forceinline__ void write(const uint8_t* buf, int lane, long long yoff, long long roff, int c0,
                                               int Cout, bool vec, const OutView& out, const Epilogue& ep) {
    switch (ep.act * 3 + ep.res_mode) {
      case 0: write_t<0, 0>(buf, lane, yoff, roff, c0, Cout, vec, out, ep); break;
      case 1: write_t<0, 1>(buf, lane, yoff, roff, c0, Cout, vec, out, ep); break;
      case 2: write_t<0, 2>(buf, lane, yoff, roff, c0, Cout, vec, out, ep); break;
      case 3: write_t<1, 0>(buf, lane, yoff, roff, c0, Cout, vec, out, ep); break;
      case 4: write_t<1, 1>(buf, lane, yoff, roff, c0, Cout, vec, out, ep); break;
      case 5: write_t<1, 2>(buf, lane, yoff, roff, c0, Cout, vec, out, ep); break;
      case 6: write_t<2, 0>(buf, lane, yoff, roff, c0, Cout, vec, out, ep); break;
      case 7: write_t<2, 1>(buf, lane, yoff, roff, c0, Cout, vec, out, ep); break;
      default: write_t<2, 2>(buf, lane, yoff, roff, c0, Cout, vec, out, ep); break;
    }
  }

  template <int ACT, int RES>
  __device__ static __forceinline__ void write_t(const uint8_t* buf, int lane, long long yoff, long long roff,
                                                 int c0, int Cout, bool vec, const OutView& out,
                                                 const Epilogue& ep) {
    const int j = lane % kLpp;
    const int c = c0 + 4 * j;
    const bool cvec = vec && c + 4 <= Cout;
    constexpr bool res = RES != 0;
    float sc[4], bi[4];
    if (cvec) {
      const float4 s4 = __ldg(reinterpret_cast<const float4*>(ep.scale + c));
      const float4 b4 = __ldg(reinterpret_cast<const float4*>(ep.bias + c));
      sc[0] = s4.x, sc[1] = s4.y, sc[2] = s4.z, sc[3] = s4.w;
      bi[0] = b4.x, bi[1] = b4.y, bi[2] = b4.z, bi[3] = b4.w;
    } else {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        sc[jj] = c + jj < Cout ? __ldg(ep.scale + c + jj) : 0.0f;
        bi[jj] = c + jj < Cout ? __ldg(ep.bias + c + jj) : 0.0f;
      }
    }
#pragma unroll
    for (int pass = 0; pass < kLpp; ++pass) {
      const int p = pass * kPpi + lane / kLpp;
      const long long yo = __shfl_sync(0xffffffffu, yoff, p);
      const long long ro = res ? __shfl_sync(0xffffffffu, roff, p) : 0;
      if (yo < 0 || c >= Cout) continue;
      const uint4 u = *reinterpret_cast<const uint4*>(buf + p * kRowBytes + ((j ^ swz(p)) << 4));
      const float acc[4] = {__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w)};
      float r[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if constexpr (res) {
        const float* rp = ep.r + ro + c;
        if (cvec) {
          const float4 t = *reinterpret_cast<const float4*>(rp);
          r[0] = t.x, r[1] = t.y, r[2] = t.z, r[3] = t.w;
        } else {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
            if (c + jj < Cout) r[jj] = rp[jj];
        }
      }
      float o[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) o[jj] = tc_epi_t<ACT, RES>(acc[jj], sc[jj], bi[jj], r[jj]);
      float* yp = out.y + yo + c;
      if (cvec) {
        *reinterpret_cast<float4*>(yp) = make_float4(o[0], o[1], o[2], o[3]);
      } else {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
          if (c + jj < Cout) yp[jj] = o[jj];
      }
    }
  }
};

}  // namespace cb
