// Bilinear resampling arithmetic of the u8 preprocess (half-pixel centres,
// border clamps, u8 rounding), shared by the preprocess kernels and the
// stem kernel that runs the preprocess in its input staging.  Every fp32
// operation is rounded separately (explicit _rn intrinsics, no contraction),
// so all users produce identical values ("A fused Ampere preprocess
// kernel": bilinear is a contract with the reference resize).
#pragma once

#include <cstdint>

namespace cb {

struct AxisSample {
  int i0, i1;
  float a;
};

// Exact small-integer conversions without the quarter-rate convert unit:
// adding 2^23 leaves an integer in the low mantissa bits.
__device__ __forceinline__ float u8_to_float(uint32_t b) { return __int_as_float(0x4B000000 | b) - 8388608.0f; }
// floor(x) for 0 <= x < 2^22: round the sum down, then read the integer back.
__device__ __forceinline__ int floor_nonneg(float x) { return __float_as_int(__fadd_rd(x, 8388608.0f)) - 0x4B000000; }

// scale = S / D (IEEE fp32 division, computed once per launch row).  A
// negative f is clamped to 0 before the floor, which gives the same
// (i0 = 0, a = 0) as flooring it and then clamping i0.
__device__ __forceinline__ AxisSample axis_sample(int d, int S, float scale) {
  const float f = fmaxf(__fsub_rn(__fmul_rn(__fadd_rn(static_cast<float>(d), 0.5f), scale), 0.5f), 0.0f);
  int k = floor_nonneg(f);
  float t = __fsub_rn(f, static_cast<float>(k));
  if (k >= S - 1) {
    k = S - 1;
    t = 0.0f;
  }
  AxisSample s;
  s.i0 = k;
  s.i1 = (k + 1 < S) ? k + 1 : S - 1;
  s.a = t;
  return s;
}

__device__ __forceinline__ float bilinear(float p00, float p01, float p10, float p11, float ax, float ay) {
  const float bx = __fsub_rn(1.0f, ax), by = __fsub_rn(1.0f, ay);
  const float top = __fadd_rn(__fmul_rn(bx, p00), __fmul_rn(ax, p01));
  const float bot = __fadd_rn(__fmul_rn(bx, p10), __fmul_rn(ax, p11));
  return __fadd_rn(__fmul_rn(by, top), __fmul_rn(ay, bot));
}

// u8 code of a bilinear value: floor(v + 0.5); v is a convex combination of
// u8 samples, so the code is already within [0, 255].
__device__ __forceinline__ int round_u8(float v) { return floor_nonneg(__fadd_rn(v, 0.5f)); }

// Sums of the horizontal sample pairs of one staged source row for the 4
// destination pixels of group g at an exact 2:1 width ratio: destination
// column dx samples source columns 2dx and 2dx + 1 with weight 1/2 each, so
// the bilinear row value 0.5 * p0 + 0.5 * p1 is exactly (p0 + p1) / 2; this
// keeps the integer sum p0 + p1 (as a float) per channel and pixel.
__device__ __forceinline__ void pair_sums_int(const uint8_t* row, int g, uint32_t (&h)[12]) {
  const uint2* w2 = reinterpret_cast<const uint2*>(row + g * 24);
  uint32_t w[6];
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const uint2 t = w2[i];
    w[2 * i] = t.x, w[2 * i + 1] = t.y;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      const int b0 = q * 6 + c, b1 = q * 6 + 3 + c;  // byte offsets of the two samples
      h[q * 3 + c] = __byte_perm(w[b0 >> 2], 0u, 0x4440u | (b0 & 3)) + __byte_perm(w[b1 >> 2], 0u, 0x4440u | (b1 & 3));
    }
}

__device__ __forceinline__ void pair_sums(const uint8_t* row, int g, float (&h)[12]) {
  uint32_t s[12];
  pair_sums_int(row, g, s);
#pragma unroll
  for (int i = 0; i < 12; ++i) h[i] = u8_to_float(s[i]);  // sum <= 510: exact
}

// The u8 codes of 2:1-width samples from the pair sums of the top (ht) and
// bottom (hb) source rows at vertical weight ay:
//   u = floor(hbw * ht + haw * hb + 0.5), hbw = (1 - ay) / 2, haw = ay / 2,
// each fp32 operation rounded.  When ay is a multiple of 2^-14 (the 720 ->
// 480 ratio gives 1/4 and 3/4) every one of those operations is exact --
// products of a 9-bit integer and a 15-bit dyadic fraction, and a sum below
// 256 on a 2^-15 grid, all within fp32's 24 bits -- so the same code comes out
// of integer arithmetic: u = (hbI * ht + haI * hb + 2^14) >> 15 with
// haI = ay * 2^14, hbI = 2^14 - haI.  Otherwise the fp32 operations run.
__device__ __forceinline__ void blend_pairs(const uint8_t* top, const uint8_t* bot, float ay, int (&o)[12]) {
  uint32_t ht[12], hb[12];
  pair_sums_int(top, 0, ht);
  pair_sums_int(bot, 0, hb);
  const float t = __fmul_rn(ay, 16384.0f);
  if (t == truncf(t)) {
    const uint32_t wa = static_cast<uint32_t>(t), wt = 16384u - wa;
#pragma unroll
    for (int k = 0; k < 12; ++k) o[k] = static_cast<int>((wt * ht[k] + wa * hb[k] + 16384u) >> 15);
  } else {
    const float wt = __fmul_rn(0.5f, __fsub_rn(1.0f, ay)), wb = __fmul_rn(0.5f, ay);
#pragma unroll
    for (int k = 0; k < 12; ++k)
      o[k] = round_u8(__fadd_rn(__fmul_rn(wt, u8_to_float(ht[k])), __fmul_rn(wb, u8_to_float(hb[k]))));
  }
}

}  // namespace cb
