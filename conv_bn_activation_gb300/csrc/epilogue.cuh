// The fused per-channel epilogue: folded BatchNorm (scale, bias), optional
// residual before or after the activation, ReLU or SiLU.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace cb {

// SiLU(z) = z / (1 + e^-z), with e^-z = 2^(-z log2 e) from the hardware base-2
// exponential and the quotient as z times the hardware reciprocal, both
// approximate instructions with subnormals flushed (each about 2^-22
// relative): five instructions per value, relative error a few 1e-7, inside
// the 1e-5 bar of the fp32 paths.  Large negative z: 2^(+big) = inf, the
// reciprocal 0, the result -0 (the limit); large positive z: e^-z = 0,
// the result z.
__device__ __forceinline__ float silu(float z) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(z * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return z * r;
}

__device__ __forceinline__ float act_apply(float z, int act) {
  if (act == 1) return fmaxf(z, 0.0f);
  if (act == 2) return silu(z);
  return z;
}

// The epilogue with the activation and residual placement fixed at compile
// time, so that the exponentials of neighbouring elements overlap.
template <int ACT, int RES>
__device__ __forceinline__ float epi_t(float acc, float sc, float bi, float r) {
  float z = fmaf(acc, sc, bi);
  if constexpr (RES == 1) z += r;
  if constexpr (ACT == 1) z = fmaxf(z, 0.0f);
  if constexpr (ACT == 2) z = silu(z);
  if constexpr (RES == 2) z += r;
  return z;
}

__device__ __forceinline__ float epi_apply(float acc, float sc, float bi, float r, int act, int res_mode) {
  float z = fmaf(acc, sc, bi);
  if (res_mode == 1) z += r;
  z = act_apply(z, act);
  if (res_mode == 2) z += r;
  return z;
}

__device__ __forceinline__ float4 epi_apply4(float4 acc, float4 sc, float4 bi, float4 r, int act, int res_mode) {
  return make_float4(epi_apply(acc.x, sc.x, bi.x, r.x, act, res_mode), epi_apply(acc.y, sc.y, bi.y, r.y, act, res_mode),
                     epi_apply(acc.z, sc.z, bi.z, r.z, act, res_mode), epi_apply(acc.w, sc.w, bi.w, r.w, act, res_mode));
}

__device__ __forceinline__ float4 ldg4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

__device__ __forceinline__ void fma4(float4& acc, float4 a, float4 b) {
  acc.x = fmaf(a.x, b.x, acc.x);
  acc.y = fmaf(a.y, b.y, acc.y);
  acc.z = fmaf(a.z, b.z, acc.z);
  acc.w = fmaf(a.w, b.w, acc.w);
}

// Four consecutive channels as fp32, from fp32 or bf16 storage (a bf16 value
// is the upper half of the fp32 with the same bits: widening is exact), and
// back (bf16: rounded to nearest even).
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u), __uint_as_float(v.y << 16),
                     __uint_as_float(v.y & 0xFFFF0000u));
}
__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&lo);
  u.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}

}  // namespace cb
