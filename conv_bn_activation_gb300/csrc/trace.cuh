// Optional timeline of one CTA of the tensor-core kernels (profiling aid,
// compiled in only with -DCB_IGEMM_TRACE): each role keeps clock64 stamps in
// a local array and copies them out when it finishes.
#pragma once

#include <cuda_runtime.h>

namespace cb {

#ifdef CB_IGEMM_TRACE
constexpr int kTraceRecords = 512;
static __device__ unsigned long long g_igemm_trace[3 * kTraceRecords];  // one copy per translation unit
static __device__ int g_igemm_trace_n[3];
struct TraceBuf {
  unsigned long long t[kTraceRecords];
  int n = 0;
  __device__ __forceinline__ void add(bool on) {
    if (on && n < kTraceRecords) t[n++] = clock64();
  }
  __device__ __forceinline__ void flush(bool on, int role) {
    if (!on) return;
    for (int i = 0; i < n; ++i) g_igemm_trace[role * kTraceRecords + i] = t[i];
    g_igemm_trace_n[role] = n;
  }
};
// Start / end (global timer, ns) and SM of every CTA of the traced launch.
constexpr int kTraceCtas = 1024;
static __device__ unsigned long long g_igemm_cta_span[2 * 3 * kTraceCtas];  // two launch slots
__device__ __forceinline__ unsigned long long trace_globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// trace: 1 or 2 = launch slot; which: 0 start, 1 end.
__device__ __forceinline__ void trace_cta_span(int trace, int which, unsigned long long t) {
  if (trace >= 1 && trace <= 2 && blockIdx.x < kTraceCtas) {
    unsigned int sm;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    unsigned long long* row = g_igemm_cta_span + 3 * ((trace - 1) * kTraceCtas + blockIdx.x);
    row[which] = t;
    row[2] = sm;
  }
}
#else
__device__ __forceinline__ unsigned long long trace_globaltimer() { return 0; }
__device__ __forceinline__ void trace_cta_span(int, int, unsigned long long) {}
struct TraceBuf {
  __device__ __forceinline__ void add(bool) {}
  __device__ __forceinline__ void flush(bool, int) {}
};
#endif


// Copies the per-CTA spans of the last traced launch out (3 words per CTA).
static inline int igemm_read_spans_tu(unsigned long long* out, int max_ctas) {
#ifdef CB_IGEMM_TRACE
  if (max_ctas < 2 * kTraceCtas) return -1;
  if (cudaMemcpyFromSymbol(out, g_igemm_cta_span, sizeof(g_igemm_cta_span)) != cudaSuccess) return -1;
  const unsigned long long zero[3 * kTraceCtas] = {};
  cudaMemcpyToSymbol(g_igemm_cta_span, zero, sizeof(zero));
  cudaMemcpyToSymbol(g_igemm_cta_span, zero, sizeof(zero), sizeof(zero));
  return 2 * kTraceCtas;
#else
  (void)out;
  (void)max_ctas;
  return 0;
#endif
}

// Copies this translation unit's trace out (see TraceBuf); returns the record count.
static inline int igemm_read_trace_tu(unsigned long long* out, int max_records) {
#ifdef CB_IGEMM_TRACE
  int n[3] = {0, 0, 0};
  if (cudaMemcpyFromSymbol(n, g_igemm_trace_n, sizeof(n)) != cudaSuccess) return -1;
  if (n[0] + n[1] + n[2] == 0) return 0;
  if (max_records < 3 * kTraceRecords + 3) return -1;
  if (cudaMemcpyFromSymbol(out + 3, g_igemm_trace, sizeof(unsigned long long) * 3 * kTraceRecords) != cudaSuccess)
    return -1;
  out[0] = n[0];
  out[1] = n[1];
  out[2] = n[2];
  const int zero[3] = {0, 0, 0};
  cudaMemcpyToSymbol(g_igemm_trace_n, zero, sizeof(zero));
  return n[0] + n[1] + n[2];
#else
  (void)out;
  (void)max_records;
  return 0;
#endif
}

}  // namespace cb
