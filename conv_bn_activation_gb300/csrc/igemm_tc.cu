// Host-side sizing and dispatch of the tensor-core implicit GEMM
// (igemm_tc.cuh).  The kernel is instantiated per channel-chunk width in
// igemm_kc8.cu / igemm_kc16.cu / igemm_kc32.cu so that they compile in
// parallel.
#include "igemm_tc.cuh"

namespace cb {

cudaError_t launch_igemm_kc8(const CUtensorMap&, const CUtensorMap&, const IgemmArgs&, int, int, size_t, cudaStream_t);
cudaError_t launch_igemm_kc16(const CUtensorMap&, const CUtensorMap&, const IgemmArgs&, int, int, size_t, cudaStream_t);
cudaError_t launch_igemm_kc32(const CUtensorMap&, const CUtensorMap&, const IgemmArgs&, int, int, size_t, cudaStream_t);

int igemm_read_trace_kc8(unsigned long long* out, int max_records);
int igemm_read_trace_kc16(unsigned long long* out, int max_records);
int igemm_read_trace_kc32(unsigned long long* out, int max_records);
int igemm_read_trace_halo(unsigned long long* out, int max_records);
int igemm_read_trace_halo_cm(unsigned long long* out, int max_records);
int igemm_read_trace_halo_cm192(unsigned long long* out, int max_records);
int igemm_read_trace_halo_kc16(unsigned long long* out, int max_records);
int dw_block_read_trace(unsigned long long* out, int max_records);

// The trace of whichever instantiation recorded one (profiling builds only).
int igemm_read_trace(unsigned long long* out, int max_records) {
  int n = igemm_read_trace_kc32(out, max_records);
  if (n == 0) n = igemm_read_trace_kc16(out, max_records);
  if (n == 0) n = igemm_read_trace_kc8(out, max_records);
  if (n == 0) n = igemm_read_trace_halo(out, max_records);
  if (n == 0) n = igemm_read_trace_halo_cm(out, max_records);
  if (n == 0) n = igemm_read_trace_halo_cm192(out, max_records);
  if (n == 0) n = igemm_read_trace_halo_kc16(out, max_records);
  if (n == 0) n = dw_block_read_trace(out, max_records);
  return n;
}

int igemm_stages(int bn, int kc) {
  const int per = igemm_a_bytes(kc) + igemm_b_bytes(bn, kc);
  int s = (224 * 1024 - 2048 - kIgemmStagingBytes) / per;
  if (s > 16) s = 16;
  if (s < 2) s = 2;
  return s;
}

size_t igemm_smem_bytes(int bn, int kc, int stages) {
  return 1024 /*alignment slack*/ + static_cast<size_t>(stages) * (igemm_a_bytes(kc) + igemm_b_bytes(bn, kc)) +
         kIgemmStagingBytes +
         (2 * stages + 2 * 4) * sizeof(uint64_t) + 16;
}

cudaError_t launch_igemm_bf16_kc8(const CUtensorMap&, const CUtensorMap&, const IgemmArgs&, int, int, size_t,
                                  cudaStream_t);
cudaError_t launch_igemm_bf16_kc16(const CUtensorMap&, const CUtensorMap&, const IgemmArgs&, int, int, size_t,
                                   cudaStream_t);
cudaError_t launch_igemm_bf16_kc32(const CUtensorMap&, const CUtensorMap&, const IgemmArgs&, int, int, size_t,
                                   cudaStream_t);

cudaError_t launch_igemm(const CUtensorMap& amap, const CUtensorMap& bmap, const IgemmArgs& a, int bn, int kc,
                         int grid, size_t smem, cudaStream_t s) {
  if (a.bf16) {
    if (kc == 32) return launch_igemm_bf16_kc32(amap, bmap, a, bn, grid, smem, s);
    if (kc == 16) return launch_igemm_bf16_kc16(amap, bmap, a, bn, grid, smem, s);
    if (kc == 8) return launch_igemm_bf16_kc8(amap, bmap, a, bn, grid, smem, s);
    return cudaErrorInvalidValue;
  }
  if (kc == 32) return launch_igemm_kc32(amap, bmap, a, bn, grid, smem, s);
  if (kc == 16) return launch_igemm_kc16(amap, bmap, a, bn, grid, smem, s);
  if (kc == 8) return launch_igemm_kc8(amap, bmap, a, bn, grid, smem, s);
  return cudaErrorInvalidValue;
}

}  // namespace cb
