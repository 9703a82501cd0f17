// Host-side sizing and dispatch of the halo-tile implicit GEMM
// (igemm_halo.cuh).
#include "igemm_halo.cuh"
#include "launch_util.h"

namespace cb {

// A tile covers q in [q0, q0 + 128) with q0 - y_lo * Wp in [0, Wp): at most
// 127 / Wp + 2 output rows, plus one halo row above and below.
int halo_rows(int wp) { return 127 / wp + 4; }

int halo_buffer_bytes(int wp) {
  const int bytes = (halo_rows(wp) * wp + 8) * kHaloKc * 4;
  return (bytes + 1023) / 1024 * 1024;
}

size_t halo_smem_bytes(int bn, int halo_bytes, int nb_stages) {
  return 1024 /*alignment slack*/ + 2 * static_cast<size_t>(halo_bytes) +
         static_cast<size_t>(nb_stages) * bn * kHaloKc * 4 + kHaloStagingBytes +
         (4 + 2 * nb_stages + 2 * 4) * sizeof(uint64_t) + 16;
}

template <int BN>
static cudaError_t halo_launch_bn(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int grid,
                                  size_t smem, cudaStream_t s) {
  cudaError_t e = smem_attr_once<igemm_halo_kernel<BN>>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(igemm_halo_kernel<BN>, dim3(grid), dim3(kHaloThreads), smem, s, xmap, wmap, a);
}

int igemm_read_trace_halo(unsigned long long* out, int max_records) { return igemm_read_trace_tu(out, max_records); }
int igemm_read_spans_halo(unsigned long long* out, int max_ctas) { return igemm_read_spans_tu(out, max_ctas); }

cudaError_t launch_igemm_halo(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int bn, int grid,
                              size_t smem, cudaStream_t s) {
  if (a.nb_stages < 2 || a.nb_stages > 16) return cudaErrorInvalidValue;
  switch (bn) {
    case 32: return halo_launch_bn<32>(xmap, wmap, a, grid, smem, s);
    case 64: return halo_launch_bn<64>(xmap, wmap, a, grid, smem, s);
    case 128: return halo_launch_bn<128>(xmap, wmap, a, grid, smem, s);
    case 256: return halo_launch_bn<256>(xmap, wmap, a, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cb
