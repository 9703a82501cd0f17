// Host-side sizing and dispatch of the halo-tile implicit GEMM
// (igemm_halo.cuh).  The pixel-major tiles are instantiated here, the
// channel-major one in igemm_halo_cm.cu, so that they compile in parallel.
#include "igemm_halo.cuh"
#include "launch_util.h"

namespace cb {

// A tile covers q in [q0, q0 + px) with q0 - y_lo * Wp in [0, Wp): at most
// (px - 1) / Wp + 2 output rows, plus one halo row above and below.
int halo_rows(int wp, int px) { return (px - 1) / wp + 4; }

int halo_buffer_bytes(int wp, int px) {
  const int bytes = (halo_rows(wp, px) * wp + 8) * kHaloKc * 4;
  return (bytes + 1023) / 1024 * 1024;
}

size_t halo_smem_bytes(int co, int halo_bytes, int nb_stages) {
  return 1024 /*alignment slack*/ + 2 * static_cast<size_t>(halo_bytes) +
         static_cast<size_t>(nb_stages) * co * kHaloKc * 4 + kHaloStagingBytes +
         (4 + 2 * nb_stages + 2 * 4) * sizeof(uint64_t) + 16;
}

int igemm_read_trace_halo(unsigned long long* out, int max_records) { return igemm_read_trace_tu(out, max_records); }
int igemm_read_spans_halo(unsigned long long* out, int max_ctas) { return igemm_read_spans_tu(out, max_ctas); }

template <int PX, int CO, bool CM>
cudaError_t halo_launch(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int grid, size_t smem,
                        cudaStream_t s) {
  cudaError_t e = smem_attr_once<igemm_halo_kernel<PX, CO, CM>>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(igemm_halo_kernel<PX, CO, CM>, dim3(grid), dim3(kHaloThreads), smem, s, xmap, wmap, a);
}

cudaError_t launch_igemm_halo_cm(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int grid,
                                 size_t smem, cudaStream_t s);

cudaError_t launch_igemm_halo(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int px, int co,
                              bool cm, int grid, size_t smem, cudaStream_t s) {
  if (a.nb_stages < 2 || a.nb_stages > 16) return cudaErrorInvalidValue;
  if (cm) return px == 256 && co == 128 ? launch_igemm_halo_cm(xmap, wmap, a, grid, smem, s) : cudaErrorInvalidValue;
  if (px != 128) return cudaErrorInvalidValue;
  switch (co) {
    case 32: return halo_launch<128, 32, false>(xmap, wmap, a, grid, smem, s);
    case 64: return halo_launch<128, 64, false>(xmap, wmap, a, grid, smem, s);
    case 128: return halo_launch<128, 128, false>(xmap, wmap, a, grid, smem, s);
    case 256: return halo_launch<128, 256, false>(xmap, wmap, a, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cb
