// Host-side sizing and dispatch of the halo-tile implicit GEMM
// (igemm_halo.cuh).  The pixel-major tiles are instantiated here, the
// channel-major ones in igemm_halo_cm.cu and igemm_halo_cm192.cu, so that
// they compile in parallel.
#include <map>
#include <mutex>
#include <tuple>

#include "igemm_halo.cuh"
#include "launch_util.h"

namespace cb {

// A tile covers q in [q0, q0 + px) with q0 - y_lo * Wp in [0, Wp): at most
// (px - 1) / Wp + 2 output rows, plus one halo row above and below (stride 1);
// at stride 2 a phase tile holds those output rows and the one above.
int halo_rows(int wp, int px, int stride) { return (px - 1) / wp + (stride == 1 ? 4 : 3); }

// Bytes of one halo buffer: one tile (stride 1) or four phase tiles (stride
// 2) of rows x Wp pixels of kc channels, plus 8 pixels that only the
// discarded padding columns of the last rows read; 1 KB multiples.
int halo_buffer_bytes(int wp, int px, int kc, int stride) {
  const int bytes = ((halo_rows(wp, px, stride) * wp + 8) * kc * 4 + 1023) / 1024 * 1024;
  return stride == 1 ? bytes : 4 * bytes;
}

size_t halo_smem_bytes(int co, int halo_bytes, int nb_stages, int taps_per_stage, int kc) {
  return 1024 /*alignment slack*/ + 2 * static_cast<size_t>(halo_bytes) +
         static_cast<size_t>(nb_stages) * taps_per_stage * co * kc * 4 + kHaloStagingBytes +
         (4 + 2 * nb_stages + 2 * 8 + 2) * sizeof(uint64_t) + 16;
}

size_t halo_split_recv_bytes(int px, int co, bool cm) { return static_cast<size_t>(cm ? px : co) / 2 * 128 * 4; }

int igemm_read_trace_halo(unsigned long long* out, int max_records) { return igemm_read_trace_tu(out, max_records); }
int igemm_read_spans_halo(unsigned long long* out, int max_ctas) { return igemm_read_spans_tu(out, max_ctas); }

int halo_max_pairs_cm256(size_t smem);
int halo_max_pairs_cm192(size_t smem);

int halo_max_pairs(int px, int co, bool cm, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, size_t>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, px, co, cm ? 1 : 0, smem);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int n = 0;
  if (cm) n = co != 128 ? 0 : px == 256 ? halo_max_pairs_cm256(smem) : px == 192 ? halo_max_pairs_cm192(smem) : 0;
  else if (px == 128 && co == 64) n = halo_pairs<128, 64, false>(smem);
  else if (px == 128 && co == 128) n = halo_pairs<128, 128, false>(smem);
  else if (px == 128 && co == 256) n = halo_pairs<128, 256, false>(smem);
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = n;
  return n;
}

cudaError_t launch_igemm_halo_cm256(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int grid,
                                    size_t smem, cudaStream_t s);
cudaError_t launch_igemm_halo_cm192(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int grid,
                                    size_t smem, cudaStream_t s);
cudaError_t launch_igemm_halo_kc16(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int co,
                                   int grid, size_t smem, cudaStream_t s);
cudaError_t launch_igemm_halo_kc8(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int co,
                                  int grid, size_t smem, cudaStream_t s);

cudaError_t launch_igemm_halo_bf16(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int px,
                                   int co, bool cm, int grid, size_t smem, cudaStream_t s);

cudaError_t launch_igemm_halo(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int px, int co,
                              bool cm, int grid, size_t smem, cudaStream_t s) {
  if (a.nb_stages < (a.w_resident ? 1 : 2) || a.nb_stages > 16) return cudaErrorInvalidValue;
  if (a.taps_per_stage != 1 && a.taps_per_stage != 3 && a.taps_per_stage != 9) return cudaErrorInvalidValue;
  if (a.split_k != 1 && a.split_k != 2) return cudaErrorInvalidValue;
  if (a.stride != 1 && a.stride != 2) return cudaErrorInvalidValue;
  if (a.sub < 1 || a.sub > kHaloMaxSub || (a.sub > 1 && (cm || co > 64 || a.split_k != 1))) return cudaErrorInvalidValue;
  if (a.w_resident &&
      (a.num_kc != 1 || a.n_tiles != 1 || a.split_k != 1 || a.taps_per_stage != 9 || a.nb_stages != 1))
    return cudaErrorInvalidValue;
  if (a.stride == 2 && ((a.kc != 16 && !(a.bf16 && a.kc == 8)) || a.phase_bytes * 4 != a.halo_bytes ||
                        a.Wp * 2 > 256 || a.rows * 2 > 256))
    return cudaErrorInvalidValue;
  if (a.split_k == 2) {
    // one tile per cluster, a channel-chunk per CTA at least, the partner's
    // half accumulator within the operand buffers, a shape that splits
    if (grid != 2 * a.m_tiles * a.n_tiles || a.num_kc < 2 || (!cm && co < 64) ||
        halo_split_recv_bytes(px, co, cm) > 2 * static_cast<size_t>(a.halo_bytes) +
                                                static_cast<size_t>(a.nb_stages) * a.taps_per_stage * co * a.kc * 4)
      return cudaErrorInvalidValue;
  }
  if (cm && co == 128 && px == 192 && a.kc == 32) return launch_igemm_halo_cm192(xmap, wmap, a, grid, smem, s);
  if (a.bf16) return launch_igemm_halo_bf16(xmap, wmap, a, px, co, cm, grid, smem, s);
  if (a.kc == 16) return !cm && px == 128 ? launch_igemm_halo_kc16(xmap, wmap, a, co, grid, smem, s) : cudaErrorInvalidValue;
  if (a.kc == 8) return !cm && px == 128 ? launch_igemm_halo_kc8(xmap, wmap, a, co, grid, smem, s) : cudaErrorInvalidValue;
  if (a.kc != 32) return cudaErrorInvalidValue;
  if (cm) return px == 256 && co == 128 ? launch_igemm_halo_cm256(xmap, wmap, a, grid, smem, s) : cudaErrorInvalidValue;
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
