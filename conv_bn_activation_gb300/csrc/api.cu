// The C ABI: argument validation, per-shape kernel choice, TMA descriptor
// encoding and launches.  Host code only (the kernels live in the other .cu
// files of this directory).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "cb.h"
#include "internal.h"
#include "launch_util.h"

namespace cb {
int dw_tma_blocks_per_sm(int stride, int threads, size_t smem, bool bf16);
int igemm_read_spans_halo(unsigned long long* out, int max_ctas);
}

using namespace cb;

// Device error word: kernels record CB_ERR_TIMEOUT here when a bounded wait gives up.
__device__ int g_cb_device_error;

namespace {

constexpr int kVersion = 100;  // 0.1.0
thread_local int t_last_cuda_error = 0;
std::atomic<int> g_policy{0};

cb_status cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return CB_ERR_CUDA;
}

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int* err = nullptr;
};
std::mutex g_mu;
DeviceInfo g_devices[128];

cb_status current_device(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 128) return CB_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_devices[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_cb_device_error);
    if (e != cudaSuccess) return cuda_fail(e);
    d.err = static_cast<int*>(p);
    d.ready = true;
  }
  *out = &d;
  return CB_OK;
}

uint64_t timeout_ns();  // the CB_TIMEOUT_MS tuning knob, in nanoseconds

// ---------------------------------------------------------- driver entry points
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
using EncodeIm2colFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const int*, const int*, cuuint32_t, cuuint32_t,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

void* driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return p;
}

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = reinterpret_cast<EncodeTiledFn>(driver_fn("cuTensorMapEncodeTiled"));
  return fn;
}

EncodeIm2colFn encode_im2col() {
  static EncodeIm2colFn fn = reinterpret_cast<EncodeIm2colFn>(driver_fn("cuTensorMapEncodeIm2col"));
  return fn;
}

// Tensor maps, cached: encoding one costs microseconds, as much as the launch
// itself, and a network calls the same layers with the same buffers over and
// over.  The key is every argument of the encode call (the map is a pure
// function of them), so a buffer freed and reallocated at the same address
// with the same shape maps to the same, still correct, descriptor.
struct MapCache {
  std::mutex mu;
  std::unordered_map<std::string, CUtensorMap> maps;
};
MapCache g_maps;

template <typename... Parts>
std::string map_key(const Parts&... parts) {
  std::string k;
  (k.append(reinterpret_cast<const char*>(&parts), sizeof(parts)), ...);
  return k;
}

bool cached_map(const std::string& key, CUtensorMap* out) {
  std::lock_guard<std::mutex> lock(g_maps.mu);
  auto it = g_maps.maps.find(key);
  if (it == g_maps.maps.end()) return false;
  *out = it->second;
  return true;
}

void store_map(const std::string& key, const CUtensorMap& m) {
  std::lock_guard<std::mutex> lock(g_maps.mu);
  if (g_maps.maps.size() >= 4096) g_maps.maps.clear();
  g_maps.maps.emplace(key, m);
}

// fp32 tiled map of rank <= 5 (no interleave, 256-byte L2 promotion, zero fill).
CUresult tiled_map(CUtensorMap* out, int rank, const void* ptr, const cuuint64_t* dims, const cuuint64_t* strides,
                   const cuuint32_t* box, const cuuint32_t* estr, CUtensorMapSwizzle swz,
                   CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_FLOAT32) {
  cuuint64_t d[5] = {}, st[4] = {};
  cuuint32_t b[5] = {}, e[5] = {};
  for (int i = 0; i < rank; ++i) d[i] = dims[i], b[i] = box[i], e[i] = estr[i];
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
  const int kind = dtype == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? 0 : 16 + static_cast<int>(dtype);
  const std::string key = map_key(kind, rank, ptr, d, st, b, e, swz);
  if (cached_map(key, out)) return CUDA_SUCCESS;
  const CUresult r = encode_tiled()(out, dtype, static_cast<cuuint32_t>(rank),
                                    const_cast<void*>(ptr), d, st, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) store_map(key, *out);
  return r;
}

// 4-D im2col map (same fixed options as tiled_map).
CUresult im2col_map(CUtensorMap* out, const void* ptr, const cuuint64_t* dims, const cuuint64_t* strides,
                    const int* lower, const int* upper, cuuint32_t channels, cuuint32_t pixels,
                    const cuuint32_t* estr, CUtensorMapSwizzle swz,
                    CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_FLOAT32) {
  cuuint64_t d[4], st[3];
  cuuint32_t e[4];
  int lo[2] = {lower[0], lower[1]}, up[2] = {upper[0], upper[1]};
  for (int i = 0; i < 4; ++i) d[i] = dims[i], e[i] = estr[i];
  for (int i = 0; i < 3; ++i) st[i] = strides[i];
  const int kind = 1 + 16 * static_cast<int>(dtype);
  const std::string key = map_key(kind, ptr, d, st, lo, up, channels, pixels, e, swz);
  if (cached_map(key, out)) return CUDA_SUCCESS;
  const CUresult r = encode_im2col()(out, dtype, 4, const_cast<void*>(ptr), d, st, lo, up,
                                     channels, pixels, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) store_map(key, *out);
  return r;
}

// ------------------------------------------------------------------ validation
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bytes per element of a view.
size_t elem_bytes(const cb_tensor* t) { return t->dtype == CB_DTYPE_BF16 ? 2 : 4; }
bool is_f32(const cb_tensor* t) { return t->dtype == CB_DTYPE_F32; }

bool view_ok(const cb_tensor* t) {
  if (!t) return false;
  if (t->dtype != CB_DTYPE_F32 && t->dtype != CB_DTYPE_BF16) return false;
  if (t->n < 0 || t->h < 1 || t->w < 1 || t->c < 1) return false;
  if (t->layout != CB_LAYOUT_NHWC && t->layout != CB_LAYOUT_NCHW) return false;
  if (t->stride_n < 0 || t->stride_h < 0 || t->stride_w < 0 || t->stride_c < 0) return false;
  if (t->layout == CB_LAYOUT_NHWC && t->stride_c != 1) return false;
  if (t->layout == CB_LAYOUT_NCHW && t->stride_w != 1) return false;
  if (t->n > 0 && !t->data) return false;
  return true;
}

// Byte range [lo, hi) spanned by a view (strides are non-negative).
void view_range(const cb_tensor* t, uintptr_t* lo, uintptr_t* hi) {
  const long long last = (static_cast<long long>(t->n) - 1) * t->stride_n + (t->h - 1LL) * t->stride_h +
                         (t->w - 1LL) * t->stride_w + (t->c - 1LL) * t->stride_c;
  *lo = reinterpret_cast<uintptr_t>(t->data);
  *hi = *lo + static_cast<uintptr_t>(last + 1) * elem_bytes(t);
}

// Disjoint channel slices of one NHWC buffer (same n/h/w strides, both
// slices inside one pixel's stride_w elements, every stride a multiple of
// stride_w) share no element even though their byte ranges interleave.
bool disjoint_channel_slices(const cb_tensor* a, const cb_tensor* b) {
  if (a->layout != CB_LAYOUT_NHWC || b->layout != CB_LAYOUT_NHWC || a->dtype != b->dtype) return false;
  const uintptr_t eb = elem_bytes(a);
  if (a->stride_n != b->stride_n || a->stride_h != b->stride_h || a->stride_w != b->stride_w) return false;
  const long long sw = a->stride_w;
  if (sw <= 0 || a->stride_h % sw != 0 || a->stride_n % sw != 0) return false;
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a->data), pb = reinterpret_cast<uintptr_t>(b->data);
  const uintptr_t base = pa < pb ? pa : pb;
  if ((pa - base) % eb != 0 || (pb - base) % eb != 0) return false;
  const long long da = static_cast<long long>((pa - base) / eb);
  const long long db = static_cast<long long>((pb - base) / eb);
  if (da + a->c > sw || db + b->c > sw) return false;
  return da + a->c <= db || db + b->c <= da;
}

bool overlap(const cb_tensor* a, const cb_tensor* b) {
  if (a->n == 0 || b->n == 0) return false;
  uintptr_t alo, ahi, blo, bhi;
  view_range(a, &alo, &ahi);
  view_range(b, &blo, &bhi);
  if (!(alo < bhi && blo < ahi)) return false;
  return !disjoint_channel_slices(a, b);
}

bool same_view(const cb_tensor* a, const cb_tensor* b) {
  return a->data == b->data && a->n == b->n && a->h == b->h && a->w == b->w && a->c == b->c &&
         a->stride_n == b->stride_n && a->stride_h == b->stride_h && a->stride_w == b->stride_w &&
         a->stride_c == b->stride_c && a->layout == b->layout && a->dtype == b->dtype;
}

bool strides_mult4(const cb_tensor* t) {
  return t->stride_n % 4 == 0 && t->stride_h % 4 == 0 && t->stride_w % 4 == 0;
}

Epilogue make_epilogue(const float* scale, const float* bias, cb_act act, const cb_tensor* r, cb_res_mode mode) {
  Epilogue e{};
  e.scale = scale;
  e.bias = bias;
  e.act = static_cast<int>(act);
  e.res_mode = static_cast<int>(mode);
  if (mode != CB_RES_NONE) {
    e.r = static_cast<const float*>(r->data);
    e.rs_n = r->stride_n;
    e.rs_h = r->stride_h;
    e.rs_w = r->stride_w;
  }
  return e;
}

OutView make_out(const cb_tensor* y) {
  OutView o{};
  o.y = static_cast<float*>(y->data);
  o.ys_n = y->stride_n;
  o.ys_h = y->stride_h;
  o.ys_w = y->stride_w;
  return o;
}

// Which dense layers go to the tensor cores.  A 3x3 layer with under 16
// input channels runs faster on the CUDA-core direct kernel: on the im2col
// path it spends nine narrow gathers per tile (an SM completes about one
// copy per 400-700 cycles), and a halo tile of 8-channel rows over a wide
// image moves four 32-byte rows per output pixel (measured on 8 -> 8 at
// 320x320: 457 us against 155 us direct).  1x1 layers take the tensor cores
// from 8 channels on.
bool tc_channels_ok(int ci, int k, int stride) {
  (void)stride;
  return k == 1 ? ci >= 8 : ci >= 16;
}

// ----------------------------------------------------------- tuning overrides
// Constraints on a halo plan (0 / false = free): tile shape, ring depth,
// split K, taps per weight stage.
struct HaloForce {
  int co = 0;
  bool cm = false;
  int px = 0;  // channel-major pixels per tile (256 or 192; 0: either)
  int nb = 0, split = 0, tps = 0, sub = 0;
  int res = -1;  // resident weights: -1 the model's choice, 0 off, 1 on
};

// Plan overrides and profiling aids (none is needed for normal use).  Each
// starts from the environment variable of the same name, read once per
// process on first use; afterwards only cb_set_tuning changes it.  The hot
// path never calls getenv, and a test can switch plans without writing to
// the environment of a live process.
struct Tuning {
  int dw_force[3] = {0, 0, 0};     // CB_DW_FORCE = "rows,tile_w,ctas_per_sm" (0 = free)
  int igemm_force[3] = {0, 0, 0};  // CB_IGEMM_FORCE = "bn,stages,grid"
  int igemm_blocks = -1;           // CB_IGEMM_BLOCKS = 0 / 1 (-1: the planner's choice)
  HaloForce halo;                  // CB_HALO_FORCE = "cm[,stages[,split[,taps]]]" or
                                   //   "co[,stages[,split[,taps[,subtiles[,resident]]]]]"
  int dw_block = -1;               // CB_DW_BLOCK_FORCE = 0 / 1 (-1: the shape rule)
  bool debug_plan = false;         // CB_DEBUG_PLAN: print each plan to stderr
  int trace_cta = -1;              // CB_IGEMM_TRACE = cta (trace builds: timeline of one CTA)
  int span_slot = 1;               // CB_SPAN_SLOT = 1 / 2 (trace builds)
  int timeout_ms = 2000;           // CB_TIMEOUT_MS: bound of every device wait
  int dw_skip_row = 0;             // CB_DEBUG_DW_SKIP_ROW = 1: fault injection (see cb_set_tuning)
  int stem_kernel = 0;             // CB_STEM_KERNEL = "cuda" / "tc" (0: tensor cores for NHWC input)
  int stage_skip_x = 0;            // CB_DEBUG_STAGE_SKIP_X = 1: fault injection (see cb_set_tuning)
};

const char* const kTuningNames[] = {"CB_DW_FORCE",    "CB_IGEMM_FORCE", "CB_IGEMM_BLOCKS", "CB_HALO_FORCE",
                                    "CB_DW_BLOCK_FORCE", "CB_DEBUG_PLAN", "CB_IGEMM_TRACE", "CB_SPAN_SLOT",
                                    "CB_TIMEOUT_MS",  "CB_DEBUG_DW_SKIP_ROW", "CB_STEM_KERNEL",
                                    "CB_DEBUG_STAGE_SKIP_X"};

// Sets knob `name` of *t from `v` (NULL or "" restores the knob's default);
// false for an unknown name.
bool parse_tuning(Tuning* t, const char* name, const char* v) {
  const Tuning d;
  const bool unset = v == nullptr || v[0] == '\0';
  if (!std::strcmp(name, "CB_DW_FORCE")) {
    std::memcpy(t->dw_force, d.dw_force, sizeof(d.dw_force));
    if (!unset) std::sscanf(v, "%d,%d,%d", &t->dw_force[0], &t->dw_force[1], &t->dw_force[2]);
  } else if (!std::strcmp(name, "CB_IGEMM_FORCE")) {
    std::memcpy(t->igemm_force, d.igemm_force, sizeof(d.igemm_force));
    if (!unset) std::sscanf(v, "%d,%d,%d", &t->igemm_force[0], &t->igemm_force[1], &t->igemm_force[2]);
  } else if (!std::strcmp(name, "CB_IGEMM_BLOCKS")) {
    t->igemm_blocks = unset ? d.igemm_blocks : (v[0] == '1' ? 1 : 0);
  } else if (!std::strcmp(name, "CB_HALO_FORCE")) {
    HaloForce f;
    if (!unset) {
      if (v[0] == 'c' && v[1] == 'm') {
        // "cm[PX][,nb,split,tps]"
        f.cm = true;
        const char* r = v + 2;
        if (*r >= '0' && *r <= '9') f.px = static_cast<int>(std::strtol(r, const_cast<char**>(&r), 10));
        if (*r == ',') std::sscanf(r + 1, "%d,%d,%d", &f.nb, &f.split, &f.tps);
      } else {
        std::sscanf(v, "%d,%d,%d,%d,%d,%d", &f.co, &f.nb, &f.split, &f.tps, &f.sub, &f.res);
      }
    }
    t->halo = f;
  } else if (!std::strcmp(name, "CB_DW_BLOCK_FORCE")) {
    t->dw_block = unset ? d.dw_block : (v[0] == '1' ? 1 : 0);
  } else if (!std::strcmp(name, "CB_DEBUG_PLAN")) {
    t->debug_plan = !unset;
  } else if (!std::strcmp(name, "CB_IGEMM_TRACE")) {
    t->trace_cta = unset ? d.trace_cta : std::atoi(v);
  } else if (!std::strcmp(name, "CB_SPAN_SLOT")) {
    t->span_slot = unset ? d.span_slot : (std::atoi(v) == 2 ? 2 : 1);
  } else if (!std::strcmp(name, "CB_TIMEOUT_MS")) {
    const int ms = unset ? 0 : std::atoi(v);
    t->timeout_ms = ms > 0 ? ms : d.timeout_ms;
  } else if (!std::strcmp(name, "CB_DEBUG_DW_SKIP_ROW")) {
    t->dw_skip_row = unset ? 0 : (std::atoi(v) != 0 ? 1 : 0);
  } else if (!std::strcmp(name, "CB_DEBUG_STAGE_SKIP_X")) {
    t->stage_skip_x = unset ? 0 : (std::atoi(v) != 0 ? 1 : 0);
  } else if (!std::strcmp(name, "CB_STEM_KERNEL")) {
    t->stem_kernel = unset ? 0 : !std::strcmp(v, "cuda") ? 1 : !std::strcmp(v, "tc") ? 2 : 0;
  } else {
    return false;
  }
  return true;
}

std::mutex g_tuning_mu;
Tuning* g_tuning = nullptr;  // guarded by g_tuning_mu; created from the environment on first use

Tuning& tuning_locked() {
  if (!g_tuning) {
    static Tuning t;
    for (const char* n : kTuningNames) parse_tuning(&t, n, std::getenv(n));
    g_tuning = &t;
  }
  return *g_tuning;
}

// A copy of the current overrides (a few dozen bytes under an uncontended lock).
Tuning tuning() {
  std::lock_guard<std::mutex> lock(g_tuning_mu);
  return tuning_locked();
}

uint64_t timeout_ns() { return static_cast<uint64_t>(tuning().timeout_ms) * 1000000ull; }

// ----------------------------------------------------------------- depthwise
cb_status run_depthwise(const cb_tensor* x, const float* w, const Epilogue& ep, int stride, int pad,
                        const cb_tensor* y, cudaStream_t s) {
  DeviceInfo* dev = nullptr;
  cb_status st = current_device(&dev);
  if (st != CB_OK) return st;
  DwArgs a{};
  a.x = static_cast<const float*>(x->data);
  a.xs_n = x->stride_n;
  a.xs_h = x->stride_h;
  a.xs_w = x->stride_w;
  a.w = w;
  a.N = x->n;
  a.H = x->h;
  a.W = x->w;
  a.C = x->c;
  a.OH = y->h;
  a.OW = y->w;
  a.stride = stride;
  a.pad = pad;
  a.out = make_out(y);
  a.ep = ep;
  a.bf16 = x->dtype == CB_DTYPE_BF16 ? 1 : 0;
  const int policy = g_policy.load();
  if (a.bf16) {
    // bf16 storage: the TMA kernel only (16-byte pixel rows of 8 channels)
    auto mult8 = [](const cb_tensor* t) { return t->stride_n % 8 == 0 && t->stride_h % 8 == 0 && t->stride_w % 8 == 0; };
    if (a.C % 8 != 0 || !aligned16(a.x) || !aligned16(w) || !aligned16(ep.scale) || !aligned16(ep.bias) ||
        !aligned16(a.out.y) || !mult8(x) || !mult8(y) ||
        (ep.res_mode != 0 && (!aligned16(ep.r) || ep.rs_n % 8 != 0 || ep.rs_h % 8 != 0 || ep.rs_w % 8 != 0)))
      return CB_ERR_ALIGNMENT;
    if (policy == 1 || encode_tiled() == nullptr) return CB_ERR_UNSUPPORTED;
  }
  const bool vec = a.C % 4 == 0 && aligned16(a.x) && aligned16(w) && aligned16(ep.scale) && aligned16(ep.bias) &&
                   aligned16(a.out.y) && strides_mult4(x) && strides_mult4(y) &&
                   (ep.res_mode == 0 || (aligned16(ep.r) && ep.rs_n % 4 == 0 && ep.rs_h % 4 == 0 && ep.rs_w % 4 == 0));
  const bool tma_ok = vec && policy != 1 && encode_tiled() != nullptr && a.OW >= 1;
  if (!tma_ok) {
    cudaError_t e = launch_dw_simple(a, vec, s);
    return e == cudaSuccess ? CB_OK : cuda_fail(e);
  }

  // Plan.  Output-column tiles of at most 120 columns (fp32: 8 consumer
  // threads per column pair; bf16: 16 threads per group of 4 columns at
  // stride 1, of 2 columns (tiles of 60) at stride 2), 128-byte
  // chunks of each pixel (32 fp32 or 64 bf16 channels: an SM completes its
  // row copies one after another, so the copy count, not their bytes, sets
  // the pace) and short strips of output rows: measured on the
  // 64x56x56x384 layer, 4-row strips with two CTAs per SM beat longer
  // strips (which stage fewer halo rows) by 10-15%, because the CTAs in
  // flight then cover a narrow band of rows whose halos hit in L2.  Strips
  // shrink further when a layer has too few items to fill the GPU.
  const int ch = a.bf16 ? 64 : 32, tpp = ch / 4;
  const int cols = a.bf16 && stride == 1 ? 4 : 2;  // output columns per consumer thread (the kernel's rule)
  const int max_tile = a.bf16 && stride == 2 ? 60 : 120;  // at most 480 consumer threads
  const int chunks = (a.C + ch - 1) / ch;
  // Tuning override (CB_DW_FORCE="rows,tile_w,ctas_per_sm"; 0 = free).
  const Tuning tu = tuning();
  const int force_r = tu.dw_force[0], force_tw = tu.dw_force[1], force_cps = tu.dw_force[2];
  DwTmaPlan best{};
  {
    const int wt = (a.OW + max_tile - 1) / max_tile;
    const int tile_w = force_tw > 0 ? std::min({force_tw, a.OW, max_tile}) : (a.OW + wt - 1) / wt;
    const int wtiles = (a.OW + tile_w - 1) / tile_w;
    const int groups = (tile_w + cols - 1) / cols;
    const int box_w = (cols * groups - 1) * stride + 3;  // every column of the last group is covered
    const int consumer_warps = (groups * tpp + 31) / 32;
    const int threads = 32 * (1 + consumer_warps);
    int cps = dw_tma_blocks_per_sm(stride, threads, 96 * 1024, a.bf16 != 0) >= 2 ? 2 : 1;
    if (force_cps == 1 || force_cps == 2) cps = force_cps;
    const int stage_bytes = box_w * 128;  // a ring slot: one row of 128-byte pixel chunks
    // four-column threads read the taps from shared memory when they fit
    const size_t w_bytes = cols == 4 && 36ull * a.C <= 48 * 1024 ? 36ull * a.C : 0;
    const size_t ring = (cps == 2 ? 96 * 1024 : 192 * 1024) - w_bytes;
    const int stages = static_cast<int>(std::min<size_t>(32, ring / stage_bytes));
    const int cap = dev->sms * cps;
    // bf16 at stride 1: 8-row strips (the kernel is bound by its instruction
    // issue there, and a longer strip re-reads fewer halo rows per output row)
    int R = force_r > 0 ? std::min(force_r, a.OH) : std::min(a.OH, a.bf16 && stride == 1 ? 8 : 4);
    auto items_for = [&](int r) {
      return static_cast<long long>(a.N) * chunks * wtiles * ((a.OH + r - 1) / r);
    };
    while (force_r <= 0 && R > 1 && items_for(R) < 2LL * cap) --R;
    const long long items = items_for(R);
    if (box_w <= 256 && stages >= 3 && items <= (1LL << 30)) {
      best.rows_per_item = R;
      best.num_items = static_cast<int>(items);
      best.tile_w = tile_w;
      best.box_w = box_w;
      best.stages = stages;
      best.grid = static_cast<int>(std::min<long long>(items, cap));
      best.consumer_warps = consumer_warps;
      best.w_smem = w_bytes ? 1 : 0;
      best.smem_bytes = static_cast<size_t>(stages) * stage_bytes + 2 * stages * sizeof(uint64_t) + 16 + w_bytes;
    }
  }
  if (tu.debug_plan)
    std::fprintf(stderr, "[cb] dw plan: N=%d H=%d W=%d C=%d s=%d -> rows=%d items=%d box_w=%d stages=%d grid=%d warps=%d smem=%zu\n",
                 a.N, a.H, a.W, a.C, stride, best.rows_per_item, best.num_items, best.box_w, best.stages, best.grid,
                 best.consumer_warps, best.smem_bytes);
  if (best.grid == 0) {
    if (a.bf16) return CB_ERR_UNSUPPORTED;
    cudaError_t e = launch_dw_simple(a, vec, s);
    return e == cudaSuccess ? CB_OK : cuda_fail(e);
  }
  CUtensorMap map;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(a.C), static_cast<cuuint64_t>(a.W), static_cast<cuuint64_t>(a.H),
                        static_cast<cuuint64_t>(a.N)};
  const cuuint64_t eb = a.bf16 ? 2 : 4;
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(a.xs_w) * eb, static_cast<cuuint64_t>(a.xs_h) * eb,
                           static_cast<cuuint64_t>(a.xs_n) * eb};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(ch), static_cast<cuuint32_t>(best.box_w), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = tiled_map(&map, 4, a.x, dims, strides, box, estr, CU_TENSOR_MAP_SWIZZLE_NONE,
                         a.bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
  if (r != CUDA_SUCCESS) {
    if (a.bf16) return CB_ERR_UNSUPPORTED;
    cudaError_t e = launch_dw_simple(a, vec, s);
    return e == cudaSuccess ? CB_OK : cuda_fail(e);
  }
  cudaError_t e = launch_dw_tma(map, a, best, dev->err, static_cast<uint64_t>(tu.timeout_ms) * 1000000ull,
                                tu.dw_skip_row, s);
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

// -------------------------------------------------------------------- dense
struct HaloPlan {
  int px = 0, co = 0;  // tile: px pixels x co output channels
  bool cm = false;     // channel-major accumulator (px = 256 or 192, co = 128)
  int nb = 0, grid = 0;
  int split = 1;       // 2: clusters of two CTAs split each tile's channel chunks
  int tps = 1;         // filter taps per weight-ring stage (one copy per stage)
  int kc = 32;         // input channels per chunk (32, or 16 for Ci % 32 == 16 and for stride 2)
  int stride = 1;      // 2: four phase tiles per chunk
  int blk_w = 0, n_blk = 1, wp = 0;  // column blocks and the padded width of the pixel numbering
  int sub = 1;
  bool resident = false;  // weights loaded once per CTA (one chunk, one channel tile)
  int eb = 4;             // bytes per element of x, w and y: 4 (fp32, TF32 MMAs) or 2 (bf16)
  size_t smem = 0;
  double cost = 0;     // the cost model's cycles per CTA
};
struct ImPlan {        // im2col kernel choices (0 = the cost model's)
  int bn = 0, stages = 0;
  int blocks = 0;      // 1: 128 consecutive pixels (im2col copies); 2: pixel blocks (tiled copies)
};
bool plan_halo(const cb_tensor* x, const cb_tensor* y, int stride, int sms, const HaloForce& f, HaloPlan* out);

// ------------------------------------------------------------ autotuner
// Plans measured by cb_autotune_conv, per layer shape (and device, policy):
// they override the cost models for that shape.  The tuner only chooses
// among kernels of the path's own arithmetic class (tensor-core variants for
// a tensor-core layer), so cb_layer_uses_tensor_cores stays true.
struct ConvPlan {
  cb_path path = CB_PATH_DIRECT;
  HaloPlan halo;
  ImPlan im;
};
struct ConvKey {
  int dev, policy, n, h, w, ci, co, kh, stride, pad, dtype;
  bool operator==(const ConvKey& o) const { return std::memcmp(this, &o, sizeof(ConvKey)) == 0; }
};
struct ConvKeyHash {
  size_t operator()(const ConvKey& k) const {
    uint64_t h = 1469598103934665603ull;
    const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
    for (size_t i = 0; i < sizeof(ConvKey); ++i) h = (h ^ p[i]) * 1099511628211ull;
    return static_cast<size_t>(h);
  }
};
std::mutex g_tune_mu;
std::unordered_map<ConvKey, ConvPlan, ConvKeyHash> g_tuned;

ConvKey conv_key(const cb_tensor* x, const cb_tensor* y, int kh, int stride, int pad) {
  ConvKey k;
  std::memset(&k, 0, sizeof(k));
  cudaGetDevice(&k.dev);
  k.policy = g_policy.load();
  k.n = x->n, k.h = x->h, k.w = x->w, k.ci = x->c, k.co = y->c, k.kh = kh, k.stride = stride, k.pad = pad;
  k.dtype = static_cast<int>(x->dtype);
  return k;
}

bool tuned_plan(const ConvKey& k, ConvPlan* out) {
  std::lock_guard<std::mutex> lock(g_tune_mu);
  auto it = g_tuned.find(k);
  if (it == g_tuned.end()) return false;
  *out = it->second;
  return true;
}

// Kernel for a dense (groups 1) layer under the current policy; fills
// *plan for the halo kernel and *im for the im2col kernel (a measured plan
// for the shape, when the tuner made one, else the cost models').
cb_path dense_path(const cb_tensor* x, const cb_tensor* y, int kh, int stride, int pad, HaloPlan* plan,
                   ImPlan* im = nullptr);

// Pixel blocks of bw x bh = 128 output pixels for the tiled-copy A operand:
// the shape that covers OH x OW with the fewest wasted rows (*waste = covered
// / real pixels); stride * bw and stride * bh stay within a copy box (256).
void pick_blocks(int OH, int OW, int stride, int* bw_out, int* bh_out, double* waste) {
  double best = 1e300;
  for (int bw = 128; bw >= 1; bw >>= 1) {
    const int bh = 128 / bw;
    if (stride * bw > 256 || stride * bh > 256) continue;
    const double cov = static_cast<double>((OW + bw - 1) / bw) * bw * static_cast<double>((OH + bh - 1) / bh) * bh;
    const double w = cov / (static_cast<double>(OW) * OH);
    if (w < best - 1e-9) {
      best = w;
      *bw_out = bw;
      *bh_out = bh;
    }
  }
  *waste = best;
}

int pick_bn(int M, int Cout, int k_iters, int sms, int* n_tiles_out) {
  static const int kBn[] = {16, 32, 48, 64, 96, 128, 192, 256};
  const int m_tiles = (M + 127) / 128;
  double best = 1e300;
  int best_bn = 16, best_nt = (Cout + 15) / 16;
  for (int bn : kBn) {
    const int n_tiles = (Cout + bn - 1) / bn;
    if (n_tiles > 1 && bn < 64 && Cout > 256) continue;
    const long long tiles = static_cast<long long>(m_tiles) * n_tiles;
    const long long waves = (tiles + sms - 1) / sms;
    // per k-step: smem operand bytes / 128 B per clock vs tensor work (M=128, K=32, N=bn)
    const double step = std::max(128.0 + bn, 2.2 * bn);
    const double epi = 2.0 * bn;  // epilogue cycles per tile, roughly
    const double cost = static_cast<double>(waves) * (k_iters * step + epi);
    if (cost < best - 1e-9) {
      best = cost;
      best_bn = bn;
      best_nt = n_tiles;
    }
  }
  *n_tiles_out = best_nt;
  return best_bn;
}

cb_status run_igemm(const cb_tensor* x, const float* w, const Epilogue& ep, int k, int stride, int pad,
                    const cb_tensor* y, cudaStream_t s, const ImPlan& im = ImPlan{}) {
  DeviceInfo* dev = nullptr;
  cb_status st = current_device(&dev);
  if (st != CB_OK) return st;
  const int Ci = x->c, Co = y->c;
  IgemmArgs a{};
  a.M = x->n * y->h * y->w;
  a.OHW = y->h * y->w;
  a.OW = y->w;
  a.Cout = Co;
  a.kw = k;
  a.taps = k * k;
  // K step rows of kc x 4 bytes: kc fp32 or 2 kc bf16 channels (no padding
  // channels for 8 / 16-channel fp32 or 16 / 32-channel bf16 layers)
  const int eb = is_f32(x) ? 4 : 2, cpu = 4 / eb;
  const int kc = Ci <= 8 * cpu ? 8 : (Ci <= 16 * cpu ? 16 : 32);
  const int chan = kc * cpu;
  a.num_kc = (Ci + chan - 1) / chan;
  a.bf16 = eb == 2 ? 1 : 0;
  a.k_iters = a.taps * a.num_kc;
  a.stride = stride;
  a.pad = pad;
  a.out = make_out(y);
  a.ep = ep;
  a.err = dev->err;
  a.timeout_ns = timeout_ns();
  const Tuning tu = tuning();
  if (tu.trace_cta >= 0) {  // profiling aid: timeline of one CTA
    a.trace = 1;
    a.trace_cta = tu.trace_cta;
  }
  a.vec_store = (aligned16(a.out.y) && strides_mult4(y) && aligned16(ep.scale) && aligned16(ep.bias) &&
                 (ep.res_mode == 0 || (aligned16(ep.r) && ep.rs_n % 4 == 0 && ep.rs_h % 4 == 0 && ep.rs_w % 4 == 0)))
                    ? 1
                    : 0;
  int n_tiles = 1;
  int bn = pick_bn(a.M, Co, a.k_iters, dev->sms, &n_tiles);
  // Tuning override (a measured plan, else CB_IGEMM_FORCE="bn,stages,grid"; 0 = free).
  int force_bn = im.bn, force_stages = im.stages, force_grid = 0;
  if (im.bn == 0) force_bn = tu.igemm_force[0], force_stages = tu.igemm_force[1], force_grid = tu.igemm_force[2];
  if (force_bn == 16 || force_bn == 32 || force_bn == 48 || force_bn == 64 || force_bn == 96 || force_bn == 128 ||
      force_bn == 192 || force_bn == 256) {
    bn = force_bn;
    n_tiles = (Co + bn - 1) / bn;
  }
  // Pixel blocks (tiled copies, ~1 row per clock) unless they would waste
  // more than 15 % of the tile rows on the image edges; then 128 consecutive
  // pixels gathered in im2col mode.  CB_IGEMM_BLOCKS=0/1 overrides.
  int bw = 0, bh = 0;
  double waste = 1e300;
  pick_blocks(y->h, y->w, stride, &bw, &bh, &waste);
  int blocks = im.blocks;
  if (blocks == 0) {
    blocks = waste <= 1.15 ? 2 : 1;
    if (tu.igemm_blocks >= 0) blocks = tu.igemm_blocks == 1 ? 2 : 1;
  }
  if (blocks == 2 && bw > 0) {
    a.blk_w = bw;
    a.blk_h = bh;
    a.blocks_x = (y->w + bw - 1) / bw;
    a.blocks_y = (y->h + bh - 1) / bh;
    const long long mt = static_cast<long long>(x->n) * a.blocks_x * a.blocks_y;
    if (mt >= (1LL << 31)) return CB_ERR_UNSUPPORTED;
    a.m_tiles = static_cast<int>(mt);
  } else {
    a.m_tiles = (a.M + 127) / 128;
  }
  a.n_tiles = n_tiles;
  a.stages = igemm_stages(bn, kc);
  if (force_stages >= 2 && igemm_smem_bytes(bn, kc, force_stages) <= 227 * 1024) a.stages = force_stages;
  const size_t smem = igemm_smem_bytes(bn, kc, a.stages);
  const long long tiles = static_cast<long long>(a.m_tiles) * a.n_tiles;
  int grid = static_cast<int>(std::min<long long>(tiles, dev->sms));
  if (force_grid > 0 && force_grid < grid) grid = force_grid;
  if (tu.debug_plan)
    std::fprintf(stderr,
                 "[cb] igemm plan: M=%d Ci=%d Co=%d k=%d s=%d -> bn=%d kc=%d n_tiles=%d m_tiles=%d stages=%d grid=%d "
                 "blocks=%dx%d\n",
                 a.M, Ci, Co, k, stride, bn, kc, n_tiles, a.m_tiles, a.stages, grid, a.blk_h, a.blk_w);

  CUtensorMap amap, bmap;
  const CUtensorMapDataType dt = eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const CUtensorMapSwizzle swz = kc == 32 ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : kc == 16 ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_32B;
  {
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(Ci), static_cast<cuuint64_t>(x->w), static_cast<cuuint64_t>(x->h),
                          static_cast<cuuint64_t>(x->n)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(x->stride_w) * eb, static_cast<cuuint64_t>(x->stride_h) * eb,
                             static_cast<cuuint64_t>(x->stride_n) * eb};
    int lower[2] = {-pad, -pad};
    int upper[2] = {pad - (k - 1), pad - (k - 1)};
    cuuint32_t estr[4] = {1, static_cast<cuuint32_t>(stride), static_cast<cuuint32_t>(stride), 1};
    CUresult r;
    if (a.blk_w) {
      cuuint32_t box[4] = {static_cast<cuuint32_t>(chan), static_cast<cuuint32_t>(stride * a.blk_w),
                           static_cast<cuuint32_t>(stride * a.blk_h), 1};
      r = tiled_map(&amap, 4, x->data, dims, strides, box, estr, swz, dt);
    } else {
      r = im2col_map(&amap, x->data, dims, strides, lower, upper, static_cast<cuuint32_t>(chan), 128, estr, swz, dt);
    }
    if (r != CUDA_SUCCESS) return CB_ERR_UNSUPPORTED;
  }
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(Ci), static_cast<cuuint64_t>(k * k), static_cast<cuuint64_t>(Co)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(Ci) * eb, static_cast<cuuint64_t>(k * k) * Ci * eb};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(chan), 1, static_cast<cuuint32_t>(bn)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = tiled_map(&bmap, 3, w, dims, strides, box, estr, swz, dt);
    if (r != CUDA_SUCCESS) return CB_ERR_UNSUPPORTED;
  }
  cudaError_t e = launch_igemm(amap, bmap, a, bn, kc, grid, smem, s);
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

// 3x3 stride-1 pad-1 layers with Cin % 32 == 0 and an image width whose
// halo tile leaves room for a weight ring: the halo-tile kernel.
// Weight ring of a halo tile shape: the most filter taps per stage (9, 3 or
// 1) that leaves at least two stages (three for single taps) in shared memory.
// An SM completes about one copy per 400-700 cycles whatever its size up to
// ~48 KB (measured), so fewer, larger weight copies keep the MMAs fed.
bool halo_ring(int co, int hb, int force_nb, int force_tps, int* nb_out, int* tps_out, int kc = 32) {
  constexpr size_t kSmemMax = 227 * 1024;
  for (int tps : {9, 3, 1}) {
    if (force_tps && tps != force_tps) continue;
    const int nb_max = force_nb >= 2 ? std::min(force_nb, 16) : (tps == 1 ? 8 : 4);
    int nb = nb_max;
    while (nb >= 2 && halo_smem_bytes(co, hb, nb, tps, kc) > kSmemMax) --nb;
    if (nb >= ((force_nb >= 2 || tps > 1) ? 2 : 3)) {
      *nb_out = nb;
      *tps_out = tps;
      return true;
    }
  }
  return false;
}


bool plan_halo(const cb_tensor* x, const cb_tensor* y, int stride, int sms, const HaloForce& f, HaloPlan* out) {
  const int N = x->n, Ci = x->c, Co = y->c, OH = y->h, OW = y->w;
  // 32-channel chunks (128-byte rows); 16-channel chunks (64-byte rows) for
  // Ci % 32 == 16 and at stride 2 (four phase tiles per chunk), in the
  // pixel-major 128 x {32, 64, 128} tiles
  // kc counts a chunk's pixel row in 4-byte units (32: 128-byte rows): kc
  // fp32 channels, or 2 kc bf16 channels
  const int eb = is_f32(x) ? 4 : 2;
  const int cpu = 4 / eb;  // channels per 4-byte unit
  // (bf16 at stride 2 may take 32-byte rows too: 16-channel layers)
  const int kc = (stride == 1 && Ci % (32 * cpu) == 0)          ? 32
                 : Ci % (16 * cpu) == 0                         ? 16
                 : ((stride == 1 || eb == 2) && Ci % (8 * cpu) == 0) ? 8
                                                                  : 0;
  if (kc == 0) return false;
  const int num_kc = Ci / (kc * cpu);
  constexpr size_t kSmemMax = 227 * 1024;
  struct Shape {
    int px, co;
    bool cm;
  };
  static const Shape kShapes[] = {{256, 128, true}, {192, 128, true}, {128, 256, false}, {128, 128, false}, {128, 64, false},
                                  {128, 32, false}};
  // Column blocks: the padded width of the pixel numbering must fit a copy
  // box (256 elements traversed: blk_w + 2 at stride 1, 2 (blk_w + 1) at
  // stride 2); more blocks shrink the halo when it does not fit.
  const int max_blk = stride == 1 ? 254 : 127;
  const int min_blocks = (OW + max_blk - 1) / max_blk;
  double best = 1e300;
  HaloPlan plan;
  for (const Shape& sh : kShapes) {
    if (f.cm && !sh.cm) continue;
    if (f.px && sh.cm && sh.px != f.px) continue;
    if (f.co && (sh.cm || sh.co != f.co)) continue;
    if (kc == 16 && (sh.cm || sh.co > 128)) continue;
    if (kc == 16 && sh.co == 128 && stride == 1) continue;
    if (kc == 8 && (sh.cm || sh.co != 32)) continue;
    for (int sub = 1; sub <= kHaloMaxSub; sub *= 2) {
      if (f.sub && sub != f.sub) continue;
      if (sub > 1 && (sh.cm || sh.co > 64)) continue;
      for (int n_blk = min_blocks; n_blk <= min_blocks + 3 && n_blk <= OW; ++n_blk) {
        const int blk_w = (OW + n_blk - 1) / n_blk;
        const int wp = blk_w + (stride == 1 ? 2 : 1);
        const int rows = halo_rows(wp, sh.px * sub, stride);
        if (rows * stride > 256) continue;
        const int hb = halo_buffer_bytes(wp, sh.px * sub, kc, stride);
        int nb = 0, tps = 1;
        // Resident weights: a layer of one channel chunk and one channel tile
        // may keep its nine taps in a single stage, copied once per CTA; each
        // tile then costs its MMAs (one stage) against its halo copy alone.
        const bool res_ok = num_kc == 1 && Co <= sh.co && f.res != 0 && (f.split == 0 || f.split == 1) &&
                            (f.tps == 0 || f.tps == 9) && (f.nb == 0 || f.nb == 1) &&
                            halo_smem_bytes(sh.co, hb, 1, 9, kc) <= kSmemMax;
        const bool ring_ok = f.res != 1 && halo_ring(sh.co, hb, f.nb, f.tps, &nb, &tps, kc);
        if (!ring_ok && !res_ok) continue;
        const long long px_tiles = (static_cast<long long>(OH) * wp + sh.px - 1) / sh.px;
        const long long m_tiles = static_cast<long long>(N) * n_blk * ((px_tiles + sub - 1) / sub);
        const long long tiles = m_tiles * ((Co + sh.co - 1) / sh.co);
        if (tiles >= (1LL << 31)) continue;
        const long long grid = std::min<long long>(tiles, sms);
        const long long per_cta = (tiles + grid - 1) / grid;
        // Cycles, fitted to forced-plan timings of the dense-sweep and
        // YOLO-chain 3x3 layers (mean regret of the pick 3.5 %).  Per
        // (tile, chunk) the larger of: the MMAs (nine taps of kc / 8 per
        // sub-tile, ~64 cycles each up to N = 128, in proportion above)
        // plus ~200 cycles per weight stage (~130 more per extra sub-tile);
        // and the copies (~200 per halo copy, four at stride 2; ~280 per
        // weight copy, plus bytes).  Per tile ~3500 cycles of pipeline fill,
        // unless the epilogue (~0.37 cycles per output element of the tile)
        // is slower; plus one exposed epilogue.
        const int n = sh.cm ? sh.px : sh.co;
        const double mma = sub * 9.0 * (kc / 8) * 64.0 * std::max(1.0, n / 128.0) +
                           (9.0 / tps) * (204.0 + 128.0 * (sub - 1));
        const double wcopy = 279.0 + 0.013 * tps * sh.co * kc * 4;
        const double hcopy = (stride == 1 ? 1.0 : 4.0) * 199.0 + 0.0016 * hb;
        const double copy = hcopy + 9.0 / tps * wcopy;
        const double epi = 0.444 * sh.px * sh.co;
        const double epi_tile = 0.374 * sub * sh.px * sh.co;
        const size_t smem = halo_smem_bytes(sh.co, hb, nb, tps, kc);
        if (res_ok) {
          const size_t smem_r = halo_smem_bytes(sh.co, hb, 1, 9, kc);
          {
            const double mma_r = sub * 9.0 * (kc / 8) * 64.0 * std::max(1.0, n / 128.0) + 204.0;
            double cost = static_cast<double>(per_cta) * std::max(std::max(mma_r, hcopy) + 3546.0, epi_tile) + epi;
            cost *= 1.0 + 0.02 * (n_blk - min_blocks);
            if (cost < best * 0.97) {
              best = cost;
              plan.px = sh.px;
              plan.co = sh.co;
              plan.cm = sh.cm;
              plan.nb = 1;
              plan.tps = 9;
              plan.kc = kc;
              plan.stride = stride;
              plan.blk_w = blk_w;
              plan.n_blk = n_blk;
              plan.wp = wp;
              plan.sub = sub;
              plan.split = 1;
              plan.resident = true;
              plan.grid = static_cast<int>(grid);
              plan.smem = smem_r;
              plan.cost = cost;
            }
          }
        }
        for (int split = 1; ring_ok && split <= 2; ++split) {
          if (f.split && split != f.split) continue;
          double cost;
          if (split == 1) {
            cost = static_cast<double>(per_cta) * std::max(num_kc * std::max(mma, copy) + 3546.0, epi_tile) + epi;
          } else {
            // one tile per CTA pair, each CTA half of the chunks; the partner's
            // half accumulator comes over distributed shared memory (~16 B per
            // clock) and each CTA stores half the tile
            const size_t recv = halo_split_recv_bytes(sh.px, sh.co, sh.cm);
            if (sub != 1 || stride != 1 || kc != 32 || num_kc < 2 || (!sh.cm && sh.co < 64) ||
                recv > 2 * static_cast<size_t>(hb) + nb * tps * sh.co * 128ull || 2 * tiles > sms ||
                halo_max_pairs(sh.px, sh.co, sh.cm, smem) < tiles)
              continue;
            cost = (num_kc - num_kc / 2) * std::max(mma, copy) + 3546.0 + recv / 16.0 + 1000.0 + epi / 2;
          }
          cost *= 1.0 + 0.02 * (n_blk - min_blocks);  // fewer blocks: less halo overlap
          if (cost < best * 0.97) {
            best = cost;
            plan.px = sh.px;
            plan.co = sh.co;
            plan.cm = sh.cm;
            plan.nb = nb;
            plan.tps = tps;
            plan.kc = kc;
            plan.stride = stride;
            plan.blk_w = blk_w;
            plan.n_blk = n_blk;
            plan.wp = wp;
            plan.sub = sub;
            plan.resident = false;
            plan.split = split;
            plan.grid = static_cast<int>(split == 2 ? 2 * tiles : grid);
            plan.smem = smem;
            plan.cost = cost;
          }
        }
        break;  // the fewest blocks that fit
      }
    }
  }
  if (plan.px == 0) return false;
  plan.eb = eb;
  *out = plan;
  return true;
}

// A 1x1 stride-1 layer with at most 32 input and output channels: the
// streaming CUDA-core kernel (the tensor cores do less useful work per cycle
// at these widths, and the layer is HBM-bound).
bool pointwise_shape(int ci, int co, int kh, int stride, int pad) {
  return g_policy.load() != 1 && kh == 1 && stride == 1 && pad == 0 && pointwise_small_ok(ci, co);
}

// The 3 -> 16 stride-2 stem kernel: planar (NCHW) or packed NHWC input with
// 16-byte aligned rows of a multiple of 4 pixels, 16-byte aligned output.
bool stem_path(const cb_tensor* x, const cb_tensor* y, int kh, int stride, int pad) {
  if (g_policy.load() == 1 || x->c != 3 || y->c != 16 || kh != 3 || stride != 2 || pad != 1) return false;
  if (x->w % 4 != 0 || !aligned16(x->data) || !aligned16(y->data) || !strides_mult4(y)) return false;
  if (x->n > 65535 || static_cast<long long>(x->n) * ((y->h + 7) / 8) * ((y->w + 63) / 64) >= (1LL << 31))
    return false;
  if (!is_f32(x))  // bf16: packed NHWC, 16-byte groups of 8 pixels, 16-byte rows
    return x->layout == CB_LAYOUT_NHWC && x->stride_w == 3 && x->w % 8 == 0 && x->stride_n % 8 == 0 &&
           x->stride_h % 8 == 0;
  if (x->layout == CB_LAYOUT_NCHW)
    return x->stride_n % 4 == 0 && x->stride_h % 4 == 0 && x->stride_c % 4 == 0;
  return x->stride_w == 3 && x->stride_n % 4 == 0 && x->stride_h % 4 == 0;
}

// Shape rule of the tensor-core paths (views aside).
bool tc_shape(int ci, int co, int kh, int stride, int pad) {
  return g_policy.load() != 1 && ci % 4 == 0 && tc_channels_ok(ci, kh, stride) &&
         !pointwise_shape(ci, co, kh, stride, pad);
}

// bf16 storage on a dense layer: the pointwise kernel's 1x1 shapes with
// 16-byte aligned NHWC views; x is copied in 16-byte pieces (strides that
// are multiples of 8 elements), y written 4 channels (8 bytes) at a time
// (multiples of 4).
bool pointwise_bf16_views(const cb_tensor* x, const cb_tensor* y, int kh, int stride, int pad) {
  auto mult8 = [](const cb_tensor* t) { return t->stride_n % 8 == 0 && t->stride_h % 8 == 0 && t->stride_w % 8 == 0; };
  return g_policy.load() != 1 && kh == 1 && stride == 1 && pad == 0 && pointwise_small_ok(x->c, y->c, true) &&
         x->layout == CB_LAYOUT_NHWC && aligned16(x->data) && aligned16(y->data) && mult8(x) && strides_mult4(y);
}

// bf16 storage on the tensor cores (kind::f16 MMAs): the tensor-core shape
// rule with whole 16-byte rows per TMA element row (Ci % 8 == 0, x strides
// multiples of 8 elements), NHWC views with 16-byte aligned data, y strides
// multiples of 4 elements (8-byte stores of 4 channels).
bool tc_bf16_views(const cb_tensor* x, const cb_tensor* y, int kh, int stride, int pad) {
  auto mult8 = [](const cb_tensor* t) { return t->stride_n % 8 == 0 && t->stride_h % 8 == 0 && t->stride_w % 8 == 0; };
  return tc_shape(x->c, y->c, kh, stride, pad) && x->c % 8 == 0 && x->layout == CB_LAYOUT_NHWC &&
         aligned16(x->data) && mult8(x) && aligned16(y->data) && strides_mult4(y) && x->n <= 65535 &&
         x->w <= 65535 && x->h <= 65535 && encode_tiled() && encode_im2col();
}

// bf16 storage on the 8 -> 8 channel 3x3 stride-1 kernel (conv3x3_c8.cu):
// NHWC views, 16-byte aligned, x strides multiples of 8 elements (a pixel is
// one 16-byte piece), y strides multiples of 4.
bool c8_bf16_views(const cb_tensor* x, const cb_tensor* y, int kh, int stride, int pad) {
  auto mult8 = [](const cb_tensor* t) { return t->stride_n % 8 == 0 && t->stride_h % 8 == 0 && t->stride_w % 8 == 0; };
  return g_policy.load() != 1 && x->c == 8 && y->c == 8 && kh == 3 && stride == 1 && pad == 1 &&
         x->layout == CB_LAYOUT_NHWC && aligned16(x->data) && mult8(x) && aligned16(y->data) && strides_mult4(y);
}

cb_path dense_path(const cb_tensor* x, const cb_tensor* y, int kh, int stride, int pad, HaloPlan* plan, ImPlan* im) {
  const int policy = g_policy.load();
  if (!is_f32(x)) {
    if (pointwise_bf16_views(x, y, kh, stride, pad)) return CB_PATH_POINTWISE;
    if (stem_path(x, y, kh, stride, pad)) return CB_PATH_STEM;
    if (c8_bf16_views(x, y, kh, stride, pad)) return CB_PATH_DIRECT;
    if (!tc_bf16_views(x, y, kh, stride, pad)) return static_cast<cb_path>(0);
  }
  {
    // a measured plan for the shape, unless a plan override is set (an
    // explicit override wins over the tuner's table)
    const Tuning tu = tuning();
    const bool forced = tu.halo.co || tu.halo.cm || tu.halo.nb || tu.halo.split || tu.halo.tps || tu.halo.sub ||
                        tu.halo.res >= 0 || tu.igemm_force[0] || tu.igemm_blocks >= 0;
    ConvPlan cp;
    const bool tc_views = policy != 1 && x->layout == CB_LAYOUT_NHWC && aligned16(x->data) && strides_mult4(x) &&
                          x->n <= 65535 && x->w <= 65535 && x->h <= 65535 && encode_tiled() && encode_im2col();
    if (tc_views && !forced && tuned_plan(conv_key(x, y, kh, stride, pad), &cp) &&
        (cp.path == CB_PATH_TC_HALO || cp.path == CB_PATH_TC_HALO_CM || cp.path == CB_PATH_TC_IM2COL)) {
      if (plan) *plan = cp.halo;
      if (im) *im = cp.im;
      return cp.path;
    }
  }
  if (is_f32(x)) {
    if (stem_path(x, y, kh, stride, pad)) return CB_PATH_STEM;
    if (pointwise_shape(x->c, y->c, kh, stride, pad) && x->layout == CB_LAYOUT_NHWC && aligned16(x->data) &&
        strides_mult4(x) && aligned16(y->data) && strides_mult4(y))
      return CB_PATH_POINTWISE;
    const bool tc_ok = tc_shape(x->c, y->c, kh, stride, pad) && x->layout == CB_LAYOUT_NHWC &&
                       aligned16(x->data) && strides_mult4(x) && x->n <= 65535 && x->w <= 65535 &&
                       x->h <= 65535 && encode_tiled() && encode_im2col();
    if (!tc_ok) return CB_PATH_DIRECT;
  }
  if (policy == 0 && kh == 3 && pad == 1) {
    DeviceInfo* dev = nullptr;
    HaloPlan tmp;
    HaloPlan& p = plan ? *plan : tmp;
    const HaloForce f = tuning().halo;
    // Every 3x3 layer the halo tiles can take: they measured ahead of the
    // im2col-path kernel (two copies per tap and chunk) on each layer of
    // the dense sweep, stride 1 and 2.
    if (current_device(&dev) == CB_OK && plan_halo(x, y, stride, dev->sms, f, &p))
      return p.cm ? CB_PATH_TC_HALO_CM : CB_PATH_TC_HALO;
  }
  return CB_PATH_TC_IM2COL;
}

cb_status run_igemm_halo(const cb_tensor* x, const float* w, const Epilogue& ep, const HaloPlan& plan,
                         const cb_tensor* y, cudaStream_t s) {
  DeviceInfo* dev = nullptr;
  cb_status st = current_device(&dev);
  if (st != CB_OK) return st;
  const int Ci = x->c, Co = y->c;
  HaloArgs a{};
  a.H = x->h;
  a.W = x->w;
  a.stride = plan.stride;
  a.OH = y->h;
  a.OW = y->w;
  a.blk_w = plan.blk_w;
  a.n_blk = plan.n_blk;
  a.Wp = plan.wp;
  a.Cout = Co;
  a.kc = plan.kc;
  const int chan = plan.kc * 4 / plan.eb;  // channels per chunk
  a.num_kc = Ci / chan;
  a.bf16 = plan.eb == 2 ? 1 : 0;
  a.px_tiles_per_blk = (a.OH * a.Wp + plan.px - 1) / plan.px;
  a.sub = plan.sub;
  a.tiles_per_blk = (a.px_tiles_per_blk + plan.sub - 1) / plan.sub;
  a.tiles_per_img = a.n_blk * a.tiles_per_blk;
  a.m_tiles = x->n * a.tiles_per_img;
  a.n_tiles = (Co + plan.co - 1) / plan.co;
  a.rows = halo_rows(a.Wp, plan.px * plan.sub, plan.stride);
  a.halo_bytes = halo_buffer_bytes(a.Wp, plan.px * plan.sub, plan.kc, plan.stride);
  a.phase_bytes = plan.stride == 2 ? a.halo_bytes / 4 : 0;
  a.nb_stages = plan.nb;
  a.taps_per_stage = plan.tps;
  a.w_resident = plan.resident ? 1 : 0;
  a.split_k = plan.split;
  a.out = make_out(y);
  a.ep = ep;
  a.err = dev->err;
  a.timeout_ns = timeout_ns();
  a.vec_store = (aligned16(a.out.y) && strides_mult4(y) && aligned16(ep.scale) && aligned16(ep.bias) &&
                 (ep.res_mode == 0 || (aligned16(ep.r) && ep.rs_n % 4 == 0 && ep.rs_h % 4 == 0 && ep.rs_w % 4 == 0)))
                    ? 1
                    : 0;
  const Tuning tu = tuning();
  if (tu.trace_cta >= 0) {  // profiling aid: timeline of one CTA
    a.trace = tu.span_slot;
    a.trace_cta = tu.trace_cta;
  }
  if (tu.debug_plan)
    std::fprintf(stderr,
                 "[cb] halo plan: N=%d H=%d W=%d Ci=%d Co=%d s=%d -> %s px=%dx%d co=%d kc=%d nb=%d tps=%d "
                 "split=%d%s blocks=%dx%d rows=%d halo=%d tiles=%d grid=%d smem=%zu\n",
                 x->n, a.H, a.W, Ci, Co, plan.stride, plan.cm ? "channel-major" : "pixel-major", plan.sub, plan.px,
                 plan.co, plan.kc, plan.nb, plan.tps, plan.split, plan.resident ? " resident" : "", plan.n_blk, plan.blk_w,
                 a.rows, a.halo_bytes,
                 a.m_tiles * a.n_tiles, plan.grid, plan.smem);
  CUtensorMap xmap, wmap;
  const cuuint64_t eb = static_cast<cuuint64_t>(plan.eb);
  const CUtensorMapDataType dt = plan.eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const CUtensorMapSwizzle swz = plan.kc == 32   ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : plan.kc == 16 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                 : CU_TENSOR_MAP_SWIZZLE_32B;
  {
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(Ci), static_cast<cuuint64_t>(x->w), static_cast<cuuint64_t>(x->h),
                          static_cast<cuuint64_t>(x->n)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(x->stride_w) * eb, static_cast<cuuint64_t>(x->stride_h) * eb,
                             static_cast<cuuint64_t>(x->stride_n) * eb};
    // stride 2: each phase tile traverses 2 Wp columns and 2 rows rows of the
    // input with element strides 2
    const cuuint32_t st = static_cast<cuuint32_t>(plan.stride);
    cuuint32_t box[4] = {static_cast<cuuint32_t>(chan), st * static_cast<cuuint32_t>(a.Wp),
                         st * static_cast<cuuint32_t>(a.rows), 1};
    cuuint32_t estr[4] = {1, st, st, 1};
    CUresult r = tiled_map(&xmap, 4, x->data, dims, strides, box, estr, swz, dt);
    if (r != CUDA_SUCCESS) return CB_ERR_UNSUPPORTED;
  }
  {
    // OHWI weights viewed as (Ci, Co, tap): a box of plan.tps taps lands as
    // plan.tps consecutive [co x chunk] slices
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(Ci), static_cast<cuuint64_t>(Co), 9};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(9) * Ci * eb, static_cast<cuuint64_t>(Ci) * eb};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(chan), static_cast<cuuint32_t>(plan.co),
                         static_cast<cuuint32_t>(plan.tps)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = tiled_map(&wmap, 3, w, dims, strides, box, estr, swz, dt);
    if (r != CUDA_SUCCESS) return CB_ERR_UNSUPPORTED;
  }
  cudaError_t e = launch_igemm_halo(xmap, wmap, a, plan.px, plan.co, plan.cm, plan.grid, plan.smem, s);
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

cb_status run_direct(const cb_tensor* x, const float* w, const Epilogue& ep, int k, int stride, int pad,
                     const cb_tensor* y, cudaStream_t s);

bool pixel_flat(const cb_tensor* t) {
  return t->stride_h == static_cast<long long>(t->w) * t->stride_w &&
         t->stride_n == static_cast<long long>(t->h) * t->stride_h;
}

cb_status run_pointwise(const cb_tensor* x, const float* w, const Epilogue& ep, const cb_tensor* residual,
                        const cb_tensor* y, cudaStream_t s) {
  DeviceInfo* dev = nullptr;
  cb_status st = current_device(&dev);
  if (st != CB_OK) return st;
  DirectArgs a{};
  a.x = static_cast<const float*>(x->data);
  a.xs_n = x->stride_n;
  a.xs_h = x->stride_h;
  a.xs_w = x->stride_w;
  a.xs_c = 1;
  a.w = w;
  a.N = x->n;
  a.H = x->h;
  a.W = x->w;
  a.Ci = x->c;
  a.Co = y->c;
  a.OH = y->h;
  a.OW = y->w;
  a.kh = a.kw = 1;
  a.stride = 1;
  a.pad = 0;
  a.out = make_out(y);
  a.ep = ep;
  a.bf16 = x->dtype == CB_DTYPE_BF16 ? 1 : 0;
  const bool flat = pixel_flat(x) && pixel_flat(y) && (ep.res_mode == 0 || pixel_flat(residual));
  cudaError_t e = launch_pointwise_small(a, flat, dev->sms, s);
  // a shape the kernel does not take: the direct kernel (fp32 views only)
  if (e == cudaErrorInvalidValue) return a.bf16 ? CB_ERR_UNSUPPORTED : run_direct(x, w, ep, 1, 1, 0, y, s);
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

cb_status run_stem(const cb_tensor* x, const float* w, const Epilogue& ep, const cb_tensor* y, cudaStream_t s) {
  DeviceInfo* dev = nullptr;
  cb_status st = current_device(&dev);
  if (st != CB_OK) return st;
  StemArgs a{};
  a.src = x->data;
  a.xs_n = x->stride_n;
  a.xs_h = x->stride_h;
  a.xs_c = x->stride_c;
  a.N = x->n;
  a.H = x->h;
  a.W = x->w;
  a.OH = y->h;
  a.OW = y->w;
  a.w = w;
  a.ep = ep;
  a.out = make_out(y);
  stem_tile_grid(a.OH, a.OW, &a.tiles_y, &a.tiles_x);
  a.err = dev->err;
  a.timeout_ns = timeout_ns();
  const int kind = !is_f32(x) ? 3 : x->layout == CB_LAYOUT_NCHW ? 0 : 1;
  // packed NHWC input: the tensor-core kernel (fp32 accuracy from split TF32
  // operands), unless CB_STEM_KERNEL = "cuda"; planar input: the CUDA-core kernel
  const bool tc = (kind == 1 || kind == 3) && tuning().stem_kernel != 1 && stem_tc_ok(a);
  const cudaError_t e =
      tc ? launch_stem_tc(a, kind == 3, dev->sms, s) : launch_stem(a, kind, stem_smem_bytes(kind, 0, 0), dev->sms, s);
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

cb_status run_direct(const cb_tensor* x, const float* w, const Epilogue& ep, int k, int stride, int pad,
                     const cb_tensor* y, cudaStream_t s) {
  DirectArgs a{};
  a.x = static_cast<const float*>(x->data);
  a.xs_n = x->stride_n;
  a.xs_h = x->stride_h;
  a.xs_w = x->stride_w;
  a.xs_c = x->stride_c;
  a.w = w;
  a.N = x->n;
  a.H = x->h;
  a.W = x->w;
  a.Ci = x->c;
  a.Co = y->c;
  a.OH = y->h;
  a.OW = y->w;
  a.kh = k;
  a.kw = k;
  a.stride = stride;
  a.pad = pad;
  a.out = make_out(y);
  a.ep = ep;
  a.bf16 = x->dtype == CB_DTYPE_BF16 ? 1 : 0;  // the 8-channel kernel only
  DeviceInfo* dev = nullptr;
  cb_status st = current_device(&dev);
  if (st != CB_OK) return st;
  cudaError_t e = launch_direct(a, dev->sms, s);
  if (e == cudaErrorInvalidValue) return CB_ERR_UNSUPPORTED;
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

}  // namespace

// =============================================================================
extern "C" {

cb_status cb_fold_bn(const float* gamma, const float* beta, const float* mean, const float* var, float eps, int C,
                     float* scale, float* bias) {
  if (!gamma || !beta || !mean || !var || !scale || !bias || C <= 0 || !(eps >= 0.0f)) return CB_ERR_INVALID_ARG;
  for (int c = 0; c < C; ++c)
    if (!(static_cast<double>(var[c]) + eps > 0.0)) return CB_ERR_INVALID_ARG;
  for (int c = 0; c < C; ++c) {
    const double sc = static_cast<double>(gamma[c]) / std::sqrt(static_cast<double>(var[c]) + static_cast<double>(eps));
    scale[c] = static_cast<float>(sc);
    bias[c] = static_cast<float>(static_cast<double>(beta[c]) - static_cast<double>(mean[c]) * sc);
  }
  return CB_OK;
}

cb_status cb_repack_weights(const float* w_oihw, int Co, int Ci_per_group, int kh, int kw, int groups,
                            float* w_out) {
  if (!w_oihw || !w_out || Co <= 0 || Ci_per_group <= 0 || kh <= 0 || kw <= 0 || groups <= 0)
    return CB_ERR_INVALID_ARG;
  if (groups == 1) {
    for (int o = 0; o < Co; ++o)
      for (int i = 0; i < kh; ++i)
        for (int j = 0; j < kw; ++j)
          for (int c = 0; c < Ci_per_group; ++c)
            w_out[((static_cast<long long>(o) * kh + i) * kw + j) * Ci_per_group + c] =
                w_oihw[((static_cast<long long>(o) * Ci_per_group + c) * kh + i) * kw + j];
    return CB_OK;
  }
  if (groups == Co && Ci_per_group == 1) {
    for (int o = 0; o < Co; ++o)
      for (int i = 0; i < kh; ++i)
        for (int j = 0; j < kw; ++j)
          w_out[(static_cast<long long>(i) * kw + j) * Co + o] = w_oihw[(static_cast<long long>(o) * kh + i) * kw + j];
    return CB_OK;
  }
  return CB_ERR_UNSUPPORTED;
}

cb_status cb_round_weights_tf32(const float* w, long long n, float* out) {
  if (!w || !out || n < 0) return CB_ERR_INVALID_ARG;
  for (long long i = 0; i < n; ++i) {
    uint32_t b;
    std::memcpy(&b, &w[i], sizeof(b));
    if ((b & 0x7F800000u) != 0x7F800000u) {  // finite: round the low 13 bits to nearest, ties to even
      const uint32_t lsb = (b >> 13) & 1u;
      b = (b + 0x0FFFu + lsb) & ~0x1FFFu;
    }
    std::memcpy(&out[i], &b, sizeof(b));
  }
  return CB_OK;
}

cb_status cb_convert_weights_bf16(const float* w, long long n, void* out) {
  if (!w || !out || n < 0) return CB_ERR_INVALID_ARG;
  uint16_t* o = static_cast<uint16_t*>(out);
  for (long long i = 0; i < n; ++i) {
    uint32_t b;
    std::memcpy(&b, &w[i], 4);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu) != 0) {
      o[i] = static_cast<uint16_t>((b >> 16) | 0x0040u);  // NaN stays a (quiet) NaN
      continue;
    }
    // round to nearest, ties to even, on the upper 16 bits (an overflow carries into inf)
    b += 0x7FFFu + ((b >> 16) & 1u);
    o[i] = static_cast<uint16_t>(b >> 16);
  }
  return CB_OK;
}

namespace {
// Argument checks of cb_conv_bn_act (no launch).  *empty: nothing to compute.
cb_status validate_conv(const cb_tensor* x, const float* w, const float* scale, const float* bias, int kh, int kw,
                        int stride, int pad, int groups, cb_act act, const cb_tensor* residual, cb_res_mode res_mode,
                        const cb_tensor* y, bool* depthwise_out, bool* empty) {
  if (!view_ok(x) || !view_ok(y) || !w || !scale || !bias) return CB_ERR_INVALID_ARG;
  if (act < CB_ACT_NONE || act > CB_ACT_SILU || res_mode < CB_RES_NONE || res_mode > CB_RES_POST_ACT)
    return CB_ERR_INVALID_ARG;
  if (kh != kw || (kh != 1 && kh != 3)) return CB_ERR_UNSUPPORTED;
  if (stride != 1 && stride != 2) return CB_ERR_UNSUPPORTED;
  if (pad < 0 || pad > kh / 2) return CB_ERR_UNSUPPORTED;
  if (y->layout != CB_LAYOUT_NHWC) return CB_ERR_UNSUPPORTED;
  if (x->h + 2 * pad < kh || x->w + 2 * pad < kw) return CB_ERR_INVALID_ARG;
  const int OH = (x->h + 2 * pad - kh) / stride + 1, OW = (x->w + 2 * pad - kw) / stride + 1;
  if (y->n != x->n || y->h != OH || y->w != OW) return CB_ERR_INVALID_ARG;
  const bool depthwise = groups == x->c && groups == y->c && groups > 1;
  if (!depthwise && groups != 1) return CB_ERR_UNSUPPORTED;
  if (x->dtype != y->dtype) return CB_ERR_INVALID_ARG;
  // bf16 storage: the depthwise kernel, the pointwise kernel's 1x1 shapes and
  // the tensor-core shapes
  if (!is_f32(x) && !depthwise &&
      (g_policy.load() == 1 ||
       !((kh == 1 && stride == 1 && pad == 0 && pointwise_small_ok(x->c, y->c, true)) ||
         (tc_shape(x->c, y->c, kh, stride, pad) && x->c % 8 == 0) ||
         (x->c == 3 && y->c == 16 && kh == 3 && stride == 2 && pad == 1 && x->layout == CB_LAYOUT_NHWC) ||
         (x->c == 8 && y->c == 8 && kh == 3 && stride == 1 && pad == 1 && x->layout == CB_LAYOUT_NHWC))))
    return CB_ERR_UNSUPPORTED;
  if (res_mode != CB_RES_NONE) {
    if (!view_ok(residual) || residual->layout != CB_LAYOUT_NHWC || residual->dtype != y->dtype)
      return CB_ERR_INVALID_ARG;
    if (residual->n != y->n || residual->h != y->h || residual->w != y->w || residual->c != y->c)
      return CB_ERR_INVALID_ARG;
    if (!same_view(residual, y) && overlap(residual, y)) return CB_ERR_INVALID_ARG;
  }
  if (overlap(x, y)) return CB_ERR_INVALID_ARG;
  const long long M = static_cast<long long>(x->n) * OH * OW;
  if (M > (1LL << 31) - 129) return CB_ERR_UNSUPPORTED;
  if (depthwise && (kh != 3 || x->layout != CB_LAYOUT_NHWC)) return CB_ERR_UNSUPPORTED;
  *depthwise_out = depthwise;
  *empty = x->n == 0;
  return CB_OK;
}

// One launch of a validated layer: the depthwise kernel, or the dense path
// (a forced plan when `force` is given, else the tuned or modelled one).
cb_status launch_conv(const cb_tensor* x, const float* w, const float* scale, const float* bias, int kh, int stride,
                      int pad, bool depthwise, cb_act act, const cb_tensor* residual, cb_res_mode res_mode,
                      const cb_tensor* y, cudaStream_t s, const ConvPlan* force) {
  const Epilogue ep = make_epilogue(scale, bias, act, residual, res_mode);
  if (depthwise) return run_depthwise(x, w, ep, stride, pad, y, s);
  if (!is_f32(x)) {
    // bf16 storage (a pointwise or tensor-core shape, checked in
    // validation): aligned views and operands, else no kernel takes it
    if (!aligned16(w) || !aligned16(scale) || !aligned16(bias) ||
        (res_mode != CB_RES_NONE && (!aligned16(residual->data) || !strides_mult4(residual))))
      return CB_ERR_ALIGNMENT;
    if (pointwise_bf16_views(x, y, kh, stride, pad)) return run_pointwise(x, w, ep, residual, y, s);
    if (x->c == 3 && y->c == 16 && kh == 3)  // the stem shape (validated): its bf16 kernel, else no kernel
      return stem_path(x, y, kh, stride, pad) ? run_stem(x, w, ep, y, s) : CB_ERR_ALIGNMENT;
    if (x->c == 8 && y->c == 8 && kh == 3)  // the 8-channel kernel
      return c8_bf16_views(x, y, kh, stride, pad) ? run_direct(x, w, ep, kh, stride, pad, y, s) : CB_ERR_ALIGNMENT;
    if (!tc_bf16_views(x, y, kh, stride, pad)) return CB_ERR_ALIGNMENT;
  }
  HaloPlan plan;
  ImPlan im;
  const cb_path path = force ? force->path : dense_path(x, y, kh, stride, pad, &plan, &im);
  if (force) plan = force->halo, im = force->im;
  if (path == CB_PATH_STEM) {
    // 16-byte residual accesses, else the direct kernel
    const bool vec = res_mode == CB_RES_NONE || (aligned16(residual->data) && strides_mult4(residual));
    return vec ? run_stem(x, w, ep, y, s) : run_direct(x, w, ep, kh, stride, pad, y, s);
  }
  if (path == CB_PATH_POINTWISE) {
    // 16-byte weight, scale / bias and residual accesses, else the direct kernel
    const bool vec = aligned16(w) && aligned16(scale) && aligned16(bias) &&
                     (res_mode == CB_RES_NONE || (aligned16(residual->data) && strides_mult4(residual)));
    return vec ? run_pointwise(x, w, ep, residual, y, s) : run_direct(x, w, ep, kh, stride, pad, y, s);
  }
  if (!aligned16(w) && path != CB_PATH_DIRECT) {
    // the tensor-core paths read w through TMA: an unaligned copy goes to the direct kernel
    return run_direct(x, w, ep, kh, stride, pad, y, s);
  }
  switch (path) {
    case CB_PATH_TC_HALO:
    case CB_PATH_TC_HALO_CM: return run_igemm_halo(x, w, ep, plan, y, s);
    case CB_PATH_TC_IM2COL: return run_igemm(x, w, ep, kh, stride, pad, y, s, im);
    default: return run_direct(x, w, ep, kh, stride, pad, y, s);
  }
}

// Every plan of the dense tensor-core paths that fits this layer.
std::vector<ConvPlan> tc_candidates(const cb_tensor* x, const cb_tensor* y, int kh, int stride, int pad, int sms) {
  std::vector<ConvPlan> out;
  const int Ci = x->c, Co = y->c;
  if (kh == 3 && pad == 1 && Ci % 8 == 0 && g_policy.load() == 0) {
    // every halo tile shape x taps per weight stage x split, each planned
    // under those constraints (ring depth, column blocks and grid follow)
    struct Shape {
      int co;
      bool cm;
      int px;
    };
    static const Shape kShapes[] = {{128, true, 256}, {128, true, 192}, {256, false, 128}, {128, false, 128},
                                    {64, false, 128},  {32, false, 128}};
    for (const Shape& sh : kShapes) {
      if (!sh.cm && sh.co > 2 * ((Co + 15) / 16 * 16)) continue;  // a tile mostly beyond Co
      for (int tps : {9, 3, 1})
        for (int split : {1, 2})
          for (int sb : {1, 2, 4}) {
          if (sb > 1 && (sh.cm || sh.co > 64 || split == 2)) continue;
          HaloForce f;
          f.co = sh.cm ? 0 : sh.co;
          f.cm = sh.cm;
          f.px = sh.cm ? sh.px : 0;
          f.tps = tps;
          f.split = split;
          f.sub = sb;
          f.res = 0;
          ConvPlan p;
          if (!plan_halo(x, y, stride, sms, f, &p.halo)) continue;
          p.path = p.halo.cm ? CB_PATH_TC_HALO_CM : CB_PATH_TC_HALO;
          out.push_back(p);
        }
      // resident weights (one chunk, one channel tile)
      for (int sb : {1, 2, 4}) {
        if (sb > 1 && (sh.cm || sh.co > 64)) continue;
        HaloForce f;
        f.co = sh.cm ? 0 : sh.co;
        f.cm = sh.cm;
        f.px = sh.cm ? sh.px : 0;
        f.sub = sb;
        f.res = 1;
        ConvPlan p;
        if (!plan_halo(x, y, stride, sms, f, &p.halo)) continue;
        p.path = p.halo.cm ? CB_PATH_TC_HALO_CM : CB_PATH_TC_HALO;
        out.push_back(p);
      }
    }
  }
  for (int bn : {16, 32, 48, 64, 96, 128, 192, 256}) {
    if (bn > 2 * ((Co + 15) / 16 * 16) && bn > 16) continue;
    ConvPlan p;
    p.path = CB_PATH_TC_IM2COL;
    p.im.bn = bn;
    out.push_back(p);
  }
  return out;
}
}  // namespace

cb_status cb_conv_bn_act(const cb_tensor* x, const float* w, const float* scale, const float* bias, int kh, int kw,
                         int stride, int pad, int groups, cb_act act, const cb_tensor* residual,
                         cb_res_mode res_mode, cb_tensor* y, void* stream) {
  bool depthwise = false, empty = false;
  cb_status st = validate_conv(x, w, scale, bias, kh, kw, stride, pad, groups, act, residual, res_mode, y,
                               &depthwise, &empty);
  if (st != CB_OK || empty) return st;
  return launch_conv(x, w, scale, bias, kh, stride, pad, depthwise, act, residual, res_mode, y,
                     static_cast<cudaStream_t>(stream), nullptr);
}

cb_status cb_autotune_conv(const cb_tensor* x, const float* w, const float* scale, const float* bias, int kh, int kw,
                           int stride, int pad, int groups, cb_act act, const cb_tensor* residual,
                           cb_res_mode res_mode, cb_tensor* y, void* stream) {
  bool depthwise = false, empty = false;
  cb_status st = validate_conv(x, w, scale, bias, kh, kw, stride, pad, groups, act, residual, res_mode, y,
                               &depthwise, &empty);
  if (st != CB_OK) return st;
  // Every candidate launch writes y: an in-place residual (residual == y)
  // would be added again on each launch and be lost after the first.
  if (res_mode != CB_RES_NONE && overlap(residual, y)) return CB_ERR_INVALID_ARG;
  if (empty) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const ConvKey key = conv_key(x, y, kh, stride, pad);
  {
    std::lock_guard<std::mutex> lock(g_tune_mu);
    g_tuned.erase(key);  // decide afresh
  }
  HaloPlan hp;
  const cb_path path = depthwise ? CB_PATH_DEPTHWISE : dense_path(x, y, kh, stride, pad, &hp);
  const bool tc = path == CB_PATH_TC_HALO || path == CB_PATH_TC_HALO_CM || path == CB_PATH_TC_IM2COL;
  if (!tc || !aligned16(w)) {  // one kernel only: nothing to choose
    return launch_conv(x, w, scale, bias, kh, stride, pad, depthwise, act, residual, res_mode, y, s, nullptr);
  }
  DeviceInfo* dev = nullptr;
  st = current_device(&dev);
  if (st != CB_OK) return st;
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return cuda_fail(cudaGetLastError());
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return cuda_fail(cudaGetLastError());
  }
  // Every candidate is timed in each of kRounds passes over the list and
  // keeps its best pass, so that one disturbed sample (a clock step, another
  // stream's work) does not decide between plans a few per cent apart.
  constexpr int kReps = 5, kRounds = 2;
  constexpr float kUntimed = 1e30f;
  const std::vector<ConvPlan> cands = tc_candidates(x, y, kh, stride, pad, dev->sms);
  std::vector<float> cand_ms(cands.size(), kUntimed);
  for (int round = 0; round < kRounds; ++round) {
    for (size_t i = 0; i < cands.size(); ++i) {
      if (round > 0 && cand_ms[i] == kUntimed) continue;  // this layer cannot take it
      const ConvPlan& cand = cands[i];
      // warm-up launch (also rejects plans this layer cannot take), then kReps timed ones
      if (launch_conv(x, w, scale, bias, kh, stride, pad, false, act, residual, res_mode, y, s, &cand) != CB_OK)
        continue;
      cudaEventRecord(e0, s);
      bool ok = true;
      for (int r = 0; r < kReps && ok; ++r)
        ok = launch_conv(x, w, scale, bias, kh, stride, pad, false, act, residual, res_mode, y, s, &cand) == CB_OK;
      cudaEventRecord(e1, s);
      if (cudaEventSynchronize(e1) != cudaSuccess || !ok) continue;
      float ms = 0.0f;
      cudaEventElapsedTime(&ms, e0, e1);
      cand_ms[i] = std::min(cand_ms[i], ms);
    }
  }
  float best_ms = kUntimed;
  ConvPlan best;
  bool found = false;
  for (size_t i = 0; i < cands.size(); ++i) {
    if (cand_ms[i] < best_ms) {
      best_ms = cand_ms[i];
      best = cands[i];
      found = true;
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (found) {
    std::lock_guard<std::mutex> lock(g_tune_mu);
    g_tuned[key] = best;
  }
  if (tuning().debug_plan && found)
    std::fprintf(stderr,
                 "[cb] autotune: Ci=%d Co=%d %dx%d k=%d s=%d -> path %d (px=%d co=%d nb=%d split=%d bn=%d) %.1f us\n",
                 x->c, y->c, x->h, x->w, kh, stride, static_cast<int>(best.path), best.halo.px, best.halo.co,
                 best.halo.nb, best.halo.split, best.im.bn, 1000.0f * best_ms / kReps);
  // leave y holding the chosen plan's result
  st = launch_conv(x, w, scale, bias, kh, stride, pad, false, act, residual, res_mode, y, s, found ? &best : nullptr);
  if (st != CB_OK) return st;
  const cudaError_t e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

void cb_autotune_clear(void) {
  std::lock_guard<std::mutex> lock(g_tune_mu);
  g_tuned.clear();
}

int cb_autotune_entries(void) {
  std::lock_guard<std::mutex> lock(g_tune_mu);
  return static_cast<int>(g_tuned.size());
}

namespace {
// The one-kernel block (dw_block.cu) takes these shapes and views.  It is
// chosen where it measured faster than the three layer kernels: blocks with
// a conv skip (three launches become one) and at least 64 tiles of 128
// pixels.  Its CTAs gather the depthwise taps from L2 with plain loads, one
// round trip per pixel and chunk, so with fewer tiles (or only two layer
// kernels to replace) the TMA-fed layer kernels win.
// Tuning override: CB_DW_BLOCK_FORCE=1 takes the one kernel wherever its
// shape rule allows, =0 never.
bool dw_block_fusable(const cb_tensor* x, const cb_tensor* y, const float* pw_w, const float* skip_w) {
  const long long pix = static_cast<long long>(y->n) * y->h * y->w;
  bool pick = skip_w && (pix + 127) / 128 >= 64;
  const int force = tuning().dw_block;
  if (force >= 0) pick = force == 1;
  return g_policy.load() == 0 && pick && x->layout == CB_LAYOUT_NHWC && y->layout == CB_LAYOUT_NHWC && x->c % 4 == 0 &&
         x->c <= 1024 && y->c % 32 == 0 && y->c <= 256 && pix < (1LL << 31) && aligned16(x->data) &&
         strides_mult4(x) && aligned16(y->data) && strides_mult4(y) && aligned16(pw_w) &&
         (!skip_w || aligned16(skip_w)) && x->n <= 65535 && encode_tiled();
}
}  // namespace

int cb_dw_separable_block_fused(const cb_tensor* x, const cb_tensor* y, const float* pw_w, const float* skip_w) {
  if (!view_ok(x) || !view_ok(y) || !pw_w || !is_f32(x) || !is_f32(y)) return 0;
  return dw_block_fusable(x, y, pw_w, skip_w) ? 1 : 0;
}

cb_status cb_dw_separable_block_workspace(const cb_tensor* x, int c_out, int stride, size_t* bytes) {
  if (!view_ok(x) || !bytes || c_out < 1 || (stride != 1 && stride != 2)) return CB_ERR_INVALID_ARG;
  if (!is_f32(x)) return CB_ERR_UNSUPPORTED;
  const long long OH = (x->h + 2 - 3) / stride + 1, OW = (x->w + 2 - 3) / stride + 1;
  if (x->h < 1 || x->w < 1 || OH < 1 || OW < 1) return CB_ERR_INVALID_ARG;
  const long long pix = static_cast<long long>(x->n) * OH * OW;
  const size_t t_bytes = (static_cast<size_t>(pix) * x->c * sizeof(float) + 255) & ~size_t(255);
  const size_t s_bytes = (static_cast<size_t>(pix) * c_out * sizeof(float) + 255) & ~size_t(255);
  *bytes = t_bytes + s_bytes;
  return CB_OK;
}

cb_status cb_dw_separable_block(const cb_tensor* x, const float* dw_w, const float* dw_scale, const float* dw_bias,
                                const float* pw_w, const float* pw_scale, const float* pw_bias, const float* skip_w,
                                const float* skip_scale, const float* skip_bias, int stride, cb_tensor* y,
                                void* workspace, size_t workspace_bytes, void* stream) {
  if (!view_ok(x) || !view_ok(y) || !dw_w || !dw_scale || !dw_bias || !pw_w || !pw_scale || !pw_bias)
    return CB_ERR_INVALID_ARG;
  if (!is_f32(x) || !is_f32(y)) return CB_ERR_UNSUPPORTED;
  if (x->layout != CB_LAYOUT_NHWC || y->layout != CB_LAYOUT_NHWC) return CB_ERR_UNSUPPORTED;
  if (stride != 1 && stride != 2) return CB_ERR_UNSUPPORTED;
  const int Ci = x->c, Co = y->c;
  const int OH = (x->h - 1) / stride + 1, OW = (x->w - 1) / stride + 1;
  if (y->n != x->n || y->h != OH || y->w != OW) return CB_ERR_INVALID_ARG;
  if (skip_w && (!skip_scale || !skip_bias)) return CB_ERR_INVALID_ARG;
  if (!skip_w && (stride != 1 || Ci != Co)) return CB_ERR_INVALID_ARG;
  if (overlap(x, y)) return CB_ERR_INVALID_ARG;
  size_t need = 0;
  cb_status st = cb_dw_separable_block_workspace(x, Co, stride, &need);
  if (st != CB_OK) return st;
  if (x->n == 0) return CB_OK;
  if (!workspace || workspace_bytes < need) return CB_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return CB_ERR_ALIGNMENT;

  const long long pix = static_cast<long long>(x->n) * OH * OW;
  // The whole block in one kernel when the views, weights and channel counts
  // allow it (policy 0); else three layer calls through the workspace.
  if (dw_block_fusable(x, y, pw_w, skip_w)) {
    DeviceInfo* dev = nullptr;
    st = current_device(&dev);
    if (st != CB_OK) return st;
    DwBlockArgs a{};
    a.x = static_cast<const float*>(x->data);
    a.xs_n = x->stride_n;
    a.xs_h = x->stride_h;
    a.xs_w = x->stride_w;
    a.N = x->n;
    a.H = x->h;
    a.W = x->w;
    a.Ci = Ci;
    a.Co = Co;
    a.OH = OH;
    a.OW = OW;
    a.stride = stride;
    a.M = static_cast<int>(pix);
    a.dw_w = dw_w;
    a.dw_scale = dw_scale;
    a.dw_bias = dw_bias;
    a.pw_scale = pw_scale;
    a.pw_bias = pw_bias;
    a.skip_conv = skip_w ? 1 : 0;
    a.sk_scale = skip_scale;
    a.sk_bias = skip_bias;
    a.num_kc = (Ci + 31) / 32;
    const int cols = skip_w ? 2 * Co : Co;
    a.tmem_cols = cols <= 32 ? 32 : cols <= 64 ? 64 : cols <= 128 ? 128 : cols <= 256 ? 256 : 512;
    a.out = make_out(y);
    a.err = dev->err;
    a.timeout_ns = timeout_ns();
    const int trace_cta = tuning().trace_cta;
    if (trace_cta >= 0) {  // profiling aid: timeline of one CTA
      a.trace = 1;
      a.trace_cta = trace_cta;
    }
    CUtensorMap pw_map, sk_map;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(Ci), 1, static_cast<cuuint64_t>(Co)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(Ci) * 4, static_cast<cuuint64_t>(Ci) * 4};
    cuuint32_t box[3] = {32, 1, static_cast<cuuint32_t>(Co)};
    cuuint32_t estr[3] = {1, 1, 1};
    if (tiled_map(&pw_map, 3, pw_w, dims, strides, box, estr, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return CB_ERR_UNSUPPORTED;
    sk_map = pw_map;
    if (skip_w && tiled_map(&sk_map, 3, skip_w, dims, strides, box, estr, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return CB_ERR_UNSUPPORTED;
    const cudaError_t e = launch_dw_block(pw_map, sk_map, a, static_cast<cudaStream_t>(stream));
    if (e != cudaErrorInvalidValue) return e == cudaSuccess ? CB_OK : cuda_fail(e);
  }
  const size_t t_bytes = (static_cast<size_t>(pix) * Ci * sizeof(float) + 255) & ~size_t(255);
  cb_tensor t{workspace, x->n, OH, OW, Ci, static_cast<long long>(OH) * OW * Ci, static_cast<long long>(OW) * Ci,
              Ci, 1, CB_LAYOUT_NHWC};
  cb_tensor sk{static_cast<char*>(workspace) + t_bytes, x->n, OH, OW, Co, static_cast<long long>(OH) * OW * Co,
               static_cast<long long>(OW) * Co, Co, 1, CB_LAYOUT_NHWC};
  st = cb_conv_bn_act(x, dw_w, dw_scale, dw_bias, 3, 3, stride, 1, Ci, CB_ACT_RELU, nullptr, CB_RES_NONE, &t,
                      stream);
  if (st != CB_OK) return st;
  const cb_tensor* r = x;
  if (skip_w) {
    st = cb_conv_bn_act(x, skip_w, skip_scale, skip_bias, 1, 1, stride, 0, 1, CB_ACT_NONE, nullptr, CB_RES_NONE, &sk,
                        stream);
    if (st != CB_OK) return st;
    r = &sk;
  }
  return cb_conv_bn_act(&t, pw_w, pw_scale, pw_bias, 1, 1, 1, 0, 1, CB_ACT_RELU, r, CB_RES_PRE_ACT, y, stream);
}

// ------------------------------------------------ YOLO-style stage body
// Nearest TF32 value of a finite fp32 value (ties to even), as fp32 bits.
static uint32_t tf32_nearest_bits(float w) {
  float r = 0.0f;
  cb_round_weights_tf32(&w, 1, &r);
  uint32_t b;
  std::memcpy(&b, &r, sizeof(b));
  return b;
}

// C = 32 (validated by cb_stage_body): the weights' shared-memory image, the
// folded BN and the two tensor maps into the launch.
static cb_status stage_body_tc(const cb_tensor* x1, const float* w1, const float* s1, const float* b1,
                               const float* w2, const float* s2, const float* b2, const float* w3, const float* s3,
                               const float* b3, cb_act act, cb_tensor* y, DeviceInfo* dev, void* stream) {
  StageBodyTcArgs a{};
  const bool bf = !is_f32(x1);
  a.x = x1->data;
  a.xs_n = x1->stride_n;
  a.xs_h = x1->stride_h;
  a.xs_w = x1->stride_w;
  a.N = x1->n;
  a.H = x1->h;
  a.W = x1->w;
  a.act = static_cast<int>(act);
  a.err = dev->err;
  a.timeout_ns = timeout_ns();
  a.bf16 = bf ? 1 : 0;
  a.debug_skip_x = tuning().stage_skip_x;
  // element k of row r of a K-major operand of rb-byte rows at byte r * rb +
  // ((k * eb / 16) ^ sw(r)) * 16 + k * eb % 16, sw the swizzle of rb-byte rows
  const int eb = bf ? 2 : 4;
  uint8_t* const img = reinterpret_cast<uint8_t*>(a.wimg);
  // lo: the bf16 tail w - bf16(w) of a split weight (the 1x1 layers with bf16 storage)
  auto put = [img, eb](int base, int rb, int r, int k, float w, bool lo) {
    const int sw = rb == 128 ? (r & 7) : rb == 64 ? ((r >> 1) & 3) : ((r >> 2) & 1);
    const int at = base + r * rb + ((((k * eb) >> 4) ^ sw) << 4) + ((k * eb) & 15);
    if (eb == 4) {
      const uint32_t b = tf32_nearest_bits(w);
      std::memcpy(img + at, &b, 4);
    } else {
      uint16_t h = 0;
      cb_convert_weights_bf16(&w, 1, &h);  // nearest even
      if (lo) {
        const uint32_t hb = static_cast<uint32_t>(h) << 16;
        float hf;
        std::memcpy(&hf, &hb, 4);
        const float l = w - hf;  // exact
        cb_convert_weights_bf16(&l, 1, &h);
      }
      std::memcpy(img + at, &h, 2);
    }
  };
  const int xrow = 32 * eb, arow = 16 * eb;  // bytes of a 32- and a 16-channel row
  const int w1_at = 0, w2_at = 2048, tap_bytes = bf ? 512 : 1024, w3_at = bf ? 7168 : 11264;
  for (int co = 0; co < 16; ++co)
    for (int ci = 0; ci < 32; ++ci) {
      put(w1_at, xrow, co, ci, w1[co * 32 + ci], false);
      if (bf) put(1024, xrow, co, ci, w1[co * 32 + ci], true);
    }
  for (int tap = 0; tap < 9; ++tap)
    for (int co = 0; co < 16; ++co)
      for (int ci = 0; ci < 16; ++ci) put(w2_at + tap_bytes * tap, arow, co, ci, w2[(co * 9 + tap) * 16 + ci], false);
  for (int co = 0; co < 32; ++co)
    for (int ci = 0; ci < 32; ++ci) {
      put(w3_at, xrow, co, ci, w3[co * 32 + ci], false);
      if (bf) put(9216, xrow, co, ci, w3[co * 32 + ci], true);
    }
  for (int c = 0; c < 16; ++c) {
    a.sb[c] = s1[c], a.sb[16 + c] = b1[c];
    a.sb[32 + c] = s2[c], a.sb[48 + c] = b2[c];
  }
  for (int c = 0; c < 32; ++c) a.sb[64 + c] = s3[c], a.sb[96 + c] = b3[c];
  int xw = 0, xh = 0, yw = 0, yh = 0;
  stage_body_tc_boxes(&xw, &xh, &yw, &yh);
  cuuint64_t xdims[4] = {32, static_cast<cuuint64_t>(x1->w), static_cast<cuuint64_t>(x1->h),
                         static_cast<cuuint64_t>(x1->n)};
  cuuint64_t xstr[3] = {static_cast<cuuint64_t>(x1->stride_w) * eb, static_cast<cuuint64_t>(x1->stride_h) * eb,
                        static_cast<cuuint64_t>(x1->stride_n) * eb};
  cuuint64_t ystr[3] = {static_cast<cuuint64_t>(y->stride_w) * eb, static_cast<cuuint64_t>(y->stride_h) * eb,
                        static_cast<cuuint64_t>(y->stride_n) * eb};
  cuuint32_t xbox[4] = {32, static_cast<cuuint32_t>(xw), static_cast<cuuint32_t>(xh), 1};
  cuuint32_t ybox[4] = {32, static_cast<cuuint32_t>(yw), static_cast<cuuint32_t>(yh), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUtensorMap xmap, ymap;
  const CUtensorMapSwizzle swz = bf ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  const CUtensorMapDataType dt = bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if (tiled_map(&xmap, 4, x1->data, xdims, xstr, xbox, estr, swz, dt) != CUDA_SUCCESS ||
      tiled_map(&ymap, 4, y->data, xdims, ystr, ybox, estr, swz, dt) != CUDA_SUCCESS)
    return CB_ERR_UNSUPPORTED;
  const cudaError_t e = launch_stage_body_tc(xmap, ymap, a, dev->sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

cb_status cb_stage_body(const cb_tensor* x1, const float* w1, const float* s1, const float* b1, const float* w2,
                        const float* s2, const float* b2, const float* w3, const float* s3, const float* b3,
                        cb_act act, cb_tensor* y, void* stream) {
  if (!view_ok(x1) || !view_ok(y) || !w1 || !s1 || !b1 || !w2 || !s2 || !b2 || !w3 || !s3 || !b3)
    return CB_ERR_INVALID_ARG;
  if (act != CB_ACT_NONE && act != CB_ACT_RELU && act != CB_ACT_SILU) return CB_ERR_INVALID_ARG;
  if (y->n != x1->n || y->h != x1->h || y->w != x1->w || y->c != x1->c || y->dtype != x1->dtype)
    return CB_ERR_INVALID_ARG;
  if (overlap(x1, y)) return CB_ERR_INVALID_ARG;
  if ((x1->c != 16 && x1->c != 32) || x1->layout != CB_LAYOUT_NHWC || y->layout != CB_LAYOUT_NHWC)
    return CB_ERR_UNSUPPORTED;
  // x1 pixels in whole 16-byte pieces (the copy's strides), y in pieces of 4 channels
  const long long xm = is_f32(x1) ? 4 : 8;
  if (!aligned16(x1->data) || !aligned16(y->data) || x1->stride_w % xm != 0 || x1->stride_h % xm != 0 ||
      x1->stride_n % xm != 0 || !strides_mult4(y))
    return CB_ERR_ALIGNMENT;
  // the 32-channel kernel writes y by tensor stores: strides in whole 16-byte pieces
  if (x1->c == 32 && (y->stride_w % xm != 0 || y->stride_h % xm != 0 || y->stride_n % xm != 0))
    return CB_ERR_ALIGNMENT;
  if (x1->n == 0) return CB_OK;
  if (x1->n > 65535 || x1->h > 65535 || x1->w > 65535 || !encode_tiled()) return CB_ERR_UNSUPPORTED;
  DeviceInfo* dev = nullptr;
  cb_status st = current_device(&dev);
  if (st != CB_OK) return st;
  if (x1->c == 32) return stage_body_tc(x1, w1, s1, b1, w2, s2, b2, w3, s3, b3, act, y, dev, stream);
  StageBodyArgs a{};
  a.x = x1->data;
  a.xs_n = x1->stride_n;
  a.xs_h = x1->stride_h;
  a.xs_w = x1->stride_w;
  a.y = y->data;
  a.ys_n = y->stride_n;
  a.ys_h = y->stride_h;
  a.ys_w = y->stride_w;
  a.N = x1->n;
  a.H = x1->h;
  a.W = x1->w;
  // weights (host OHWI) into the launch's parameter block, [ci pair][co][ci % 2] (per tap for w2)
  for (int cp = 0; cp < 8; ++cp)
    for (int co = 0; co < 8; ++co)
      for (int e = 0; e < 2; ++e) a.w1[(cp * 8 + co) * 2 + e] = w1[co * 16 + 2 * cp + e];
  for (int tap = 0; tap < 9; ++tap)
    for (int cp = 0; cp < 4; ++cp)
      for (int co = 0; co < 8; ++co)
        for (int e = 0; e < 2; ++e) a.w2[((tap * 4 + cp) * 8 + co) * 2 + e] = w2[(co * 9 + tap) * 8 + 2 * cp + e];
  for (int cp = 0; cp < 8; ++cp)
    for (int co = 0; co < 16; ++co)
      for (int e = 0; e < 2; ++e) a.w3[(cp * 16 + co) * 2 + e] = w3[co * 16 + 2 * cp + e];
  for (int c = 0; c < 8; ++c) {
    a.sb[c] = s1[c], a.sb[8 + c] = b1[c];
    a.sb[16 + c] = s2[c], a.sb[24 + c] = b2[c];
  }
  for (int c = 0; c < 16; ++c) a.sb[32 + c] = s3[c], a.sb[48 + c] = b3[c];
  a.act = static_cast<int>(act);
  a.bf16 = is_f32(x1) ? 0 : 1;
  a.err = dev->err;
  a.timeout_ns = timeout_ns();
  // x1 as (C = 16, W, H, N); one box is a tile's haloed pixels
  const cuuint64_t eb = elem_bytes(x1);
  int bc = 0, bw = 0, bh = 0;
  stage_body_box(&bc, &bw, &bh);
  cuuint64_t dims[4] = {16, static_cast<cuuint64_t>(x1->w), static_cast<cuuint64_t>(x1->h),
                        static_cast<cuuint64_t>(x1->n)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(x1->stride_w) * eb, static_cast<cuuint64_t>(x1->stride_h) * eb,
                           static_cast<cuuint64_t>(x1->stride_n) * eb};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(bc), static_cast<cuuint32_t>(bw), static_cast<cuuint32_t>(bh), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUtensorMap xmap;
  if (tiled_map(&xmap, 4, x1->data, dims, strides, box, estr,
                is_f32(x1) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
                is_f32(x1) ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != CUDA_SUCCESS)
    return CB_ERR_UNSUPPORTED;
  const cudaError_t e = launch_stage_body(xmap, a, dev->sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

// ------------------------------------------------ no-allocation block variant
// The scratch of cb_dw_separable_block_static.  Host code cannot use this
// name as a device address; it looks the address up per device below.
static __device__ __align__(256) unsigned char g_block_scratch[CB_STATIC_SCRATCH_BYTES];

static std::mutex g_scratch_mu;
static void* g_scratch_addr[128];

cb_status cb_dw_separable_block_static(const cb_tensor* x, const float* dw_w, const float* dw_scale,
                                       const float* dw_bias, const float* pw_w, const float* pw_scale,
                                       const float* pw_bias, const float* skip_w, const float* skip_scale,
                                       const float* skip_bias, int stride, cb_tensor* y, void* stream) {
  if (!view_ok(x) || !view_ok(y)) return CB_ERR_INVALID_ARG;
  if (!is_f32(x) || !is_f32(y)) return CB_ERR_UNSUPPORTED;
  size_t need = 0;
  cb_status st = cb_dw_separable_block_workspace(x, y->c, stride, &need);
  if (st != CB_OK) return st;
  if (need > CB_STATIC_SCRATCH_BYTES) return CB_ERR_WORKSPACE;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 128) return CB_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_block_scratch);
      if (e != cudaSuccess) return cuda_fail(e);
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  return cb_dw_separable_block(x, dw_w, dw_scale, dw_bias, pw_w, pw_scale, pw_bias, skip_w, skip_scale, skip_bias,
                               stride, y, scratch, CB_STATIC_SCRATCH_BYTES, stream);
}

cb_status cb_avgpool_linear(const cb_tensor* x, const float* fc_w, const float* fc_b, int out_features, float* out,
                            void* stream) {
  if (!view_ok(x) || x->layout != CB_LAYOUT_NHWC || !fc_w || !fc_b || !out || out_features < 1)
    return CB_ERR_INVALID_ARG;
  if (!is_f32(x)) return CB_ERR_UNSUPPORTED;
  if (x->c > 12 * 1024) return CB_ERR_UNSUPPORTED;
  if (x->n == 0) return CB_OK;
  PoolFcArgs a{};
  a.x = static_cast<const float*>(x->data);
  a.xs_n = x->stride_n;
  a.xs_h = x->stride_h;
  a.xs_w = x->stride_w;
  a.N = x->n;
  a.H = x->h;
  a.W = x->w;
  a.C = x->c;
  a.out_features = out_features;
  a.fc_w = fc_w;
  a.fc_b = fc_b;
  a.out = out;
  cudaError_t e = launch_pool_fc(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

static cb_status check_preprocess(const unsigned char* src, int n, int src_h, int src_w, long long src_pitch,
                                  const float* dst, int dst_h, int dst_w) {
  if (!src || !dst || n < 0 || src_h < 1 || src_w < 1 || dst_h < 1 || dst_w < 1) return CB_ERR_INVALID_ARG;
  if (src_pitch < 3LL * src_w) return CB_ERR_INVALID_ARG;
  if (8LL * ((3LL * src_w + 15) & ~15LL) > 224 * 1024) return CB_ERR_UNSUPPORTED;  // two buffers of four rows
  if (dst_h > 65535 || n > 65535) return CB_ERR_UNSUPPORTED;
  return CB_OK;
}

cb_status cb_preprocess_u8(const unsigned char* src, int n, int src_h, int src_w, long long src_pitch, float* dst,
                           int dst_h, int dst_w, void* stream) {
  cb_status st = check_preprocess(src, n, src_h, src_w, src_pitch, dst, dst_h, dst_w);
  if (st != CB_OK) return st;
  DeviceInfo* dev = nullptr;
  st = current_device(&dev);
  if (st != CB_OK) return st;
  cudaError_t e = launch_preprocess_fused(src, n, src_h, src_w, src_pitch, dst, dst_h, dst_w, dev->sms,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

cb_status cb_preprocess_stem_u8(const unsigned char* src, int n, int src_h, int src_w, long long src_pitch,
                                int dst_h, int dst_w, const float* w, const float* scale, const float* bias, cb_act act,
                                cb_tensor* y, void* stream) {
  if (!src || !w || !scale || !bias || !view_ok(y) || n < 0 || src_h < 1 || src_w < 1 || dst_h < 1 || dst_w < 1)
    return CB_ERR_INVALID_ARG;
  if (!is_f32(y)) return CB_ERR_UNSUPPORTED;
  if (src_pitch < 3LL * src_w || act < CB_ACT_NONE || act > CB_ACT_SILU) return CB_ERR_INVALID_ARG;
  if (y->layout != CB_LAYOUT_NHWC || y->n != n || y->c != 16 || y->h != (dst_h - 1) / 2 + 1 ||
      y->w != (dst_w - 1) / 2 + 1)
    return CB_ERR_INVALID_ARG;
  if (n == 0) return CB_OK;
  if (!aligned16(src) || src_pitch % 16 != 0 || (3LL * src_w) % 16 != 0 || dst_w % 4 != 0) return CB_ERR_ALIGNMENT;
  if (!aligned16(y->data) || !strides_mult4(y)) return CB_ERR_ALIGNMENT;
  if (n > 65535 || src_h > (1 << 22) || src_w > (1 << 20) || dst_h > (1 << 22) || dst_w > (1 << 20))
    return CB_ERR_UNSUPPORTED;
  uintptr_t ylo, yhi;
  view_range(y, &ylo, &yhi);
  const uintptr_t slo = reinterpret_cast<uintptr_t>(src);
  const uintptr_t shi = slo + static_cast<uintptr_t>((static_cast<long long>(n) * src_h - 1) * src_pitch + 3LL * src_w);
  if (slo < yhi && ylo < shi) return CB_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  cb_status st = current_device(&dev);
  if (st != CB_OK) return st;
  StemArgs a{};
  a.src = src;
  a.N = n;
  a.H = dst_h;
  a.W = dst_w;
  a.OH = y->h;
  a.OW = y->w;
  a.hs = src_h;
  a.ws = src_w;
  a.pitch = src_pitch;
  int rows = 0;
  stem_src_bounds(src_h, src_w, dst_h, dst_w, &rows, &a.row_cap);
  a.w = w;
  a.ep = make_epilogue(scale, bias, act, nullptr, CB_RES_NONE);
  a.out = make_out(y);
  stem_tile_grid(a.OH, a.OW, &a.tiles_y, &a.tiles_x);
  if (static_cast<long long>(n) * a.tiles_y * a.tiles_x >= (1LL << 31)) return CB_ERR_UNSUPPORTED;
  const size_t smem = stem_smem_bytes(2, rows, a.row_cap);
  if (smem > 227 * 1024) return CB_ERR_UNSUPPORTED;  // too strong a downscale for one tile's source rows
  const cudaError_t e = launch_stem(a, 2, smem, dev->sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

cb_status cb_preprocess_u8_three_pass(const unsigned char* src, int n, int src_h, int src_w, long long src_pitch,
                                      unsigned char* tmp_u8, float* tmp_f32, float* dst, int dst_h, int dst_w,
                                      void* stream) {
  cb_status st = check_preprocess(src, n, src_h, src_w, src_pitch, dst, dst_h, dst_w);
  if (st != CB_OK) return st;
  if (!tmp_u8 || !tmp_f32) return CB_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_preprocess_resize(src, n, src_h, src_w, src_pitch, tmp_u8, dst_h, dst_w, s);
  if (e == cudaSuccess) e = launch_preprocess_normalize(tmp_u8, static_cast<long long>(n) * dst_h * dst_w * 3, tmp_f32, s);
  if (e == cudaSuccess) e = launch_preprocess_layout(tmp_f32, n, dst_h, dst_w, dst, s);
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

cb_status cb_get_device_error(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  DeviceInfo* dev = nullptr;
  cb_status st = current_device(&dev);
  if (st != CB_OK) return st;
  int v = 0;
  e = cudaMemcpy(&v, dev->err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpy(dev->err, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e);
    return static_cast<cb_status>(v);
  }
  return CB_OK;
}

cb_status cb_debug_sample_coords(int src_extent, int dst_extent, int* i0, int* i1, float* frac, void* stream) {
  if (src_extent < 1 || dst_extent < 1 || !i0 || !i1 || !frac) return CB_ERR_INVALID_ARG;
  const cudaError_t e =
      launch_sample_coords(src_extent, dst_extent, i0, i1, frac, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

cb_status cb_debug_timeout_probe(int timeout_ms, void* stream) {
  if (timeout_ms < 1 || timeout_ms > 10000) return CB_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  cb_status st = current_device(&dev);
  if (st != CB_OK) return st;
  cudaError_t e = launch_timeout_probe(dev->err, static_cast<uint64_t>(timeout_ms) * 1000000ull,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CB_OK : cuda_fail(e);
}

int cb_last_cuda_error(void) { return t_last_cuda_error; }

const char* cb_status_string(cb_status s) {
  switch (s) {
    case CB_OK: return "CB_OK";
    case CB_ERR_INVALID_ARG: return "CB_ERR_INVALID_ARG";
    case CB_ERR_UNSUPPORTED: return "CB_ERR_UNSUPPORTED";
    case CB_ERR_ALIGNMENT: return "CB_ERR_ALIGNMENT";
    case CB_ERR_CUDA: return "CB_ERR_CUDA";
    case CB_ERR_TIMEOUT: return "CB_ERR_TIMEOUT";
    case CB_ERR_WORKSPACE: return "CB_ERR_WORKSPACE";
  }
  return "CB_ERR_UNKNOWN";
}

int cb_version(void) { return kVersion; }

cb_status cb_set_tuning(const char* name, const char* value) {
  if (!name) return CB_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_tuning_mu);
  Tuning t = tuning_locked();
  if (!parse_tuning(&t, name, value)) return CB_ERR_INVALID_ARG;
  tuning_locked() = t;
  return CB_OK;
}

cb_status cb_last_launch(cb_launch_info* info) {
  if (!info) return CB_ERR_INVALID_ARG;
  const LaunchRecord& r = last_launch();
  if (!r.kernel) return CB_ERR_INVALID_ARG;
  info->grid = static_cast<int>(r.grid.x * r.grid.y * r.grid.z);
  info->threads = static_cast<int>(r.block.x * r.block.y * r.block.z);
  info->smem_bytes = r.smem;
  info->cluster = r.cluster;
  int per_sm = 0;
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, r.kernel, info->threads, r.smem);
  if (e != cudaSuccess) return cuda_fail(e);
  info->blocks_per_sm = per_sm;
  const char* name = nullptr;
  if (cudaFuncGetName(&name, r.kernel) != cudaSuccess) {
    cudaGetLastError();
    name = nullptr;
  }
  info->kernel = name ? name : "?";
  return CB_OK;
}

cb_status cb_set_kernel_policy(int policy) {
  if (policy < 0 || policy > 2) return CB_ERR_INVALID_ARG;
  g_policy.store(policy);
  return CB_OK;
}

int cb_get_kernel_policy(void) { return g_policy.load(); }

// Profiling aid (not part of cb.h): copies out the implicit-GEMM timeline
// recorded while CB_IGEMM_TRACE is set; returns the number of records.
int cb_debug_igemm_trace(unsigned long long* out, int max_records) {
  cudaDeviceSynchronize();
  return igemm_read_trace(out, max_records);
}

// Profiling aid (not part of cb.h): per-CTA (start ns, end ns, SM) of the
// traced halo-kernel launches in slots 1 and 2 (CB_SPAN_SLOT), then cleared;
// returns the number of CTA rows copied (2 x 1024).
int cb_debug_igemm_spans(unsigned long long* out, int max_ctas) {
  cudaDeviceSynchronize();
  return igemm_read_spans_halo(out, max_ctas);
}

int cb_conv_path(const cb_tensor* x, const cb_tensor* y, int kh, int stride, int pad, int groups) {
  if (!view_ok(x) || !view_ok(y) || (kh != 1 && kh != 3) || (stride != 1 && stride != 2)) return 0;
  if (pad < 0 || pad > kh / 2) return 0;
  if (groups == x->c && groups == y->c && groups > 1) return kh == 3 && x->dtype == y->dtype ? CB_PATH_DEPTHWISE : 0;
  if (groups != 1 || x->dtype != y->dtype) return 0;
  return dense_path(x, y, kh, stride, pad, nullptr);
}

int cb_layer_uses_tensor_cores(int ci, int co, int kh, int stride, int groups) {
  if (ci < 1 || co < 1 || groups != 1 || (kh != 1 && kh != 3) || (stride != 1 && stride != 2)) return 0;
  return tc_shape(ci, co, kh, stride, kh / 2) ? 1 : 0;
}

}  // extern "C"
