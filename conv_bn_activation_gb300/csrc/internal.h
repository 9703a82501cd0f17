// Internal launch interfaces between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace cb {

// Per-channel epilogue shared by every conv kernel:
//   z = acc * scale[c] + bias[c];  z += r (pre);  z = act(z);  z += r (post)
struct Epilogue {
  const float* scale;
  const float* bias;
  int act;       // 0 none, 1 relu, 2 silu
  int res_mode;  // 0 none, 1 pre-act, 2 post-act
  const float* r;
  long long rs_n, rs_h, rs_w;  // residual strides (elements, c stride 1)
};

struct OutView {
  float* y;
  long long ys_n, ys_h, ys_w;  // c stride 1
};

// ------------------------------------------------------------ depthwise 3x3
struct DwArgs {
  const float* x;
  long long xs_n, xs_h, xs_w;  // NHWC, c stride 1
  const float* w;              // [3][3][C]
  int N, H, W, C, OH, OW, stride, pad;
  OutView out;
  Epilogue ep;
  int bf16;  // x, y and r hold bfloat16 (TMA kernel only); w, scale, bias fp32
};
// Plain CUDA-core kernel: one thread per (output pixel, 4 or 1 channels).
cudaError_t launch_dw_simple(const DwArgs& a, bool vec4, cudaStream_t s);

// TMA-fed kernel: persistent CTAs stream input rows (32-channel chunks,
// full padded width of a column tile) through a shared-memory ring; each
// consumer thread owns two adjacent output columns x 4 channels and slides
// its 3x3 windows down the rows in registers.
struct DwTmaPlan {
  int rows_per_item;  // output rows per work item
  int num_items;
  int tile_w;         // output columns per item
  int box_w;          // input columns per row copy (includes the halo)
  int stages;
  int grid;
  int consumer_warps;
  int w_smem;  // bf16 at stride 1: the 9 x C taps staged in shared memory after the barriers
  size_t smem_bytes;
};
// debug_skip_row = 1 is fault injection for tests of the bounded waits: the
// producer of CTA 0 withholds the copy (and the barrier arrive) of its first
// input row, so the consumers' wait on it runs out, the kernel records
// CB_ERR_TIMEOUT and returns.
cudaError_t launch_dw_tma(const CUtensorMap& xmap, const DwArgs& a, const DwTmaPlan& plan, int* err,
                          uint64_t timeout_ns, int debug_skip_row, cudaStream_t s);

// ---------------------------------------------------------- direct (CUDA core)
struct DirectArgs {
  const float* x;
  long long xs_n, xs_h, xs_w, xs_c;  // any layout
  const float* w;                    // OHWI [Co][kh][kw][Ci]
  int N, H, W, Ci, Co, OH, OW, kh, kw, stride, pad;
  OutView out;
  Epilogue ep;
  int bf16;  // x, y and r hold bfloat16 (pointwise kernel only); w, scale, bias fp32
};
cudaError_t launch_direct(const DirectArgs& a, int sms, cudaStream_t s);
// 3x3 stride-1 pad-1 layers with 8 input and 8 output channels (conv3x3_c8.cu):
// NHWC fp32 x, y (and residual) with 16-byte aligned pixels and strides that
// are multiples of 4 elements; cudaErrorInvalidValue for anything else.
bool conv3x3_c8_ok(const DirectArgs& a);
cudaError_t launch_conv3x3_c8(const DirectArgs& a, int sms, cudaStream_t s);
// 1x1 stride-1 layers with Ci, Co in {4, 8, 16, 32} (pointwise.cu): needs
// NHWC views with 16-byte aligned pixels; flat = every view's pixels are
// evenly spaced (stride_h = W * stride_w, stride_n = H * stride_h).  With
// bf16 storage Ci >= 8 (a pixel holds at least one 16-byte piece).
bool pointwise_small_ok(int ci, int co, bool bf16 = false);
cudaError_t launch_pointwise_small(const DirectArgs& a, bool flat, int sms, cudaStream_t s);

// ------------------------------------------------------- implicit GEMM (tcgen05)
struct IgemmArgs {
  int M;         // N*OH*OW output pixels
  int OHW, OW;   // OH*OW, OW
  int Cout;
  int kw, taps;  // filter width, kh*kw
  int num_kc;    // ceil(Cin / KC), KC = channels per K step (8, 16 or 32)
  int k_iters;   // taps * num_kc
  int m_tiles, n_tiles;
  int stride, pad;
  int stages;
  int vec_store;  // 1 when y / r rows allow 16-byte vector access
  // Pixel tiles: blk_w == 0 -> 128 consecutive output pixels in (n, oh, ow)
  // order, A gathered by an im2col-mode copy; else blocks of blk_h x blk_w
  // output pixels (blk_h * blk_w == 128) of one image, A loaded per filter
  // tap by a tiled copy with element strides = conv stride.
  int blk_w, blk_h, blocks_x, blocks_y;
  OutView out;
  Epilogue ep;
  int* err;
  uint64_t timeout_ns;
  int trace;      // 1: record the pipeline timeline of CTA trace_cta (profiling aid)
  int trace_cta;
  int bf16;       // 1: x, w, y and r hold bfloat16 (kind::f16 MMAs); kc then counts 4-byte units of a row
};
int igemm_read_trace(unsigned long long* out, int max_records);
cudaError_t launch_igemm(const CUtensorMap& amap, const CUtensorMap& bmap, const IgemmArgs& a, int bn, int kc,
                         int grid, size_t smem_bytes, cudaStream_t s);
size_t igemm_smem_bytes(int bn, int kc, int stages);
int igemm_stages(int bn, int kc);

// Halo-tile variant for 3x3 stride-1 pad-1 layers with Cin % 32 == 0: one
// shared-memory tile of input rows per 32-channel chunk serves all nine taps
// (igemm_halo.cuh).
struct HaloArgs {
  // Stride 1: input = output size; output pixels of a column block of blk_w
  // columns are numbered over Wp = blk_w + 2.  Stride 2: the input is loaded
  // as four phase tiles (even / odd rows x columns) and the output pixels are
  // numbered over Wp = blk_w + 1.  n_blk column blocks per image.
  int H, W, Wp;        // input height / width; Wp = padded width of the pixel numbering
  int stride;          // 1 or 2
  int OH, OW;          // output height / width
  int blk_w, n_blk;    // output columns per block, blocks per image row
  int px_tiles_per_blk;  // ceil(OH * Wp / PX): PX-pixel sub-tiles per column block
  int sub;             // sub-tiles per tile (one halo copy for all of them; pixel-major only)
  int tiles_per_blk;   // ceil(px_tiles_per_blk / sub)
  int phase_bytes;     // stride 2: shared-memory bytes of one phase tile (halo_bytes = 4 of them)
  int Cout;
  int kc;              // input channels per chunk: 32, or 16 (64-byte rows)
  int num_kc;          // Cin / kc
  int tiles_per_img;   // n_blk * tiles_per_blk
  int m_tiles;         // N * tiles_per_img
  int n_tiles;         // ceil(Cout / BN)
  int rows;            // input rows per halo copy
  int halo_bytes;      // shared-memory bytes of one halo buffer (multiple of 1024)
  int nb_stages;       // weight-slice ring depth
  int taps_per_stage;  // filter taps per weight-ring stage (1, 3 or 9): one copy each
  int w_resident;      // 1: one chunk and one channel tile; the nine taps stay in the single stage
  int split_k;         // 1, or 2: clusters of two CTAs split each tile's chunks (one tile per cluster)
  int vec_store;       // 1 when y / r rows allow 16-byte vector access
  OutView out;
  Epilogue ep;
  int* err;
  uint64_t timeout_ns;
  int trace;           // 1: record the pipeline timeline of CTA trace_cta (profiling aid)
  int trace_cta;
  int bf16;            // 1: x, w, y and r hold bfloat16 (kind::f16 MMAs); kc counts 4-byte units of a row
};
// Input rows one halo copy spans for a tile of px pixels at padded width
// wp, and the buffer bytes (rows * wp pixels of 128 bytes, plus 8 rows that
// only the discarded padding columns of the last rows read).
constexpr int kHaloMaxSub = 4;  // 128-pixel sub-tiles per halo tile, at most
int halo_rows(int wp, int px, int stride = 1);
int halo_buffer_bytes(int wp, int px, int kc = 32, int stride = 1);
size_t halo_smem_bytes(int co, int halo_bytes, int nb_stages, int taps_per_stage = 1, int kc = 32);
// Shared-memory bytes a split-K CTA receives from its partner (half of one
// accumulator), which must fit in its halo and weight buffers.
size_t halo_split_recv_bytes(int px, int co, bool cm);
// Clusters of two CTAs of this tile shape and shared-memory size that the
// device runs at once (0 if it cannot run them).
int halo_max_pairs(int px, int co, bool cm, size_t smem_bytes);
// px x co tile: 128 x {32, 64, 128, 256} pixel-major, or 256 x 128 / 192 x 128 channel-major (cm).
cudaError_t launch_igemm_halo(const CUtensorMap& xmap, const CUtensorMap& wmap, const HaloArgs& a, int px, int co,
                              bool cm, int grid, size_t smem_bytes, cudaStream_t s);

// ------------------------------------------- depthwise-separable block
// One block in one kernel (dw_block.cu): NHWC fp32 x and y with 16-byte
// aligned pixels, Ci % 4 == 0, Co % 32 == 0 and Co <= 256; pointwise and
// skip weights OHWI [Co][Ci] read by TMA (maps of dims (Ci, 1, Co), box
// (32, 1, Co), 128-byte swizzle).
struct DwBlockArgs {
  const float* x;
  long long xs_n, xs_h, xs_w;
  int N, H, W, Ci, Co, OH, OW, stride, M;
  const float* dw_w;       // [9][Ci]
  const float* dw_scale;
  const float* dw_bias;
  const float* pw_scale;
  const float* pw_bias;
  const float* sk_scale;   // skip conv only
  const float* sk_bias;
  int skip_conv;           // 1: 1x1 conv skip (second accumulator); 0: identity
  int num_kc;              // ceil(Ci / 32)
  uint32_t tmem_cols;      // power of two >= Co (x 2 with a conv skip)
  OutView out;
  int* err;
  uint64_t timeout_ns;
  int trace;           // 1: record the pipeline timeline of CTA trace_cta (profiling aid)
  int trace_cta;
};
size_t dw_block_smem_bytes(int ci, int co);
cudaError_t launch_dw_block(const CUtensorMap& pw_map, const CUtensorMap& sk_map, const DwBlockArgs& a,
                            cudaStream_t s);

// ------------------------------------------------------------------- stem
// 3 -> 16 channels, 3x3, stride 2, pad 1, CUDA cores (stem.cu).  Input:
// planar fp32 (src_kind 0: x[n*xs_n + c*xs_c + h*xs_h + w]), packed NHWC
// fp32 (1: x[n*xs_n + h*xs_h + 3*w + c]), u8 frames preprocessed on the
// fly (2: [n][hs][pitch] bytes, 3 channels per pixel, resized to H x W), or
// packed NHWC bf16 (3, with bf16 output and residual; W % 8 == 0, strides
// multiples of 8 elements).
// Needs W % 4 == 0, 16-byte aligned bases and strides that are multiples of
// 4 elements (of 16 bytes for the frames, whose rows are a multiple of 16
// bytes), a 16-byte aligned output view with strides that are multiples of 4.
struct StemArgs {
  const void* src;
  long long xs_n, xs_h, xs_c;
  int N, H, W, OH, OW;
  int hs, ws;          // u8 frames: source size
  long long pitch;     // u8 frames: bytes per source row
  int row_cap;         // u8 frames: bytes per staged source row
  const float* w;      // OHWI [16][3][3][3]
  Epilogue ep;         // residual (if any): 16-byte aligned, strides multiples of 4
  OutView out;
  int tiles_x, tiles_y;
  int* err;             // tensor-core kernel: device error word, bound of its waits
  uint64_t timeout_ns;
};
void stem_tile_grid(int OH, int OW, int* tiles_y, int* tiles_x);
// Staged source rows per tile and bytes per staged row for a hs x ws -> hd x wd resize.
void stem_src_bounds(int hs, int ws, int hd, int wd, int* rows, int* row_cap);
size_t stem_smem_bytes(int src_kind, int src_rows, int row_cap);
cudaError_t launch_stem(const StemArgs& a, int src_kind, size_t smem, int sms, cudaStream_t s);
// ------------------------------------------- YOLO-style stage body, C = 16
// out = act(s3 * conv1x1([a | b]) + b3) + x1 with a = act(s1 * conv1x1(x1) + b1)
// (16 -> 8) and b = act(s2 * conv3x3(a) + b2) (8 -> 8, pad 1), in one kernel
// (stage_body.cu).  x1 and out are NHWC with 16 channels, fp32 or bf16
// storage.  The weights and the folded BN travel in the launch's parameter
// block (4 KB), each weight pair where the kernel's unrolled loops read it
// by a constant offset: [input channel pair][output channel][2] (per tap
// for w2).  The caller encodes xmap: x1 as a 4-D tensor (C = 16, W, H, N)
// with the box stage_body_box gives and the 64-byte (fp32) or 32-byte
// (bf16) swizzle.
struct StageBodyArgs {
  const void* x;
  long long xs_n, xs_h, xs_w;
  void* y;
  long long ys_n, ys_h, ys_w;
  int N, H, W;
  int act;
  int bf16;
  int* err;  // device error word, bound of the kernel's waits
  uint64_t timeout_ns;
  float w1[8 * 8 * 2];      // 1x1 16 -> 8
  float w2[9 * 4 * 8 * 2];  // 3x3 8 -> 8
  float w3[8 * 16 * 2];     // 1x1 16 -> 16
  float sb[2 * (8 + 8 + 16)];  // s1[8] b1[8] s2[8] b2[8] s3[16] b3[16]
};
void stage_body_box(int* box_c, int* box_w, int* box_h);
cudaError_t launch_stage_body(const CUtensorMap& xmap, const StageBodyArgs& a, int sms, cudaStream_t s);

// The same body for C = 32 channels (h = 16) on the tensor cores
// (stage_body_tc.cu): fp32 storage with TF32 operands, or bf16 storage with
// bf16 operands.  wimg is the weights' shared-memory image: the B operands as
// K-major rows with the tensor core's swizzle (16-byte piece q of row r at
// q ^ (r % 8) for 128-byte rows, q ^ (r / 2 % 4) for 64-byte rows,
// q ^ (r / 4 % 2) for 32-byte rows).  fp32 (TF32-rounded): w1 [16 co][32 ci]
// (128-byte rows) at byte 0, w2 per tap kh * 3 + kw [16 co][16 ci] (64-byte
// rows) at 2048 + 1024 * tap, w3 [32 co][32 ci of a | b] (128-byte rows) at
// 11264.  bf16 (nearest even; 64-byte rows for w1 and w3, 32-byte for w2):
// w1 at 0 and its tail bf16(w1 - bf16(w1)) at 1024, w2 at 2048 + 512 * tap,
// w3 at 7168 and its tail at 9216.  The caller encodes xmap (x1
// as (C = 32, W, H, N) of the storage type, the swizzle of its rows: 128
// bytes fp32, 64 bf16; box 32 x x_box_w x x_box_h x 1) and ymap (y likewise,
// box 32 x y_box_w x y_box_h x 1) with the sizes stage_body_tc_boxes gives.
constexpr int kStageTcWImgWords = (2048 + 9 * 1024 + 4096) / 4;
struct StageBodyTcArgs {
  const void* x;  // x1, for the residual (fp32 or bf16)
  long long xs_n, xs_h, xs_w;
  int N, H, W;
  int act;
  int* err;  // device error word, bound of the kernel's waits
  uint64_t timeout_ns;
  int bf16;          // x1, y and the weights' image hold bfloat16
  int debug_skip_x;  // 1: fault injection for tests of the bounded waits (no warpgroup issues its first x1 copy)
  uint32_t wimg[kStageTcWImgWords];
  float sb[2 * (16 + 16 + 32)];  // s1[16] b1[16] s2[16] b2[16] s3[32] b3[32]
};
void stage_body_tc_boxes(int* x_box_w, int* x_box_h, int* y_box_w, int* y_box_h);
cudaError_t launch_stage_body_tc(const CUtensorMap& xmap, const CUtensorMap& ymap, const StageBodyTcArgs& a, int sms,
                                 cudaStream_t s);

// The same layer on the tensor cores (stem_tc.cu) at fp32 accuracy, for packed
// NHWC input (src kinds 1 and 3: fp32, or bf16 storage with a bf16 output);
// tiles_x / tiles_y are its own (2 x 64 output pixels).  stem_tc_ok: the tile
// count fits the kernel's int tile index.
bool stem_tc_ok(const StemArgs& a);
cudaError_t launch_stem_tc(const StemArgs& a, bool bf16, int sms, cudaStream_t s);

// -------------------------------------------------------------- preprocess
cudaError_t launch_preprocess_fused(const uint8_t* src, int n, int hs, int ws, long long pitch, float* dst,
                                    int hd, int wd, int sms, cudaStream_t s);
// Sample coordinates (i0, i1, a) along one axis, as the preprocess kernels compute them.
cudaError_t launch_sample_coords(int S, int D, int* i0, int* i1, float* a, cudaStream_t s);
cudaError_t launch_preprocess_resize(const uint8_t* src, int n, int hs, int ws, long long pitch,
                                     uint8_t* out, int hd, int wd, cudaStream_t s);
cudaError_t launch_preprocess_normalize(const uint8_t* in, long long count, float* out, cudaStream_t s);
cudaError_t launch_preprocess_layout(const float* in, int n, int h, int w, float* out, cudaStream_t s);

// ------------------------------------------------------------ watchdog hook
cudaError_t launch_timeout_probe(int* err, uint64_t limit_ns, cudaStream_t s);

// ----------------------------------------------------------------- pool + fc
struct PoolFcArgs {
  const float* x;
  long long xs_n, xs_h, xs_w;
  int N, H, W, C, out_features;
  const float* fc_w;
  const float* fc_b;
  float* out;
};
cudaError_t launch_pool_fc(const PoolFcArgs& a, cudaStream_t s);

}  // namespace cb
