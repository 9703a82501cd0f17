/*
 * cb.h -- C ABI of the fused convolution + BatchNorm + activation library
 * for one GB300 GPU (sm_103a).
 *
 * The operation ("YOLO26N Inference Optimisation": nsys breakdown and
 * improvement #7; "How I sped up convolutions": the Metal kernel walk-through,
 * steps 1-5) is
 *
 *     y = act( scale[c] * conv(x, w)[n,oh,ow,c] + bias[c]  (+ r, pre-act) )  (+ r, post-act)
 *
 * where (scale, bias) is inference BatchNorm folded per output channel,
 * act is identity, ReLU = max(0, z) or SiLU = z / (1 + exp(-z)).
 *
 * Conventions for every entry point:
 *  - All memory is owned by the caller.  Tensor and weight pointers are
 *    DEVICE pointers unless the argument says "host".  The library never
 *    allocates device memory and never synchronises inside the compute calls
 *    (cb_get_device_error is the one call that synchronises).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Work is enqueued asynchronously on it.
 *  - Arguments are validated on the host before anything is launched.  Bad
 *    pointers/shapes return CB_ERR_INVALID_ARG, shapes outside the supported
 *    set CB_ERR_UNSUPPORTED, misaligned data CB_ERR_ALIGNMENT.  A failed
 *    launch returns CB_ERR_CUDA (cb_last_cuda_error() gives the cudaError_t).
 *  - Kernels that wait on barriers give up after a bounded time, record
 *    CB_ERR_TIMEOUT in a device error word and return; cb_get_device_error()
 *    reports and clears it.
 *  - Activations are fp32.  Layout is NHWC (channel-last) unless a tensor
 *    says CB_LAYOUT_NCHW.  Output rows may be padded: y->stride_h may exceed
 *    y->w * y->stride_w; padding columns are never written (the OW tail of
 *    the last tile is masked -- "YOLO26N Inference Optimisation", Bug fixed:
 *    TMA overflow).
 */
#ifndef CB_H_
#define CB_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CB_OK = 0,
  CB_ERR_INVALID_ARG = 1,
  CB_ERR_UNSUPPORTED = 2,
  CB_ERR_ALIGNMENT = 3,
  CB_ERR_CUDA = 4,
  CB_ERR_TIMEOUT = 5,
  CB_ERR_WORKSPACE = 6
} cb_status;

typedef enum { CB_ACT_NONE = 0, CB_ACT_RELU = 1, CB_ACT_SILU = 2 } cb_act;

/* Where the residual r enters: act(z + r) or act(z) + r. */
typedef enum { CB_RES_NONE = 0, CB_RES_PRE_ACT = 1, CB_RES_POST_ACT = 2 } cb_res_mode;

typedef enum { CB_LAYOUT_NHWC = 0, CB_LAYOUT_NCHW = 1 } cb_layout;

/*
 * Element type of an activation view.  CB_DTYPE_F32 (0, the default of a
 * zero-initialised view) everywhere; CB_DTYPE_BF16 (bfloat16: the upper half
 * of an fp32) is the half-size storage variant, taken by the depthwise 3x3,
 * the narrow 1x1 and the tensor-core layers of cb_conv_bn_act: a 16-bit main
 * data type is the first of the next steps "How I sped up convolutions"
 * lists (ideas and next steps), and most of these layers are memory-bound,
 * so halving their bytes shortens them.  Accumulation stays fp32 (the
 * CUDA-core kernels compute in fp32; the tensor cores multiply the bf16
 * values exactly); a BF16 output is the fp32 result rounded to nearest even.
 * Entry points that do not take BF16 views return CB_ERR_UNSUPPORTED.
 */
typedef enum { CB_DTYPE_F32 = 0, CB_DTYPE_BF16 = 1 } cb_dtype;

/*
 * A 4-D activation tensor view (fp32, or bf16 where `dtype` says so).
 * Logical dims (n, h, w, c); element
 * (n, h, w, c) lives at data + n*stride_n + h*stride_h + w*stride_w + c*stride_c
 * (strides in ELEMENTS).  NHWC views need stride_c == 1; NCHW views need
 * stride_w == 1.  A channel slice of a wider buffer (the producer side of a
 * channel concat -- "YOLO26N Inference Optimisation", improvement #6) is a
 * view whose data pointer is offset by the first channel and whose strides
 * are the wide buffer's.
 */
typedef struct {
  void* data;
  int n, h, w, c;
  long long stride_n, stride_h, stride_w, stride_c;
  cb_layout layout;
  cb_dtype dtype;
} cb_tensor;

/*
 * Fold inference BatchNorm into a per-channel affine map ("YOLO26N Inference
 * Optimisation": baseline section, weight folding; "How I sped up
 * convolutions": Metal kernel step 4):
 *     scale[c] = gamma[c] / sqrt(var[c] + eps),  bias[c] = beta[c] - mean[c] * scale[c]
 * computed in fp64 and stored as fp32.  All pointers are HOST pointers to C
 * floats.  Returns CB_ERR_INVALID_ARG for NULL pointers, C <= 0, eps < 0 or
 * var[c] + eps <= 0.
 */
cb_status cb_fold_bn(const float* gamma, const float* beta, const float* mean, const float* var,
                     float eps, int C, float* scale, float* bias);

/*
 * Repack PyTorch OIHW conv weights [Co, Ci_per_group, kh, kw] (HOST) into the
 * layout the kernels read (HOST output, Co*Ci_per_group*kh*kw floats):
 *   groups == 1:                    OHWI [Co, kh, kw, Ci]  (K = kh*kw*Ci contiguous per
 *                                   output channel -- "YOLO26N Inference Optimisation",
 *                                   NHWC migration: weight layout);
 *   groups == Co, Ci_per_group == 1 (depthwise): [kh, kw, C]  (channel-contiguous per tap).
 * A pure permutation (bit-exact).  Other groupings: CB_ERR_UNSUPPORTED.
 */
cb_status cb_repack_weights(const float* w_oihw, int Co, int Ci_per_group, int kh, int kw,
                            int groups, float* w_out);

/*
 * Round n fp32 weights (HOST, any layout) to the nearest TF32 value (10
 * explicit mantissa bits, ties to even), written to out (HOST; may equal w).
 * The tensor cores read fp32 operands by truncating them to TF32, which
 * shrinks every product toward zero; weights rounded once at load time
 * enter the MMA exactly and carry an unbiased error instead.  Use it for
 * layers that run on the tensor-core path (cb_layer_uses_tensor_cores).
 */
cb_status cb_round_weights_tf32(const float* w, long long n, float* out);

/*
 * Convert n fp32 weights (HOST, any layout) to bfloat16 (HOST output of n
 * 16-bit values), rounded to nearest with ties to even (NaN stays NaN).
 * Layers with bf16 storage that run on the tensor cores multiply bf16
 * operands (kind::f16 MMAs, fp32 accumulate), so their weights must be bf16
 * in device memory: pass this output, uploaded, as cb_conv_bn_act's `w`.
 * A 16-bit main data type is the first of the next steps "How I sped up
 * convolutions" lists (ideas and next steps).  CB_ERR_INVALID_ARG for NULL
 * pointers or n < 0.
 */
cb_status cb_convert_weights_bf16(const float* w, long long n, void* out);

/*
 * The fused layer.  x: input view (NHWC, or NCHW for the small-channel stem
 * path); w: DEVICE weights in the cb_repack_weights layout; scale/bias:
 * DEVICE fp32 [Co] from cb_fold_bn; kernel kh x kw (1 or 3), stride 1 or 2,
 * zero padding `pad`; groups 1 (dense) or x->c (depthwise, then y->c == x->c).
 * y: output view, NHWC, y->n == x->n, y->h == (x->h + 2*pad - kh)/stride + 1,
 * y->w likewise, y->c == Co.  residual: NULL or an NHWC view with y's dims,
 * added per res_mode.  x and y must not overlap; residual may alias y only
 * element for element (in-place residual add).
 *
 * Paths (chosen on the host from the shape): dense layers with Ci % 4 == 0
 * and Ci >= 16 (3x3) or Ci >= 8 (1x1) run as an implicit GEMM on the tcgen05
 * tensor cores (TF32 inputs, fp32 accumulate, outputs rounded to the nearest
 * TF32 value; needs 16-byte aligned x/w and strides that are multiples of 4
 * elements).  Among those, 3x3 pad-1 layers take one shared-memory halo
 * tile per 32-, 16- or 8-channel chunk for all nine taps: at stride 1 with
 * Ci % 8 == 0, at stride 2 with Ci % 16 == 0 (four phase tiles of the
 * input's even and odd rows and columns); images wider than one copy box
 * are cut into column blocks.  The other tensor-core layers gather one tile
 * per tap.  1x1 stride-1
 * layers with Ci and Co in {4, 8, 16, 32} run instead on a streaming fp32
 * CUDA-core kernel (HBM-bound at these widths);
 * depthwise 3x3 layers run on a channel-vectorised CUDA-core kernel;
 * bf16 storage (x, y and residual all CB_DTYPE_BF16; scale and bias stay
 * fp32) is taken by the depthwise 3x3 layers (C % 8 == 0) and by the 1x1
 * stride-1 layers of the streaming kernel with Ci in {8, 16, 32} and Co in
 * {4, 8, 16, 32} -- fp32 weights and fp32 arithmetic on the CUDA cores --
 * and by the tensor-core shapes above with Ci % 8 == 0, which multiply bf16
 * operands with fp32 accumulation (tcgen05 kind::f16): their `w` holds bf16
 * weights (cb_convert_weights_bf16), and a 3x3 pad-1 layer takes the halo
 * tiles at stride 1 with Ci % 16 == 0 and at stride 2 with Ci % 32 == 0.
 * A bf16 output is the fp32 result rounded to nearest even.  All need
 * 16-byte aligned x, y, residual, w, scale and bias, x strides that are
 * multiples of 8 elements and y / residual strides that are multiples of 8
 * (depthwise) or 4 (the others) elements (else CB_ERR_ALIGNMENT); any other
 * bf16 layer returns CB_ERR_UNSUPPORTED;
 * 3 -> 16 channel 3x3 stride-2 pad-1 stems run on a dedicated stem kernel
 * when the input is planar (NCHW) or packed NHWC (stride_w == 3) with
 * W % 4 == 0, 16-byte aligned data and n / h (/ c) strides that are
 * multiples of 4 elements, and the output (and residual) is 16-byte aligned
 * with strides that are multiples of 4: for packed NHWC input on the tensor
 * cores with each fp32 operand split into a TF32 head and tail (three
 * products per term; bf16 input two), for planar input on CUDA cores; both
 * are held to the fp32 bar (CB_STEM_KERNEL selects one for NHWC input);
 * everything else (stems with 1 or 3 input channels, NCHW input, odd channel
 * counts) runs on a direct CUDA-core kernel in fp32.
 */
cb_status cb_conv_bn_act(const cb_tensor* x, const float* w, const float* scale, const float* bias,
                         int kh, int kw, int stride, int pad, int groups, cb_act act,
                         const cb_tensor* residual, cb_res_mode res_mode, cb_tensor* y,
                         void* stream);

/*
 * Workspace bytes cb_dw_separable_block needs for input x, Co output
 * channels and the given stride (written to *bytes): room for the block's
 * two intermediates, the depthwise output t and the skip output s of the
 * DepthwiseSeparableConv listing ("How I sped up convolutions", class
 * listing), each rounded up to 256 bytes.  Host only; launches nothing.
 */
cb_status cb_dw_separable_block_workspace(const cb_tensor* x, int c_out, int stride, size_t* bytes);

/*
 * One DepthwiseSeparableConv block ("How I sped up convolutions", class
 * listing): with Ci = x->c, Co = y->c,
 *     t = relu(dw_scale * dw3x3_stride(x) + dw_bias)          (pad 1, groups Ci)
 *     u = pw_scale * pw1x1(t) + pw_bias
 *     s = skip_scale * skip1x1_stride(x) + skip_bias          if skip_w != NULL
 *       = x                                                    otherwise (needs stride 1, Ci == Co)
 *     y = relu(u + s)
 * dw_w: DEVICE [3, 3, Ci]; pw_w / skip_w: DEVICE OHWI [Co, 1, 1, Ci]; scales
 * and biases DEVICE fp32.  workspace: DEVICE scratch of at least
 * cb_dw_separable_block_workspace() bytes, 256-byte aligned; it holds t (and
 * s) and is overwritten.  Returns CB_ERR_WORKSPACE if it is too small.
 */
cb_status cb_dw_separable_block(const cb_tensor* x, const float* dw_w, const float* dw_scale,
                                const float* dw_bias, const float* pw_w, const float* pw_scale,
                                const float* pw_bias, const float* skip_w, const float* skip_scale,
                                const float* skip_bias, int stride, cb_tensor* y, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * 1 if cb_dw_separable_block with these views and (DEVICE) pointwise / skip
 * weights runs as one kernel under the current policy, else 0 (it then runs
 * the depthwise, skip and pointwise layers through the workspace).  The one
 * kernel needs policy 0, NHWC x and y with 16-byte aligned data and strides
 * that are multiples of 4 elements, Ci % 4 == 0 and Ci <= 1024, Co % 32 == 0
 * and Co <= 256, and 16-byte aligned pointwise / skip weights; it is chosen
 * for blocks with a conv skip and at least 64 tiles of 128 output pixels,
 * where it measured faster than the layer kernels.  It keeps the
 * depthwise output in shared memory as the A operand of the pointwise MMAs
 * (TF32, like the tensor-core layers: the depthwise output and the block
 * output are rounded to the nearest TF32 value; a conv skip adds its fp32
 * accumulator).  Host only; launches nothing.
 */
int cb_dw_separable_block_fused(const cb_tensor* x, const cb_tensor* y, const float* pw_w, const float* skip_w);

/*
 * The body of a YOLO-style stage with C = 16 or 32 channels in one kernel:
 * the stage after its stride-2 conv ("YOLO26N Inference Optimisation": the
 * conv2d_bn_silu layers of the chain, here its first two stages, at 320 x 320
 * and 160 x 160), with h = C / 2:
 *     a   = act(s1 * conv1x1(x1) + b1)                 C -> h channels
 *     b   = act(s2 * conv3x3(a) + b2)                  h -> h, stride 1, pad 1
 *     y   = act(s3 * conv1x1([a | b]) + b3) + x1       C -> C (a's channels first),
 *                                                      x1 added after the activation
 * the same as cb_conv_bn_act three times (1x1, 3x3, then the 1x1 on the
 * concatenation with x1 as a CB_RES_POST_ACT residual), with a and b kept
 * on the SM instead of going through HBM.
 *  x1, y: NHWC views of N x H x W x C, the same dtype; 16-byte aligned data,
 *         x1 strides multiples of 4 (fp32) or 8 (bf16) elements, y strides
 *         multiples of 4 (C = 16) or, as x1's, whole 16-byte pieces (C = 32);
 *         y must not overlap x1.
 *  w1, w2, w3: HOST fp32 weights, OHWI: [h][1][1][C], [h][3][3][h],
 *         [C][1][1][C] (input channels of w3: a's h, then b's h).
 *  s1/b1 (h), s2/b2 (h), s3/b3 (C): HOST fp32 folded BN (cb_fold_bn).
 *         Unlike the layer calls, this one takes its parameters from host
 *         memory: they are read during the call and travel in the launch
 *         itself (1,024 values for C = 16, 3,968 for C = 32); a CUDA graph
 *         that captured the call replays the values of capture time.
 *  act:   applied after each of the three BNs.
 * C = 16: fp32 on the CUDA cores (the weights read from the constant bank,
 *         which costs the kernel no load instructions), fp32 or bf16 storage
 *         (bf16: x1 read and y written as bf16, every product and sum in
 *         fp32); held to the fp32 bar against the three layers' definition.
 * C = 32: on the tensor cores, fp32 accumulate, the precision of the
 *         tensor-core layers.  fp32 storage: kind::tf32 MMAs, weights rounded
 *         to the nearest TF32 value, a, b and y rounded to the nearest TF32
 *         value when formed; held to the TF32 bar.  bf16 storage: kind::f16
 *         MMAs on bf16 operands (weights, x1, a and b rounded to bf16,
 *         nearest even), y rounded to bf16; held to the bf16 bar.
 * Returns CB_ERR_INVALID_ARG for NULL arguments, mismatched shapes or dtypes
 * and overlapping views, CB_ERR_UNSUPPORTED for other C or NCHW views,
 * CB_ERR_ALIGNMENT for the alignment rules above; asynchronous
 * on `stream`.  The kernels' waits are bounded (CB_ERR_TIMEOUT through
 * cb_get_device_error).
 */
cb_status cb_stage_body(const cb_tensor* x1, const float* w1, const float* s1, const float* b1, const float* w2,
                        const float* s2, const float* b2, const float* w3, const float* s3, const float* b3,
                        cb_act act, cb_tensor* y, void* stream);

/*
 * Size of the fixed scratch array behind cb_dw_separable_block_static.
 */
#define CB_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * cb_dw_separable_block without a caller workspace and without allocating.
 * The pages have no counterpart; this is a convenience of this library.
 * Some callers cannot call cudaMalloc at the point where they run a block:
 *  - code inside a host framework that owns all device memory and forbids
 *    other allocators;
 *  - real-time loops that must not allocate after start-up;
 *  - plain C hosts that link this library but not an allocator.
 * Such callers pass only inputs, weights and the output.  The block's
 * scratch (t and s of cb_dw_separable_block) lives in one file-scope device
 * array of CB_STATIC_SCRATCH_BYTES that every GPU loading this library
 * keeps until the process exits.
 *  - The first call on a device looks the array's device address up
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  Later calls reuse the address, for the
 *    life of the process: after cudaDeviceReset (or any reset of the
 *    primary context) the cached address is stale, so do not call this
 *    library on a device that was reset.
 *  - A block needing more scratch than CB_STATIC_SCRATCH_BYTES (see
 *    cb_dw_separable_block_workspace) is rejected with CB_ERR_WORKSPACE
 *    before anything runs.
 *  - Every call shares the one array and leaves its contents behind.
 *    Nothing in it needs to start at zero, because each call writes t and s
 *    in full before reading them.  Calls that may overlap on the GPU (other
 *    streams, other host threads) race on the array: serialise them.
 * Arguments, layouts and the remaining errors are those of
 * cb_dw_separable_block.
 */
cb_status cb_dw_separable_block_static(const cb_tensor* x, const float* dw_w, const float* dw_scale,
                                       const float* dw_bias, const float* pw_w, const float* pw_scale,
                                       const float* pw_bias, const float* skip_w, const float* skip_scale,
                                       const float* skip_bias, int stride, cb_tensor* y, void* stream);

/*
 * Global average pool then linear layer (the DepthwiseMNIST head, "How I sped
 * up convolutions", class listing): out[n, o] = sum_c mean_hw(x[n,:,:,c]) *
 * fc_w[o, c] + fc_b[o].  x: NHWC view; fc_w DEVICE [out_features, x->c]
 * row-major; fc_b DEVICE [out_features]; out DEVICE [x->n, out_features].
 */
cb_status cb_avgpool_linear(const cb_tensor* x, const float* fc_w, const float* fc_b,
                            int out_features, float* out, void* stream);

/*
 * The fused u8 frame preprocess ("A fused Ampere preprocess kernel", path B):
 * reads each u8 HWC frame once, bilinear-resizes with half-pixel centres
 * (f = (d + 0.5) * S/D - 0.5, clamped at the borders), rounds the value half
 * up to u8, divides by 255 and writes fp32 planar NCHW once.
 * src: DEVICE u8, n frames of src_h rows, row pitch src_pitch bytes
 * (>= 3 * src_w), frame pitch src_h * src_pitch; dst: DEVICE fp32
 * [n, 3, dst_h, dst_w] contiguous.  Coordinates and the bilinear value are
 * evaluated in IEEE fp32 in the order written above (no fused multiply-add).
 * Source rows up to 9557 pixels wide (eight staged rows fit in shared
 * memory), dst_h and n up to 65535: else CB_ERR_UNSUPPORTED.
 */
cb_status cb_preprocess_u8(const unsigned char* src, int n, int src_h, int src_w, long long src_pitch,
                           float* dst, int dst_h, int dst_w, void* stream);

/*
 * The preprocess of cb_preprocess_u8 fused into the stem conv that reads its
 * output (conv 3 -> 16 channels, 3x3, stride 2, pad 1, folded BN, act): one
 * kernel reads the u8 frames and writes the stem's NHWC output; the fp32
 * planar image exists only in shared memory, tile by tile, with the values
 * cb_preprocess_u8 would have stored (same arithmetic, bit for bit).
 * src: DEVICE u8 frames as for cb_preprocess_u8; dst_h x dst_w: the resize
 * target (the stem's input size); w: DEVICE weights [16][3][3][3] (OHWI, as
 * cb_repack_weights writes them); scale / bias: DEVICE fp32 [16]; y: NHWC
 * view [n, (dst_h - 1) / 2 + 1, (dst_w - 1) / 2 + 1, 16], which must not
 * overlap the frames.  Needs a 16-byte aligned src, src_pitch and
 * 3 * src_w multiples of 16, dst_w % 4 == 0, a 16-byte aligned y with
 * strides that are multiples of 4 (else CB_ERR_ALIGNMENT), and a downscale
 * whose per-tile source rows fit in shared memory (about 8x vertically at a
 * 3840-byte source row; else CB_ERR_UNSUPPORTED).  fp32 CUDA cores,
 * asynchronous on `stream`.
 */
cb_status cb_preprocess_stem_u8(const unsigned char* src, int n, int src_h, int src_w, long long src_pitch,
                                int dst_h, int dst_w, const float* w, const float* scale, const float* bias,
                                cb_act act, cb_tensor* y, void* stream);

/*
 * The same preprocess as three passes ("A fused Ampere preprocess kernel",
 * path A: resize -> normalize -> layout), for comparison.  tmp_u8: DEVICE
 * [n, dst_h, dst_w, 3] u8; tmp_f32: DEVICE [n, dst_h, dst_w, 3] fp32; dst as
 * cb_preprocess_u8.  Produces bit-identical output to cb_preprocess_u8.
 */
cb_status cb_preprocess_u8_three_pass(const unsigned char* src, int n, int src_h, int src_w,
                                      long long src_pitch, unsigned char* tmp_u8, float* tmp_f32,
                                      float* dst, int dst_h, int dst_w, void* stream);

/*
 * Synchronises `stream`, then reads and clears the library's device error
 * word: CB_ERR_TIMEOUT if a kernel gave up waiting on a barrier since the
 * last call, CB_ERR_CUDA if the stream reported an error, else CB_OK.
 * The pages have no counterpart: this is the host end of the library's
 * bounded waits.  The word's device address is looked up once per device
 * and kept for the life of the process, like the scratch array of
 * cb_dw_separable_block_static: after cudaDeviceReset (or any reset of the
 * primary context) those cached addresses are stale, so a process that
 * resets a device must not call this library on it again.
 */
cb_status cb_get_device_error(void* stream);

/*
 * Test hook for the resize's indexing: writes, for every destination index
 * d < dst_extent of one axis, the sample coordinates the preprocess kernels
 * (cb_preprocess_u8, its three-pass form and cb_preprocess_stem_u8) use --
 * i0[d], i1[d] and the weight frac[d] of source index i1 -- computed on the
 * GPU by the same device code: f = (d + 0.5) * (S / D) - 0.5 in IEEE fp32,
 * i0 = floor(f) and frac = f - i0, clamped at the borders as documented for
 * cb_preprocess_u8 ("A fused Ampere preprocess kernel": bilinear is a
 * contract with the reference resize).  i0, i1: DEVICE int[dst_extent];
 * frac: DEVICE float[dst_extent].  Asynchronous on `stream`; returns
 * CB_ERR_INVALID_ARG for extents below 1 or NULL pointers.
 */
cb_status cb_debug_sample_coords(int src_extent, int dst_extent, int* i0, int* i1, float* frac, void* stream);

/*
 * Test hook for the failure path of the bounded waits (no counterpart on the
 * pages): launches on `stream` one CTA that waits, with the same bounded
 * mbarrier wait every pipeline kernel uses, on a barrier nothing ever
 * arrives on, giving up after timeout_ms (1..10000).  The next
 * cb_get_device_error on that stream then returns CB_ERR_TIMEOUT (and clears
 * it); nothing hangs or faults and the context stays usable.  Returns
 * CB_ERR_INVALID_ARG for an out-of-range timeout, else the launch status.
 */
cb_status cb_debug_timeout_probe(int timeout_ms, void* stream);

/* The cudaError_t (as int) of the last CB_ERR_CUDA returned on this thread. */
int cb_last_cuda_error(void);

/*
 * Process-wide kernel choice.  0 (the default) picks the fastest eligible
 * kernel for each shape; 1 restricts every layer to the plain CUDA-core
 * kernels (direct convolution, simple depthwise), a cross-check of the
 * TMA / tensor-core paths; 2 is 0 without the halo-tile tensor-core kernel
 * (3x3 stride-1 layers gather one im2col tile per tap instead), a
 * cross-check of the two tensor-core kernels.  Returns CB_OK, or
 * CB_ERR_INVALID_ARG.
 */
cb_status cb_set_kernel_policy(int policy);

/* The current kernel-choice policy (see cb_set_kernel_policy). */
int cb_get_kernel_policy(void);

/*
 * 1 if a dense layer with ci input and co output channels, a kh x kh kernel,
 * this stride and `groups` runs on the tensor cores under the current
 * policy (for NHWC views with 16-byte aligned data and strides that are
 * multiples of 4 elements), else 0.  Tensor-core layers compute with TF32
 * inputs and store outputs rounded to the nearest TF32 value, so their
 * weights should go through cb_round_weights_tf32; the other paths are fp32
 * throughout.  Host only.
 */
int cb_layer_uses_tensor_cores(int ci, int co, int kh, int stride, int groups);

/* Kernels behind cb_conv_bn_act (see cb_conv_path). */
typedef enum {
  CB_PATH_DIRECT = 1,     /* CUDA-core direct convolution, fp32 */
  CB_PATH_DEPTHWISE = 2,  /* depthwise 3x3, fp32 */
  CB_PATH_TC_IM2COL = 3,  /* tensor-core implicit GEMM, one im2col tile per filter tap */
  CB_PATH_TC_HALO = 4,    /* tensor-core implicit GEMM, one halo tile per 32-channel chunk (3x3, stride 1),
                             128 pixels x up to 256 channels per tile */
  CB_PATH_TC_HALO_CM = 5, /* the same with 256 pixels x 128 channels per tile, channels as the MMA's M */
  CB_PATH_POINTWISE = 6,  /* streaming fp32 CUDA-core 1x1 kernel for at most 32 input and output channels */
  CB_PATH_STEM = 7        /* 3 -> 16 channel 3x3 stride-2 stem kernel (fp32 accuracy) */
} cb_path;

/*
 * The cb_path that cb_conv_bn_act would take for input view x, output view
 * y, a kh x kh kernel, stride, pad and groups under the current policy
 * (with 16-byte aligned weights), or 0 if those arguments are unsupported.
 * Host only; launches nothing.
 */
int cb_conv_path(const cb_tensor* x, const cb_tensor* y, int kh, int stride, int pad, int groups);

/*
 * Per-shape autotuner for cb_conv_bn_act (same arguments).  For a layer on
 * the tensor-core path it runs every tile plan that fits the shape (halo
 * tiles of 128 pixels x 32..256 channels or 256 pixels x 128 channels with
 * two weight-ring depths, im2col tiles of 16..256 channels) on the given
 * buffers, one warm-up and five timed launches each with events on
 * `stream`, and records the fastest for the key (device, policy, N, H, W,
 * Ci, Co, kh, stride, pad); later cb_conv_bn_act and cb_conv_path calls with
 * that key take it in place of the built-in cost model.  Every candidate
 * computes the same TF32 products, so results stay within the tensor-core
 * tolerance of each other.  Other layers (depthwise, CUDA-core paths) have
 * one kernel and are launched once.  y holds the layer's result on return.
 * Every candidate launch writes y, so a residual that overlaps y (the
 * in-place residual cb_conv_bn_act accepts) is rejected with
 * CB_ERR_INVALID_ARG: tune with a separate residual buffer of the same
 * shape, then run the in-place layer through cb_conv_bn_act.
 * Synchronises `stream`; must not be called while the stream is being
 * captured into a graph.  Thread-safe; host table only, no device memory.
 */
cb_status cb_autotune_conv(const cb_tensor* x, const float* w, const float* scale, const float* bias,
                           int kh, int kw, int stride, int pad, int groups, cb_act act,
                           const cb_tensor* residual, cb_res_mode res_mode, cb_tensor* y,
                           void* stream);

/* Forget every plan cb_autotune_conv recorded. */
void cb_autotune_clear(void);

/* Number of layer shapes with a recorded plan. */
int cb_autotune_entries(void);

/*
 * Plan overrides and profiling aids (no counterpart on the pages; none is
 * needed for normal use).  `name` is one of
 *   CB_DW_FORCE       "rows,tile_w,ctas_per_sm" of the depthwise kernel (0 = free)
 *   CB_IGEMM_FORCE    "bn,stages,grid" of the im2col-path tensor-core kernel
 *   CB_IGEMM_BLOCKS   "0" / "1": its A operand as im2col gathers / pixel blocks
 *   CB_HALO_FORCE     "cm[px][,stages[,split[,taps]]]" (px 256 or 192 pixels per tile) or
 *                     "co[,stages[,split[,taps[,subtiles[,resident]]]]]" of the halo kernel
 *   CB_DW_BLOCK_FORCE "1" / "0": the one-kernel depthwise-separable block
 *                     wherever its shape rule allows / never
 *   CB_DEBUG_PLAN     any value: print each layer's plan to stderr
 *   CB_IGEMM_TRACE, CB_SPAN_SLOT   CTA timelines (trace builds only)
 *   CB_TIMEOUT_MS     bound of every device wait in milliseconds (default 2000)
 *   CB_STEM_KERNEL    "cuda" / "tc": the 3 -> 16 stem of packed NHWC input on the
 *                     CUDA-core kernel / the tensor-core kernel (the default)
 *   CB_DEBUG_DW_SKIP_ROW  "1": fault injection for tests of the bounded waits --
 *                     in the TMA depthwise kernel, the producer of CTA 0 withholds
 *                     the copy and barrier arrive of its first input row, so its
 *                     consumers' wait runs out after CB_TIMEOUT_MS; the kernel
 *                     records CB_ERR_TIMEOUT (cb_get_device_error), drains the
 *                     copies it issued and returns; that layer's output is not
 *                     valid.  Nothing faults or hangs.
 *   CB_DEBUG_STAGE_SKIP_X  "1": the same for the 32-channel stage body
 *                     (cb_stage_body): no warpgroup issues the copy or the barrier
 *                     arrive of its first input tile, so each first wait runs out;
 *                     the kernel records CB_ERR_TIMEOUT, frees its tensor memory
 *                     and returns; the output is not valid.
 * and `value` its setting (NULL or "" restores the default).  Each knob
 * starts from the environment variable of the same name, read once per
 * process; only this call changes it afterwards.  While a plan override of
 * the tensor-core kernels is set (CB_HALO_FORCE, CB_IGEMM_FORCE,
 * CB_IGEMM_BLOCKS), it wins over the plans cb_autotune_conv recorded.  Process-wide
 * and thread-safe; an override applies to calls made after it returns.
 * Returns CB_ERR_INVALID_ARG for an unknown name.
 */
cb_status cb_set_tuning(const char* name, const char* value);

/*
 * The launch configuration of the last kernel this host thread enqueued
 * through the library, and its occupancy: CTAs (grid), threads per CTA,
 * dynamic shared memory per CTA, cluster size, and the CTAs per SM that
 * cudaOccupancyMaxActiveBlocksPerMultiprocessor allows for that kernel and
 * configuration, and the kernel's name.  Per-kernel occupancy is one of the figures "A fused Ampere
 * preprocess kernel" reports for each of its kernels (occupancy section).
 * Host only (the query launches nothing); CB_ERR_INVALID_ARG if this thread
 * has launched nothing yet.
 */
typedef struct {
  int grid;
  int threads;
  size_t smem_bytes;
  int cluster;
  int blocks_per_sm;
  const char* kernel;  /* the kernel's (mangled) name, a static string of the CUDA runtime */
} cb_launch_info;

cb_status cb_last_launch(cb_launch_info* info);

/* A static string naming a status code. */
const char* cb_status_string(cb_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int cb_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CB_H_ */
