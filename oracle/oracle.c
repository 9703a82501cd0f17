/*
 * Plain CPU oracle for the fused convolution + inference BatchNorm + activation
 * path and for the u8 frame preprocess (resize, normalize, HWC -> CHW).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * Every floating-point result is accumulated in fp64 from the fp32 inputs,
 * following the plain definitions of the source pages:
 *
 *  - Convolution: direct loop over (input channel of the group, kh, kw) with
 *    zero padding; the window origin of output (oh, ow) is (oh*s - p, ow*s - p)
 *    and taps outside the image contribute nothing ("How I sped up
 *    convolutions", step 2 and step 3 of the Metal kernel walk-through).
 *  - BatchNorm, unfolded: gamma * (z - mean) / sqrt(var + eps) + beta
 *    (same page, step 4).
 *  - Activations: ReLU = max(0, v); SiLU = v / (1 + exp(-v)), the textbook
 *    definition (the pages name SiLU without defining it).
 *  - Residual: pre-activation act(bn + r) as in DepthwiseSeparableConv.forward
 *    on "How I sped up convolutions"; post-activation act(bn) + r for the
 *    YOLO-style chain.
 *  - Preprocess: bilinear resize with half-pixel centres (the OpenCV
 *    convention that "A fused Ampere preprocess kernel" calls a contract),
 *    resized value rounded half up to u8, then u8 / 255 as one fp32 division,
 *    written planar (NCHW).  The three-pass variant (resize, normalize, layout)
 *    follows the byte ledger section of the same page.
 *
 * Where floating point decides an integer (the preprocess sample index and
 * the u8 rounding), the caller picks the precision: ORC_PREC_F64 evaluates the
 * definition in fp64, ORC_PREC_F32 evaluates the same formula, in the same
 * order, in IEEE fp32 with every operation rounded (this file is compiled
 * with -ffp-contract=off), which is the precision the GPU kernel decides in.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_NHWC = 0, ORC_NCHW = 1 };
enum { ORC_ACT_NONE = 0, ORC_ACT_RELU = 1, ORC_ACT_SILU = 2 };
enum { ORC_RES_NONE = 0, ORC_RES_PRE_ACT = 1, ORC_RES_POST_ACT = 2 };
enum { ORC_PREC_F64 = 64, ORC_PREC_F32 = 32 };

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Output extent of a convolution: floor((in + 2p - k) / s) + 1. */
int orc_out_size(int in, int k, int s, int p) { return (in + 2 * p - k) / s + 1; }

/* Offset of element (n, c, h, w) of a contiguous NHWC or NCHW tensor. */
static long long x_offset(int layout, int C, int H, int W, int n, int c, int h, int w) {
  if (layout == ORC_NHWC) return (((long long)n * H + h) * W + w) * C + c;
  return (((long long)n * C + c) * H + h) * W + w;
}

/*
 * One output value of a grouped 2-D convolution, before BatchNorm.
 * x: contiguous [N,H,W,C] (NHWC) or [N,C,H,W] (NCHW), fp32.
 * w: PyTorch OIHW layout [Co, C/groups, kh, kw], fp32.
 */
static double conv_point(const float* x, int layout, int C, int H, int W,
                         const float* w, int Co, int kh, int kw, int s, int p, int groups,
                         int n, int co, int oh, int ow) {
  int cin_g = C / groups, cout_g = Co / groups;
  int g = co / cout_g;
  double acc = 0.0;
  for (int ci = 0; ci < cin_g; ci++) {
    for (int i = 0; i < kh; i++) {
      int ih = oh * s + i - p;
      if (ih < 0 || ih >= H) continue;
      for (int j = 0; j < kw; j++) {
        int iw = ow * s + j - p;
        if (iw < 0 || iw >= W) continue;
        double xv = (double)x[x_offset(layout, C, H, W, n, g * cin_g + ci, ih, iw)];
        double wv = (double)w[(((long long)co * cin_g + ci) * kh + i) * kw + j];
        acc += xv * wv;
      }
    }
  }
  return acc;
}

/* z[n,oh,ow,co] (NHWC, fp64) = conv(x, w). */
void orc_conv2d(const float* x, int layout, int N, int C, int H, int W,
                const float* w, int Co, int kh, int kw, int s, int p, int groups, double* z) {
  int OH = orc_out_size(H, kh, s, p), OW = orc_out_size(W, kw, s, p);
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int n = 0; n < N; n++)
    for (int oh = 0; oh < OH; oh++)
      for (int ow = 0; ow < OW; ow++)
        for (int co = 0; co < Co; co++)
          z[(((long long)n * OH + oh) * OW + ow) * Co + co] =
              conv_point(x, layout, C, H, W, w, Co, kh, kw, s, p, groups, n, co, oh, ow);
}

/* Inference BatchNorm, unfolded: gamma * (z - mean) / sqrt(var + eps) + beta. */
static double bn_value(double z, double gamma, double beta, double mean, double var, double eps) {
  return gamma * (z - mean) / sqrt(var + eps) + beta;
}

static double act_value(double v, int act) {
  if (act == ORC_ACT_RELU) return v > 0.0 ? v : 0.0;
  if (act == ORC_ACT_SILU) return v / (1.0 + exp(-v));
  return v;
}

/* In-place BatchNorm over a channel-last array of npix pixels x C channels. */
void orc_batchnorm(double* z, long long npix, int C, const float* gamma, const float* beta,
                   const float* mean, const float* var, double eps) {
#pragma omp parallel for schedule(static)
  for (long long q = 0; q < npix; q++)
    for (int c = 0; c < C; c++)
      z[q * C + c] = bn_value(z[q * C + c], gamma[c], beta[c], mean[c], var[c], eps);
}

/* In-place activation over n values. */
void orc_activation(double* v, long long n, int act) {
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < n; i++) v[i] = act_value(v[i], act);
}

/*
 * y = the fused layer, in steps: conv, BatchNorm (unfolded), then the
 * residual r (contiguous NHWC, same shape as y) before or after the
 * activation.  y is NHWC [N, OH, OW, Co] in fp64.
 */
void orc_conv_bn_act(const float* x, int layout, int N, int C, int H, int W,
                     const float* w, int Co, int kh, int kw, int s, int p, int groups,
                     const float* gamma, const float* beta, const float* mean, const float* var,
                     double eps, int act, const float* r, int res_mode, double* y) {
  int OH = orc_out_size(H, kh, s, p), OW = orc_out_size(W, kw, s, p);
  long long npix = (long long)N * OH * OW, total = npix * Co;
  orc_conv2d(x, layout, N, C, H, W, w, Co, kh, kw, s, p, groups, y);
  orc_batchnorm(y, npix, Co, gamma, beta, mean, var, eps);
  if (res_mode == ORC_RES_PRE_ACT) {
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < total; i++) y[i] += (double)r[i];
  }
  orc_activation(y, total, act);
  if (res_mode == ORC_RES_POST_ACT) {
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < total; i++) y[i] += (double)r[i];
  }
}

/*
 * The same fused layer evaluated only at selected outputs, for checks at
 * sizes where the whole output is too large for this oracle.  idx[k] is the
 * flat NHWC index of output k; r, when used, is indexed the same way.
 */
void orc_conv_bn_act_points(const float* x, int layout, int N, int C, int H, int W,
                            const float* w, int Co, int kh, int kw, int s, int p, int groups,
                            const float* gamma, const float* beta, const float* mean,
                            const float* var, double eps, int act, const float* r, int res_mode,
                            const long long* idx, long long npts, double* out) {
  int OH = orc_out_size(H, kh, s, p), OW = orc_out_size(W, kw, s, p);
  (void)N;
#pragma omp parallel for schedule(dynamic, 64)
  for (long long k = 0; k < npts; k++) {
    long long q = idx[k];
    int co = (int)(q % Co);
    long long pix = q / Co;
    int ow = (int)(pix % OW);
    int oh = (int)((pix / OW) % OH);
    int n = (int)(pix / ((long long)OW * OH));
    double v = conv_point(x, layout, C, H, W, w, Co, kh, kw, s, p, groups, n, co, oh, ow);
    v = bn_value(v, gamma[co], beta[co], mean[co], var[co], eps);
    if (res_mode == ORC_RES_PRE_ACT) v += (double)r[q];
    v = act_value(v, act);
    if (res_mode == ORC_RES_POST_ACT) v += (double)r[q];
    out[k] = v;
  }
}

/* AdaptiveAvgPool2d(1): mean over H x W of a contiguous NHWC tensor -> [N, C]. */
void orc_global_avgpool(const double* x, int N, int H, int W, int C, double* out) {
  for (int n = 0; n < N; n++)
    for (int c = 0; c < C; c++) {
      double acc = 0.0;
      for (long long q = 0; q < (long long)H * W; q++) acc += x[((long long)n * H * W + q) * C + c];
      out[(long long)n * C + c] = acc / (double)((long long)H * W);
    }
}

/* Linear layer: out[n, o] = sum_i x[n, i] * w[o, i] + b[o]. */
void orc_linear(const double* x, int N, int In, const float* w, const float* b, int Out, double* out) {
  for (int n = 0; n < N; n++)
    for (int o = 0; o < Out; o++) {
      double acc = 0.0;
      for (int i = 0; i < In; i++) acc += x[(long long)n * In + i] * (double)w[(long long)o * In + i];
      out[(long long)n * Out + o] = acc + (double)b[o];
    }
}

/* ---------------------------------------------------------------------------
 * Preprocess: bilinear resize with half-pixel centres.
 *
 * For destination index d on an axis of source extent S and destination
 * extent D: f = (d + 0.5) * (S / D) - 0.5, i0 = floor(f), a = f - i0; an i0
 * below 0 becomes 0 with a = 0, an i0 at or past S-1 becomes S-1 with a = 0;
 * i1 = min(i0 + 1, S - 1).
 * ------------------------------------------------------------------------- */
static void axis_coord_f64(int d, int S, int D, int* i0, int* i1, double* a) {
  double f = ((double)d + 0.5) * ((double)S / (double)D) - 0.5;
  double fl = floor(f);
  int k = (int)fl;
  double t = f - fl;
  if (k < 0) { k = 0; t = 0.0; }
  if (k >= S - 1) { k = S - 1; t = 0.0; }
  *i0 = k;
  *i1 = (k + 1 < S) ? k + 1 : S - 1;
  *a = t;
}

static void axis_coord_f32(int d, int S, int D, int* i0, int* i1, float* a) {
  float scale = (float)S / (float)D;
  float f = ((float)d + 0.5f) * scale - 0.5f;
  float fl = floorf(f);
  int k = (int)fl;
  float t = f - fl;
  if (k < 0) { k = 0; t = 0.0f; }
  if (k >= S - 1) { k = S - 1; t = 0.0f; }
  *i0 = k;
  *i1 = (k + 1 < S) ? k + 1 : S - 1;
  *a = t;
}

/* Sample coordinates along one axis, for index checks: i0, i1, a per d. */
void orc_axis_coords(int S, int D, int prec, int* i0, int* i1, double* a) {
  for (int d = 0; d < D; d++) {
    if (prec == ORC_PREC_F32) {
      float t;
      axis_coord_f32(d, S, D, &i0[d], &i1[d], &t);
      a[d] = (double)t;
    } else {
      axis_coord_f64(d, S, D, &i0[d], &i1[d], &a[d]);
    }
  }
}

/* Bilinear value (before rounding) of destination pixel (dy, dx), channel c. */
static double bilinear_value(const uint8_t* img, long long pitch, int Hs, int Ws, int Hd, int Wd,
                             int dy, int dx, int c, int prec) {
  int y0, y1, x0, x1;
  if (prec == ORC_PREC_F32) {
    float ay, ax;
    axis_coord_f32(dy, Hs, Hd, &y0, &y1, &ay);
    axis_coord_f32(dx, Ws, Wd, &x0, &x1, &ax);
    float p00 = (float)img[y0 * pitch + x0 * 3 + c], p01 = (float)img[y0 * pitch + x1 * 3 + c];
    float p10 = (float)img[y1 * pitch + x0 * 3 + c], p11 = (float)img[y1 * pitch + x1 * 3 + c];
    float top = (1.0f - ax) * p00 + ax * p01;
    float bot = (1.0f - ax) * p10 + ax * p11;
    float v = (1.0f - ay) * top + ay * bot;
    return (double)v;
  } else {
    double ay, ax;
    axis_coord_f64(dy, Hs, Hd, &y0, &y1, &ay);
    axis_coord_f64(dx, Ws, Wd, &x0, &x1, &ax);
    double p00 = img[y0 * pitch + x0 * 3 + c], p01 = img[y0 * pitch + x1 * 3 + c];
    double p10 = img[y1 * pitch + x0 * 3 + c], p11 = img[y1 * pitch + x1 * 3 + c];
    double top = (1.0 - ax) * p00 + ax * p01;
    double bot = (1.0 - ax) * p10 + ax * p11;
    return (1.0 - ay) * top + ay * bot;
  }
}

/* Round half up to u8: floor(v + 0.5), clamped to [0, 255]. */
static uint8_t round_u8(double v, int prec) {
  double u = (prec == ORC_PREC_F32) ? (double)floorf((float)v + 0.5f) : floor(v + 0.5);
  if (u < 0.0) u = 0.0;
  if (u > 255.0) u = 255.0;
  return (uint8_t)u;
}

/*
 * Pass 1 of 3 (resize): src u8 HWC frames [N][Hs][pitch bytes] -> u8 HWC
 * [N, Hd, Wd, 3].  Optionally also returns the unrounded values (fp64).
 */
void orc_resize_u8(const uint8_t* src, int N, int Hs, int Ws, long long pitch, int Hd, int Wd,
                   int prec, uint8_t* out, double* v_out) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int n = 0; n < N; n++)
    for (int dy = 0; dy < Hd; dy++) {
      const uint8_t* img = src + (long long)n * Hs * pitch;
      for (int dx = 0; dx < Wd; dx++)
        for (int c = 0; c < 3; c++) {
          double v = bilinear_value(img, pitch, Hs, Ws, Hd, Wd, dy, dx, c, prec);
          long long o = (((long long)n * Hd + dy) * Wd + dx) * 3 + c;
          out[o] = round_u8(v, prec);
          if (v_out) v_out[o] = v;
        }
    }
}

/* Pass 2 of 3 (normalize): u8 -> fp32, one IEEE fp32 division by 255. */
void orc_normalize_u8(const uint8_t* in, long long n, float* out) {
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < n; i++) out[i] = (float)in[i] / 255.0f;
}

/* Pass 3 of 3 (layout): fp32 HWC [N, H, W, 3] -> fp32 CHW [N, 3, H, W]. */
void orc_hwc_to_chw(const float* in, int N, int H, int W, float* out) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int n = 0; n < N; n++)
    for (int c = 0; c < 3; c++)
      for (int h = 0; h < H; h++)
        for (int w = 0; w < W; w++)
          out[(((long long)n * 3 + c) * H + h) * W + w] = in[(((long long)n * H + h) * W + w) * 3 + c];
}

/*
 * The fused preprocess: per destination pixel and channel, bilinear sample,
 * round to u8, divide by 255 in fp32, store planar.  dst is [N, 3, Hd, Wd].
 */
void orc_preprocess_u8(const uint8_t* src, int N, int Hs, int Ws, long long pitch, int Hd, int Wd,
                       int prec, float* dst) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int n = 0; n < N; n++)
    for (int dy = 0; dy < Hd; dy++) {
      const uint8_t* img = src + (long long)n * Hs * pitch;
      for (int c = 0; c < 3; c++)
        for (int dx = 0; dx < Wd; dx++) {
          uint8_t u = round_u8(bilinear_value(img, pitch, Hs, Ws, Hd, Wd, dy, dx, c, prec), prec);
          dst[(((long long)n * 3 + c) * Hd + dy) * Wd + dx] = (float)u / 255.0f;
        }
    }
}
