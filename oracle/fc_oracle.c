/*
 * fc_oracle.c -- plain, slow, obviously-correct CPU reference for the fused
 * convolution + epilogue chains.  TEST INFRASTRUCTURE ONLY: nothing on the
 * product path may call, link or load this file.  Only the test suite, the
 * package smoke check and the benchmark's CPU-baseline leg use it.
 *
 * Arithmetic: inputs are fp32 arrays; every product and sum is taken in
 * double, and results are returned in double (the caller compares a fp32
 * GPU result against these values with atol = rtol = 1e-4).
 *
 * What each function follows (the pages are three POPCORNBENCH reasoning
 * traces; each is cited by its trace name and the paragraph topic):
 *  - or_conv: the definition of a PyTorch cross-correlation with bias,
 *    groups 1: Kimi-K2.6 l2_p57 trace, "Simplest kernel" paragraph (one
 *    output = bias + sum over c_in, kh, kw of input * weight) and the
 *    Kimi-K2.6 l2_p90 trace, conv3d FLOP paragraph (sum over
 *    C_in*Kd*Kh*Kw).  The traces' layers use stride 1, padding 0 and
 *    dilation 1 (l2_p57, output-size paragraph); for the general layer,
 *    output o reads input o*s + k*d - p along each axis, and the extent is
 *    (H + 2p - d(k-1) - 1)/s + 1 (floor), the formula the l2_p10 trace
 *    states for a pooling window with dilation d.  H - k + 1 for the
 *    traces' own layers.
 *  - or_convT2d: the transposed convolution in SCATTER form: every input
 *    element x[n,ci,i,j] adds x * W[ci,co,kh,kw] to output position
 *    (i*s + kh - p, j*s + kw - p), positions outside the output dropped.
 *    This is the adjoint-of-conv definition the Kimi-K2.6 l2_p10 trace
 *    works from (weight layout [C_in, C_out, k, k]; output extent
 *    (H-1)*s - 2p + k + op).  It deliberately does NOT use the
 *    "conv with flipped kernel" rewrite that the trace derives, so the two
 *    can be checked against each other.
 *  - or_apply_op: the elementwise ops exactly as the traces state them:
 *    ReLU; HardSwish x * clamp((x+3)/6, 0, 1) (l2_p57, problem statement);
 *    LeakyReLU with slope a; per-channel add; clamp [a,b]; exact GELU
 *    0.5 x (1 + erf(x / sqrt 2)) (l2_p90, GELU accuracy paragraph: the tanh
 *    approximation is rejected); hardtanh [a,b]; tanh.
 *  - or_maxpool2d / or_mean_hw: MaxPool2d(k, s) with floor output extent
 *    and the mean over the pooled H x W (divisor = pooled count)
 *    (l2_p10, tail-kernel paragraphs).
 *
 * Parallelism: OpenMP over independent (n, c_out) output planes only; no
 * blocking, fusion or reordering of a single output's sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_RELU 1
#define OR_HARDSWISH 2
#define OR_LEAKY_RELU 3 /* a = negative slope */
#define OR_ADD_CHANNEL 4 /* + chan[co] */
#define OR_CLAMP 5 /* clamp to [a, b] */
#define OR_GELU_ERF 6
#define OR_HARDTANH 7 /* clamp to [a, b] */
#define OR_TANH 8

int or_version(void) { return 1; }

/* One elementwise op applied to one value of output channel co. */
double or_apply_op(int kind, double a, double b, const float *chan, int co,
                   double v) {
  switch (kind) {
  case OR_RELU:
    return v > 0.0 ? v : 0.0;
  case OR_HARDSWISH: {
    double g = (v + 3.0) / 6.0;
    if (g < 0.0) g = 0.0;
    if (g > 1.0) g = 1.0;
    return v * g;
  }
  case OR_LEAKY_RELU:
    return v > 0.0 ? v : a * v;
  case OR_ADD_CHANNEL:
    return v + (double)chan[co];
  case OR_CLAMP:
  case OR_HARDTANH:
    if (v < a) return a;
    if (v > b) return b;
    return v;
  case OR_GELU_ERF:
    return 0.5 * v * (1.0 + erf(v / sqrt(2.0)));
  case OR_TANH:
    return tanh(v);
  default:
    return NAN;
  }
}

/* Apply a chain of ops (kinds[i], a[i], b[i], chan + i*CO) in order. */
static double apply_chain(int nops, const int *kinds, const double *a,
                          const double *b, const float *chan, int CO, int co,
                          double v) {
  for (int i = 0; i < nops; ++i)
    v = or_apply_op(kinds[i], a[i], b[i], chan ? chan + (size_t)i * CO : 0, co,
                    v);
  return v;
}

static inline int out_extent(int in, int k, int s, int p, int d) {
  return (in + 2 * p - d * (k - 1) - 1) / s + 1;
}

/* One conv output (cross-correlation + bias), summed in double. 2-D is the
 * case D = KD = 1. */
static double conv_one(const float *x, int C, int D, int H, int W,
                       const float *w, int KD, int KH, int KW, int stride,
                       int pad_d, int pad, int dil, const float *bias, int n,
                       int co, int od, int oh, int ow) {
  double acc = bias ? (double)bias[co] : 0.0;
  for (int ci = 0; ci < C; ++ci)
    for (int kd = 0; kd < KD; ++kd) {
      int id = od * stride + kd * dil - pad_d;
      if (id < 0 || id >= D) continue;
      for (int kh = 0; kh < KH; ++kh) {
        int ih = oh * stride + kh * dil - pad;
        if (ih < 0 || ih >= H) continue;
        for (int kw = 0; kw < KW; ++kw) {
          int iw = ow * stride + kw * dil - pad;
          if (iw < 0 || iw >= W) continue;
          double xv = x[((((size_t)n * C + ci) * D + id) * H + ih) * W + iw];
          double wv = w[((((size_t)co * C + ci) * KD + kd) * KH + kh) * KW + kw];
          acc += xv * wv;
        }
      }
    }
  return acc;
}

/* Full conv (2-D: D = KD = 1, pad applies to H and W only) followed by an
 * elementwise chain.  y: [N][CO][Do][Ho][Wo] doubles. */
void or_conv_epi(const float *x, int N, int C, int D, int H, int W,
                 const float *w, int CO, int KD, int KH, int KW, int stride,
                 int pad, int dil, const float *bias, int nops,
                 const int *kinds, const double *a, const double *b,
                 const float *chan, double *y) {
  int pad_d = (D == 1 && KD == 1) ? 0 : pad;
  int Do = out_extent(D, KD, stride, pad_d, dil);
  int Ho = out_extent(H, KH, stride, pad, dil);
  int Wo = out_extent(W, KW, stride, pad, dil);
  long plane = (long)Do * Ho * Wo;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int n = 0; n < N; ++n)
    for (int co = 0; co < CO; ++co) {
      double *yp = y + ((size_t)n * CO + co) * plane;
      for (int od = 0; od < Do; ++od)
        for (int oh = 0; oh < Ho; ++oh)
          for (int ow = 0; ow < Wo; ++ow) {
            double v = conv_one(x, C, D, H, W, w, KD, KH, KW, stride, pad_d,
                                pad, dil, bias, n, co, od, oh, ow);
            yp[((size_t)od * Ho + oh) * Wo + ow] =
                apply_chain(nops, kinds, a, b, chan, CO, co, v);
          }
    }
}

/* The same conv + chain evaluated only at the given flat output indices
 * (index into [N][CO][Do][Ho][Wo]).  Used to check full-size launches on a
 * sample of their outputs. */
void or_conv_epi_points(const float *x, int N, int C, int D, int H, int W,
                        const float *w, int CO, int KD, int KH, int KW,
                        int stride, int pad, int dil, const float *bias,
                        int nops, const int *kinds, const double *a,
                        const double *b, const float *chan, const int64_t *idx,
                        long npts, double *out) {
  int pad_d = (D == 1 && KD == 1) ? 0 : pad;
  int Do = out_extent(D, KD, stride, pad_d, dil);
  int Ho = out_extent(H, KH, stride, pad, dil);
  int Wo = out_extent(W, KW, stride, pad, dil);
  (void)N;
#pragma omp parallel for schedule(static)
  for (long i = 0; i < npts; ++i) {
    int64_t t = idx[i];
    int ow = (int)(t % Wo); t /= Wo;
    int oh = (int)(t % Ho); t /= Ho;
    int od = (int)(t % Do); t /= Do;
    int co = (int)(t % CO); t /= CO;
    int n = (int)t;
    double v = conv_one(x, C, D, H, W, w, KD, KH, KW, stride, pad_d, pad, dil,
                        bias, n, co, od, oh, ow);
    out[i] = apply_chain(nops, kinds, a, b, chan, CO, co, v);
  }
}

/* Scatter-form transposed conv for one (n, co) plane, plus bias.
 * plane: [Ho][Wo] doubles, overwritten. */
static void convT_plane(const float *x, int CI, int H, int W, const float *w,
                        int CO, int K, int stride, int pad, const float *bias,
                        int n, int co, int Ho, int Wo, double *plane) {
  double b0 = bias ? (double)bias[co] : 0.0;
  for (long t = 0; t < (long)Ho * Wo; ++t) plane[t] = b0;
  for (int ci = 0; ci < CI; ++ci)
    for (int i = 0; i < H; ++i)
      for (int j = 0; j < W; ++j) {
        double xv = x[(((size_t)n * CI + ci) * H + i) * W + j];
        for (int kh = 0; kh < K; ++kh) {
          int oh = i * stride + kh - pad;
          if (oh < 0 || oh >= Ho) continue;
          for (int kw = 0; kw < K; ++kw) {
            int ow = j * stride + kw - pad;
            if (ow < 0 || ow >= Wo) continue;
            double wv = w[(((size_t)ci * CO + co) * K + kh) * K + kw];
            plane[(size_t)oh * Wo + ow] += xv * wv;
          }
        }
      }
}

/* Full scatter-form ConvTranspose2d + bias.  w: [CI][CO][K][K].
 * y: [N][CO][Ho][Wo], Ho = (H-1)*stride - 2*pad + K + out_pad. */
void or_convT2d(const float *x, int N, int CI, int H, int W, const float *w,
                int CO, int K, int stride, int pad, int out_pad,
                const float *bias, double *y) {
  int Ho = (H - 1) * stride - 2 * pad + K + out_pad;
  int Wo = (W - 1) * stride - 2 * pad + K + out_pad;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int n = 0; n < N; ++n)
    for (int co = 0; co < CO; ++co)
      convT_plane(x, CI, H, W, w, CO, K, stride, pad, bias, n, co, Ho, Wo,
                  y + ((size_t)n * CO + co) * Ho * Wo);
}

/* MaxPool2d(k, s), no padding, floor extent.  in: [NC][H][W]. */
void or_maxpool2d(const double *in, long NC, int H, int W, int k, int s,
                  double *out) {
  int Hp = (H - k) / s + 1, Wp = (W - k) / s + 1;
  for (long c = 0; c < NC; ++c)
    for (int i = 0; i < Hp; ++i)
      for (int j = 0; j < Wp; ++j) {
        double m = -INFINITY;
        for (int u = 0; u < k; ++u)
          for (int v = 0; v < k; ++v) {
            double t = in[((size_t)c * H + i * s + u) * W + j * s + v];
            if (t > m) m = t;
          }
        out[((size_t)c * Hp + i) * Wp + j] = m;
      }
}

/* Mean over each plane of `plane` elements. */
void or_mean_hw(const double *in, long NC, long plane, double *out) {
  for (long c = 0; c < NC; ++c) {
    double s = 0.0;
    for (long t = 0; t < plane; ++t) s += in[(size_t)c * plane + t];
    out[c] = s / (double)plane;
  }
}

/* convT + bias -> maxpool(pk, ps) -> hardtanh[lo, hi] -> mean(H, W) -> tanh
 * for selected (n, co) pairs (nc[2*i], nc[2*i+1]).  out[i] is the final
 * value of that pair. */
void or_convT_pool_mean_points(const float *x, int N, int CI, int H, int W,
                               const float *w, int CO, int K, int stride,
                               int pad, int out_pad, const float *bias, int pk,
                               int ps, double lo, double hi, const int *nc,
                               long npts, double *out) {
  int Ho = (H - 1) * stride - 2 * pad + K + out_pad;
  int Wo = (W - 1) * stride - 2 * pad + K + out_pad;
  int Hp = (Ho - pk) / ps + 1, Wp = (Wo - pk) / ps + 1;
  (void)N;
#pragma omp parallel for schedule(dynamic)
  for (long i = 0; i < npts; ++i) {
    double *plane = (double *)malloc(sizeof(double) * (size_t)Ho * Wo);
    double *pooled = (double *)malloc(sizeof(double) * (size_t)Hp * Wp);
    convT_plane(x, CI, H, W, w, CO, K, stride, pad, bias, nc[2 * i],
                nc[2 * i + 1], Ho, Wo, plane);
    or_maxpool2d(plane, 1, Ho, Wo, pk, ps, pooled);
    for (long t = 0; t < (long)Hp * Wp; ++t)
      pooled[t] = or_apply_op(OR_HARDTANH, lo, hi, 0, 0, pooled[t]);
    double m;
    or_mean_hw(pooled, 1, (long)Hp * Wp, &m);
    out[i] = tanh(m);
    free(plane);
    free(pooled);
  }
}

/* Whole-tensor version of the chain above: out[N*CO]. */
void or_convT_pool_mean(const float *x, int N, int CI, int H, int W,
                        const float *w, int CO, int K, int stride, int pad,
                        int out_pad, const float *bias, int pk, int ps,
                        double lo, double hi, double *out) {
  long np = (long)N * CO;
  int *nc = (int *)malloc(sizeof(int) * 2 * (size_t)np);
  for (long i = 0; i < np; ++i) {
    nc[2 * i] = (int)(i / CO);
    nc[2 * i + 1] = (int)(i % CO);
  }
  or_convT_pool_mean_points(x, N, CI, H, W, w, CO, K, stride, pad, out_pad,
                            bias, pk, ps, lo, hi, nc, np, out);
  free(nc);
}
