// fc_ffma.cu -- fp32 CUDA-core path: register-blocked direct convolution
// with the epilogue applied from registers, plus the fixed-order second
// stage of the pooled mean (shared by every variant).
//
// Design (the GB300 form of the smem-tiled direct conv that the
// Kimi-K2.6__l2_p57 trace sketches: an input halo tile plus the weights in
// shared memory, one output tile per block):
//   * block = 256 threads = 8 channel groups (one warp each, 8 output
//     channels per thread) x 32 pixel groups (one lane each, PR x PC output
//     pixels per thread), so a warp reads one weight vector by broadcast;
//   * C_in is consumed in chunks of 8 channels: the chunk's input halo
//     [8][KD][TH+2][TW+2] and its weights [8][taps][64] are staged in smem;
//   * eltwise mode (PR=1, PC=4): 32 x 4 output tile; pool mode (PR=PC=2):
//     each thread owns one 2x2 pooling window of a 16 x 8 tile, so the
//     window max, hardtanh and the per-tile partial sum need no exchange.
#include <cuda_runtime.h>

#include "fc_epi.cuh"
#include "fc_internal.h"

namespace fc {

namespace {

constexpr int kCiT = 8;   // input channels per staged chunk
constexpr int kCoT = 64;  // output channels per block

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Packed FFMA weights: wp[ci][tap][co] with ci padded to a multiple of 8
// and co to a multiple of 64 (zeros).  tap = (kd * KH + kh) * KW + kw.
// Transposed-conv weights W[ci][co][kh][kw] enter as the equivalent conv:
// wp[ci][kh'][kw'][co] = W[ci][co][KH-1-kh'][KW-1-kw'].
__global__ void ffma_pack_weights(const float *__restrict__ w, int C, int CO,
                                  int KD, int KH, int KW, int wlayout,
                                  int Cp, int COp, float *__restrict__ wp) {
  int taps = KD * KH * KW;
  long total = (long)Cp * taps * COp;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    int co = (int)(i % COp);
    int tap = (int)((i / COp) % taps);
    int ci = (int)(i / ((long)COp * taps));
    float v = 0.0f;
    if (ci < C && co < CO) {
      if (wlayout == 0) {
        v = w[((long)co * C + ci) * taps + tap];
      } else {
        int kh = tap / KW, kw = tap % KW;
        v = w[(((long)ci * CO + co) * KH + (KH - 1 - kh)) * KW + (KW - 1 - kw)];
      }
    }
    wp[i] = v;
  }
}

template <int KD, int PR, int PC, bool POOL, int CHAIN, int S, int DL>
__global__ void __launch_bounds__(256)
ffma_conv_kernel(ConvProblem p, const float *__restrict__ wp, int Cp, int COp,
                 float *__restrict__ partial, int n_th, int n_tw) {
  constexpr int K = 3;
  constexpr int TAPS = KD * K * K;
  constexpr int TW = 8 * PC, TH = 4 * PR;
  // staged input extent of an output tile at stride S, dilation DL
  constexpr int SPAN = (K - 1) * DL + 1;
  constexpr int SW = (TW - 1) * S + SPAN, SH = (TH - 1) * S + SPAN;
  static_assert(!POOL || (S == 1 && DL == 1), "the pooled path is stride 1, dilation 1");
  extern __shared__ __align__(16) float smem_f[];
  float (*s_w)[TAPS][kCoT] = reinterpret_cast<float (*)[TAPS][kCoT]>(smem_f);
  float (*s_in)[KD][SH][SW] =
      reinterpret_cast<float (*)[KD][SH][SW]>(smem_f + kCiT * TAPS * kCoT);

  const int tid = threadIdx.x;
  const int cg = tid >> 5;   // channel group (warp)
  const int pg = tid & 31;   // pixel group (lane)
  const int gr = pg >> 3, gc = pg & 7;

  long b = blockIdx.x;
  const int tw = (int)(b % n_tw); b /= n_tw;
  const int th = (int)(b % n_th); b /= n_th;
  const int od = (int)(b % p.Do); b /= p.Do;
  const int n = (int)(b % p.N); b /= p.N;
  const int cb = (int)b;

  const int oh0 = th * TH, ow0 = tw * TW;
  const int HW = p.H * p.W;
  const long x_n = (long)n * p.C * p.D * HW;

  float acc[PR][PC][8];
#pragma unroll
  for (int a = 0; a < PR; ++a)
#pragma unroll
    for (int c = 0; c < PC; ++c)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[a][c][j] = 0.0f;

  for (int ci0 = 0; ci0 < Cp; ci0 += kCiT) {
    __syncthreads();
    // stage the input halo of this channel chunk (zero padded)
    constexpr int NIN = kCiT * KD * SH * SW;
    for (int i = tid; i < NIN; i += 256) {
      int c = i % SW, r = (i / SW) % SH, kd = (i / (SW * SH)) % KD;
      int ci = i / (SW * SH * KD);
      int gci = ci0 + ci;
      int id = od * S + kd * DL - p.pad_d, ih = oh0 * S + r - p.pad, iw = ow0 * S + c - p.pad;
      float v = 0.0f;
      if (gci < p.C && id >= 0 && id < p.D && ih >= 0 && ih < p.H && iw >= 0 &&
          iw < p.W)
        v = __ldg(p.x + x_n + ((long)gci * p.D + id) * HW + (long)ih * p.W + iw);
      s_in[ci][kd][r][c] = v;
    }
    // stage the chunk's weights for this block's 64 output channels
    constexpr int NW4 = kCiT * TAPS * (kCoT / 4);
    for (int i = tid; i < NW4; i += 256) {
      int c4 = i % (kCoT / 4), t = (i / (kCoT / 4)) % TAPS, ci = i / (TAPS * (kCoT / 4));
      const float4 *src = reinterpret_cast<const float4 *>(
          wp + ((long)(ci0 + ci) * TAPS + t) * COp + cb * kCoT);
      reinterpret_cast<float4 *>(&s_w[ci][t][0])[c4] = __ldg(src + c4);
    }
    __syncthreads();

#pragma unroll 1
    for (int ci = 0; ci < kCiT; ++ci) {
#pragma unroll
      for (int kd = 0; kd < KD; ++kd) {
#pragma unroll
        for (int kh = 0; kh < K; ++kh) {
          float4 wv[K][2];
#pragma unroll
          for (int kw = 0; kw < K; ++kw) {
            const float4 *ws4 =
                reinterpret_cast<const float4 *>(&s_w[ci][(kd * K + kh) * K + kw][cg * 8]);
            wv[kw][0] = ws4[0];
            wv[kw][1] = ws4[1];
          }
#pragma unroll
          for (int a = 0; a < PR; ++a) {
            // input columns (gc*PC + c)*S + kw*DL of staged row
            // (gr*PR + a)*S + kh*DL
            float xin[(PC - 1) * S + SPAN];
#pragma unroll
            for (int q = 0; q < (PC - 1) * S + SPAN; ++q)
              xin[q] = s_in[ci][kd][(gr * PR + a) * S + kh * DL][gc * PC * S + q];
#pragma unroll
            for (int kw = 0; kw < K; ++kw)
#pragma unroll
              for (int c = 0; c < PC; ++c) {
                float xv = xin[c * S + kw * DL];
                acc[a][c][0] = fmaf(xv, wv[kw][0].x, acc[a][c][0]);
                acc[a][c][1] = fmaf(xv, wv[kw][0].y, acc[a][c][1]);
                acc[a][c][2] = fmaf(xv, wv[kw][0].z, acc[a][c][2]);
                acc[a][c][3] = fmaf(xv, wv[kw][0].w, acc[a][c][3]);
                acc[a][c][4] = fmaf(xv, wv[kw][1].x, acc[a][c][4]);
                acc[a][c][5] = fmaf(xv, wv[kw][1].y, acc[a][c][5]);
                acc[a][c][6] = fmaf(xv, wv[kw][1].z, acc[a][c][6]);
                acc[a][c][7] = fmaf(xv, wv[kw][1].w, acc[a][c][7]);
              }
          }
        }
      }
    }
  }

  const int co0 = cb * kCoT + cg * 8;
  if constexpr (!POOL) {
    const long plane = (long)p.Do * p.Ho * p.Wo;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int co = co0 + j;
      if (co >= p.CO) break;
      const float bias = p.epi.bias ? __ldg(p.epi.bias + co) : 0.0f;
      const float add = chain_addend<CHAIN>(p.epi, co);
      float *yc = p.y + ((long)n * p.CO + co) * plane + (long)od * p.Ho * p.Wo;
#pragma unroll
      for (int a = 0; a < PR; ++a) {
        const int oh = oh0 + gr * PR + a;
        if (oh >= p.Ho) continue;
#pragma unroll
        for (int c = 0; c < PC; ++c) {
          const int ow = ow0 + gc * PC + c;
          if (ow < p.Wo)
            yc[(long)oh * p.Wo + ow] = apply_chain<CHAIN>(p.epi, co, acc[a][c][j] + bias, add);
        }
      }
    }
  } else {
    // one 2x2 window per thread: window (wi, wj) of the pooled plane
    const int wi = (oh0 >> 1) + gr, wj = (ow0 >> 1) + gc;
    const bool valid = (wi < p.Ho / 2) && (wj < p.Wo / 2);
    float part[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int co = co0 + j;
      const float bias = (co < p.CO && p.epi.bias) ? __ldg(p.epi.bias + co) : 0.0f;
      float m = fmaxf(fmaxf(acc[0][0][j] + bias, acc[0][1][j] + bias),
                      fmaxf(acc[1][0][j] + bias, acc[1][1][j] + bias));
      m = fminf(fmaxf(m, p.ht_lo), p.ht_hi);
      part[j] = valid ? m : 0.0f;
    }
    // fixed-order butterfly over the 32 windows of this tile
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int j = 0; j < 8; ++j) part[j] += __shfl_xor_sync(0xffffffffu, part[j], off);
    if (pg == 0) {
      const int T = n_th * n_tw;
      const int t = th * n_tw + tw;
      float *dst = partial + ((long)n * T + t) * p.CO;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (co0 + j < p.CO) dst[co0 + j] = part[j];
    }
  }
}

// Second stage of the pooled mean: y[n][co] = tanh(sum_t partial[n][t][co] /
// count), summed in double in index order.
// y[n][c] = tanh(sum_t partial[n][t][c] * inv_count).  One block of 256
// threads per image, 64 channels at a time: thread (q, c) sums, in double and
// in index order, the t of quarter q, and the four quarter sums are added in
// the order 0, 1, 2, 3.  A fixed order, so the result does not depend on
// scheduling.
// General max-pool (window K, stride ps <= 4, floor extent) fused after a
// stride-1 3x3 conv (a transposed conv arrives rewritten as one): the
// general path of the Kimi-K2.6__l2_p10 trace's tail-kernel and max-pool
// paragraphs, computed without writing the conv output.  A block owns a
// 4 x 8 tile of pooled outputs and 64 output channels; thread (gr, gc)
// computes the K x K conv outputs of its window (conv rows
// (pi0 + gr) ps + a, columns (pj0 + gc) ps + b) for 8 channels from the
// staged input halo, takes their max, adds the bias, clamps, and the warp
// adds its 32 windows in a fixed butterfly order into one partial per
// (image, tile, channel).  Overlapping windows (K > ps) recompute the
// shared conv outputs.
constexpr int kPoolTH = 4, kPoolTW = 8;

template <int K>
__global__ void __launch_bounds__(256)
ffma_pool_general_kernel(ConvProblem p, const float *__restrict__ wp, int Cp, int COp,
                         float *__restrict__ partial, int n_th, int n_tw, int Hp, int Wp) {
  constexpr int TAPS = 9;
  constexpr int SHM = (kPoolTH - 1) * 4 + K + 2, SWM = (kPoolTW - 1) * 4 + K + 2;
  extern __shared__ __align__(16) float smem_g[];
  float (*s_w)[TAPS][kCoT] = reinterpret_cast<float (*)[TAPS][kCoT]>(smem_g);
  float (*s_in)[SHM][SWM] = reinterpret_cast<float (*)[SHM][SWM]>(smem_g + kCiT * TAPS * kCoT);
  const int ps = p.ps;
  const int SH = (kPoolTH - 1) * ps + K + 2, SW = (kPoolTW - 1) * ps + K + 2;

  const int tid = threadIdx.x;
  const int cg = tid >> 5, pg = tid & 31;
  const int gr = pg >> 3, gc = pg & 7;
  long b = blockIdx.x;
  const int tw = (int)(b % n_tw); b /= n_tw;
  const int th = (int)(b % n_th); b /= n_th;
  const int n = (int)(b % p.N); b /= p.N;
  const int cb = (int)b;
  const int pi0 = th * kPoolTH, pj0 = tw * kPoolTW;
  const int r0 = pi0 * ps, c0 = pj0 * ps;  // first conv row / column of the tile
  const int HW = p.H * p.W;
  const long x_n = (long)n * p.C * HW;

  float acc[K][K][8];
#pragma unroll
  for (int a = 0; a < K; ++a)
#pragma unroll
    for (int c = 0; c < K; ++c)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[a][c][j] = 0.0f;

  for (int ci0 = 0; ci0 < Cp; ci0 += kCiT) {
    __syncthreads();
    const int nin = kCiT * SH * SW;
    for (int i = tid; i < nin; i += 256) {
      const int c = i % SW, r = (i / SW) % SH, ci = i / (SW * SH);
      const int gci = ci0 + ci;
      const int ih = r0 + r - p.pad, iw = c0 + c - p.pad;
      float v = 0.0f;
      if (gci < p.C && ih >= 0 && ih < p.H && iw >= 0 && iw < p.W)
        v = __ldg(p.x + x_n + (long)gci * HW + (long)ih * p.W + iw);
      s_in[ci][r][c] = v;
    }
    constexpr int NW4 = kCiT * TAPS * (kCoT / 4);
    for (int i = tid; i < NW4; i += 256) {
      const int c4 = i % (kCoT / 4), t = (i / (kCoT / 4)) % TAPS, ci = i / (TAPS * (kCoT / 4));
      const float4 *src = reinterpret_cast<const float4 *>(
          wp + ((long)(ci0 + ci) * TAPS + t) * COp + cb * kCoT);
      reinterpret_cast<float4 *>(&s_w[ci][t][0])[c4] = __ldg(src + c4);
    }
    __syncthreads();
#pragma unroll 1
    for (int ci = 0; ci < kCiT; ++ci) {
#pragma unroll
      for (int kh = 0; kh < 3; ++kh) {
        float4 wv[3][2];
#pragma unroll
        for (int kw = 0; kw < 3; ++kw) {
          const float4 *ws4 = reinterpret_cast<const float4 *>(&s_w[ci][kh * 3 + kw][cg * 8]);
          wv[kw][0] = ws4[0];
          wv[kw][1] = ws4[1];
        }
#pragma unroll
        for (int a = 0; a < K; ++a) {
          float xin[K + 2];
#pragma unroll
          for (int q = 0; q < K + 2; ++q) xin[q] = s_in[ci][gr * ps + a + kh][gc * ps + q];
#pragma unroll
          for (int kw = 0; kw < 3; ++kw)
#pragma unroll
            for (int c = 0; c < K; ++c) {
              const float xv = xin[c + kw];
              acc[a][c][0] = fmaf(xv, wv[kw][0].x, acc[a][c][0]);
              acc[a][c][1] = fmaf(xv, wv[kw][0].y, acc[a][c][1]);
              acc[a][c][2] = fmaf(xv, wv[kw][0].z, acc[a][c][2]);
              acc[a][c][3] = fmaf(xv, wv[kw][0].w, acc[a][c][3]);
              acc[a][c][4] = fmaf(xv, wv[kw][1].x, acc[a][c][4]);
              acc[a][c][5] = fmaf(xv, wv[kw][1].y, acc[a][c][5]);
              acc[a][c][6] = fmaf(xv, wv[kw][1].z, acc[a][c][6]);
              acc[a][c][7] = fmaf(xv, wv[kw][1].w, acc[a][c][7]);
            }
        }
      }
    }
  }

  const int co0 = cb * kCoT + cg * 8;
  const bool valid = (pi0 + gr < Hp) && (pj0 + gc < Wp);
  float part[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int co = co0 + j;
    const float bias = (co < p.CO && p.epi.bias) ? __ldg(p.epi.bias + co) : 0.0f;
    float m = acc[0][0][j];
#pragma unroll
    for (int a = 0; a < K; ++a)
#pragma unroll
      for (int c = 0; c < K; ++c) m = fmaxf(m, acc[a][c][j]);
    m = fminf(fmaxf(m + bias, p.ht_lo), p.ht_hi);
    part[j] = valid ? m : 0.0f;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
#pragma unroll
    for (int j = 0; j < 8; ++j) part[j] += __shfl_xor_sync(0xffffffffu, part[j], off);
  if (pg == 0) {
    const int T = n_th * n_tw;
    float *dst = partial + ((long)n * T + th * n_tw + tw) * p.CO;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (co0 + j < p.CO) dst[co0 + j] = part[j];
  }
}

template <int K>
cudaError_t launch_pool_general(const ConvProblem &p, const float *wp, int Cp, int COp,
                                float *partial, int n_th, int n_tw, int Hp, int Wp,
                                cudaStream_t s) {
  constexpr int SHM = (kPoolTH - 1) * 4 + K + 2, SWM = (kPoolTW - 1) * 4 + K + 2;
  constexpr size_t smem = sizeof(float) * (kCiT * 9 * kCoT + kCiT * SHM * SWM);
  const long blocks = (long)(COp / kCoT) * p.N * n_th * n_tw;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
  auto kern = ffma_pool_general_kernel<K>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  prof_begin(s);
  kern<<<(unsigned)blocks, 256, smem, s>>>(p, wp, Cp, COp, partial, n_th, n_tw, Hp, Wp);
  prof_end(s, p.entry);
  return cudaGetLastError();
}

constexpr int kFinishQ = 4;
constexpr int kFinishThreads = 64 * kFinishQ;

__global__ void __launch_bounds__(kFinishThreads)
pool_finish_kernel(const float *__restrict__ partial, int N, int CO, int T, double inv_count,
                   float *__restrict__ y) {
  __shared__ double qsum[kFinishQ][64];
  const int n = blockIdx.x;
  const int q = threadIdx.x / 64, cl = threadIdx.x % 64;
  const int tq = (T + kFinishQ - 1) / kFinishQ;
  const int t0 = q * tq, t1 = min(T, t0 + tq);
  for (int c0 = 0; c0 < CO; c0 += 64) {
    const int co = c0 + cl;
    double s = 0.0;
    if (co < CO) {
      const float *src = partial + (long)n * T * CO + co;
      for (int t = t0; t < t1; ++t) s += (double)src[(long)t * CO];
    }
    qsum[q][cl] = s;
    __syncthreads();
    if (q == 0 && co < CO) {
      double tot = qsum[0][cl];
      for (int k = 1; k < kFinishQ; ++k) tot += qsum[k][cl];
      y[(long)n * CO + co] = (float)tanh(tot * inv_count);
    }
    __syncthreads();
  }
}

template <int KD, int PR, int PC, bool POOL, int CHAIN, int S = 1, int DL = 1>
cudaError_t launch_one(const ConvProblem &p, const float *wp, int Cp, int COp,
                       float *partial, cudaStream_t s) {
  constexpr int TW = 8 * PC, TH = 4 * PR;
  int n_tw = ceil_div(p.Wo, TW), n_th = ceil_div(p.Ho, TH);
  long blocks = (long)(COp / kCoT) * p.N * p.Do * n_th * n_tw;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
  constexpr int SPAN = 2 * DL + 1;
  constexpr size_t smem = sizeof(float) * (kCiT * KD * 9 * kCoT +
                                           kCiT * KD * ((TH - 1) * S + SPAN) * ((TW - 1) * S + SPAN));
  auto kern = ffma_conv_kernel<KD, PR, PC, POOL, CHAIN, S, DL>;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  prof_begin(s);
  kern<<<(unsigned)blocks, 256, smem, s>>>(p, wp, Cp, COp, partial, n_th, n_tw);
  prof_end(s, p.entry);
  return cudaGetLastError();
}

template <int KD, int S, int DL>
cudaError_t launch_eltwise(const ConvProblem &p, const float *wp, int Cp, int COp,
                           cudaStream_t s) {
  switch (p.chain) {
    case CHAIN_NONE:
      return launch_one<KD, 1, 4, false, CHAIN_NONE, S, DL>(p, wp, Cp, COp, nullptr, s);
    case CHAIN_RELU_HARDSWISH:
      return launch_one<KD, 1, 4, false, CHAIN_RELU_HARDSWISH, S, DL>(p, wp, Cp, COp, nullptr, s);
    case CHAIN_LEAKY_ADD_CLAMP_GELU:
      return launch_one<KD, 1, 4, false, CHAIN_LEAKY_ADD_CLAMP_GELU, S, DL>(p, wp, Cp, COp, nullptr, s);
    case CHAIN_LEAKY_ADD_CLAMP1_GELU:
      return launch_one<KD, 1, 4, false, CHAIN_LEAKY_ADD_CLAMP1_GELU, S, DL>(p, wp, Cp, COp, nullptr, s);
    default: return launch_one<KD, 1, 4, false, CHAIN_GENERIC, S, DL>(p, wp, Cp, COp, nullptr, s);
  }
}

template <int KD>
cudaError_t launch_eltwise_kd(const ConvProblem &p, const float *wp, int Cp, int COp,
                              cudaStream_t s) {
  if (p.stride == 2)
    return p.dil == 2 ? launch_eltwise<KD, 2, 2>(p, wp, Cp, COp, s)
                      : launch_eltwise<KD, 2, 1>(p, wp, Cp, COp, s);
  return p.dil == 2 ? launch_eltwise<KD, 1, 2>(p, wp, Cp, COp, s)
                    : launch_eltwise<KD, 1, 1>(p, wp, Cp, COp, s);
}

}  // namespace

// Pooled extents (floor): (Ho - pk) / ps + 1.
static int pooled_h(const ConvProblem &p) { return (p.Ho - p.pk) / p.ps + 1; }
static int pooled_w(const ConvProblem &p) { return (p.Wo - p.pk) / p.ps + 1; }
static bool pool_general(const ConvProblem &p) { return p.pk != 2 || p.ps != 2; }

bool ffma_fixed_supported(const ConvProblem &p) {
  if (p.gen || p.cl || p.subpix) return false;
  if (p.KH != 3 || p.KW != 3 || !(p.KD == 1 || p.KD == 3)) return false;
  if (p.pool) return p.KD == 1 && p.stride == 1 && p.dil == 1;
  return p.stride <= 2 && p.dil <= 2;
}

int ffma_pool_tiles_per_image(const ConvProblem &p) {
  if (!ffma_fixed_supported(p)) return ffma_gen_tiles_per_image(p);
  if (pool_general(p)) return ceil_div(pooled_h(p), kPoolTH) * ceil_div(pooled_w(p), kPoolTW);
  return ceil_div(p.Ho, 8) * ceil_div(p.Wo, 16);
}

cudaError_t pool_finish_launch(const ConvProblem &p, const float *partials,
                               int tiles_per_image, cudaStream_t s) {
  int count = pooled_h(p) * pooled_w(p);
  pool_finish_kernel<<<p.N, kFinishThreads, 0, s>>>(partials, p.N, p.CO, tiles_per_image,
                                                    1.0 / (double)count, p.y);
  return cudaGetLastError();
}

cudaError_t ffma_launch(const ConvProblem &p, void *ws, const WsLayout &L,
                        cudaStream_t s, int *launches) {
  const int Cp = ceil_div(p.C, kCiT) * kCiT;
  const int COp = ceil_div(p.CO, kCoT) * kCoT;
  float *wp = reinterpret_cast<float *>(static_cast<char *>(ws) + L.ffma_w);
  const int taps = p.KD * p.KH * p.KW;
  long total = (long)Cp * taps * COp;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 1024) blocks = 1024;
  ffma_pack_weights<<<blocks, 256, 0, s>>>(p.w, p.C, p.CO, p.KD, p.KH, p.KW,
                                           p.wlayout, Cp, COp, wp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *launches = 1;
  if (!ffma_fixed_supported(p)) {
    float *partial = reinterpret_cast<float *>(static_cast<char *>(ws) + L.partial);
    return ffma_gen_launch(p, wp, Cp, COp, p.pool ? partial : nullptr, s, launches);
  }
  if (p.pool && pool_general(p)) {
    float *partial = reinterpret_cast<float *>(static_cast<char *>(ws) + L.partial);
    const int Hp = pooled_h(p), Wp = pooled_w(p);
    const int n_th = ceil_div(Hp, kPoolTH), n_tw = ceil_div(Wp, kPoolTW);
    switch (p.pk) {
      case 1: e = launch_pool_general<1>(p, wp, Cp, COp, partial, n_th, n_tw, Hp, Wp, s); break;
      case 2: e = launch_pool_general<2>(p, wp, Cp, COp, partial, n_th, n_tw, Hp, Wp, s); break;
      case 3: e = launch_pool_general<3>(p, wp, Cp, COp, partial, n_th, n_tw, Hp, Wp, s); break;
      default: e = launch_pool_general<4>(p, wp, Cp, COp, partial, n_th, n_tw, Hp, Wp, s); break;
    }
    if (e != cudaSuccess) return e;
    e = pool_finish_launch(p, partial, n_th * n_tw, s);
    *launches += 2;
    return e;
  }
  if (p.pool) {
    float *partial = reinterpret_cast<float *>(static_cast<char *>(ws) + L.partial);
    e = launch_one<1, 2, 2, true, CHAIN_NONE>(p, wp, Cp, COp, partial, s);
    if (e != cudaSuccess) return e;
    e = pool_finish_launch(p, partial, ffma_pool_tiles_per_image(p), s);
    *launches += 2;
    return e;
  }
  e = (p.KD == 1) ? launch_eltwise_kd<1>(p, wp, Cp, COp, s)
                  : launch_eltwise_kd<3>(p, wp, Cp, COp, s);
  *launches += 1;
  return e;
}

}  // namespace fc
