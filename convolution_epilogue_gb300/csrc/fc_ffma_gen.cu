// fc_ffma_gen.cu -- general layer parameters on the CUDA cores: any kernel
// size 1..7 per axis, stride 1..4, dilation 1..4 and padding for the
// convolutions, and the transposed convolution with any stride 1..4,
// padding and output padding followed by a max pool of any window / stride
// 1..4 (floor extent), hardtanh, mean and tanh.  The fixed-size kernels of
// fc_ffma.cu and fc_tc.cu take the parameters the workloads use; this one
// takes everything else the entry points accept.
//
// One formulation covers both: an output is a cross-correlation of a
// virtual input X with packed weights,
//   out[co][o] = sum_{ci, k} X[ci][o * S + k * DL - pad] * Wp[ci][k][co]
// per spatial axis, where X is x itself for a convolution, and for a
// transposed convolution of stride s the input with s - 1 zeros inserted
// between neighbours (X[u] = x[u / s] when s divides u), read with stride 1,
// dilation 1, both taps flipped, channels swapped and padding k - 1 - p --
// the equivalence the Kimi-K2.6__l2_p10 trace derives for stride 1, with
// the stride's zero insertion written out (output extent
// (H - 1) s - 2 p + k + op, the trace's ConvTranspose2d size formula).  The
// zeros are materialised only in shared memory, where the block stages its
// input window.
//
// Block: 256 threads = 8 channel groups (warps, 8 output channels each) x
// 32 pixel groups (lanes).  Elementwise mode: lane (gr, gc) = (l / 8, l % 8)
// computes output row oh0 + gr, columns ow0 + 4 gc .. + 3 (a 4 x 32 tile).
// Pooled mode: lane (gr, gc) computes the PK x PK conv outputs of pooled
// window (pi0 + gr, pj0 + gc) (a 4 x 8 tile of windows), overlapping
// windows recomputing what they share; max, bias, clamp, then a fixed-order
// warp sum into one partial per (image, tile, channel) that the finishing
// kernel reduces in index order.
#include <cuda_runtime.h>

#include "fc_epi.cuh"
#include "fc_internal.h"

namespace fc {

namespace {

constexpr int kCoT = 64;
constexpr int kGenTH = 4, kGenTW = 32;  // elementwise output tile
constexpr int kGenPH = 4, kGenPW = 8;   // pooled-window tile
constexpr int kGenSmemMax = 200 * 1024;

// Geometry of a general launch (host-computed).
struct GenGeom {
  int KD, KH, KW, S, DL;
  int pd, ph, pw;     // padding of the virtual input (may be negative)
  int ST;             // zero-insertion stride of the virtual input (1: none)
  int XD, XH, XW;     // virtual input extents ((n - 1) ST + 1 for a transposed conv)
  int CI_T;           // input channels staged per chunk
  int SD, SH, SW;     // staged input window per chunk
  int taps;
  int tiles_h, tiles_w;
  int Hp, Wp, pk, ps; // pooled extents, window and stride (pooled mode)
};

inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// Virtual input element (zero outside, zero between the inserted samples).
__device__ __forceinline__ float virt_x(const ConvProblem &p, const GenGeom &g, long xnc, int d,
                                        int r, int c) {
  if (d < 0 || r < 0 || c < 0 || d >= g.XD || r >= g.XH || c >= g.XW) return 0.0f;
  if (g.ST > 1) {
    if (r % g.ST || c % g.ST) return 0.0f;
    r /= g.ST;
    c /= g.ST;
  }
  return __ldg(p.x + xnc + ((long)d * p.H + r) * p.W + c);
}

template <int CHAIN, int PK>
__global__ void __launch_bounds__(256)
ffma_gen_kernel(ConvProblem p, GenGeom g, const float *__restrict__ wp, int Cp, int COp,
                float *__restrict__ partial) {
  extern __shared__ __align__(16) float smem_g[];
  const int taps = g.taps;
  float *s_w = smem_g;                                  // [CI_T][taps][64]
  float *s_in = smem_g + (long)g.CI_T * taps * kCoT;     // [CI_T][SD][SH][SW]
  const int plane_in = g.SD * g.SH * g.SW;

  const int tid = threadIdx.x;
  const int cg = tid >> 5, pg = tid & 31;
  const int gr = pg >> 3, gc = pg & 7;

  long b = blockIdx.x;
  const int tw = (int)(b % g.tiles_w); b /= g.tiles_w;
  const int th = (int)(b % g.tiles_h); b /= g.tiles_h;
  const int od = (int)(b % p.Do); b /= p.Do;
  const int n = (int)(b % p.N); b /= p.N;
  const int cb = (int)b;

  // first conv output row / column of the tile
  int r0, c0;
  if constexpr (PK == 0) {
    r0 = th * kGenTH;
    c0 = tw * kGenTW;
  } else {
    r0 = th * kGenPH * g.ps;
    c0 = tw * kGenPW * g.ps;
  }
  // first virtual-input element of the staged window
  const int vd0 = od * g.S - g.pd, vr0 = r0 * g.S - g.ph, vc0 = c0 * g.S - g.pw;

  constexpr int NA = PK == 0 ? 1 : PK, NB = PK == 0 ? 4 : PK;
  float acc[NA][NB][8];
#pragma unroll
  for (int a = 0; a < NA; ++a)
#pragma unroll
    for (int c = 0; c < NB; ++c)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[a][c][j] = 0.0f;

  for (int ci0 = 0; ci0 < Cp; ci0 += g.CI_T) {
    __syncthreads();
    const int nin = g.CI_T * plane_in;
    for (int i = tid; i < nin; i += 256) {
      const int c = i % g.SW, r = (i / g.SW) % g.SH, d = (i / (g.SW * g.SH)) % g.SD;
      const int ci = i / plane_in, gci = ci0 + ci;
      float v = 0.0f;
      if (gci < p.C)
        v = virt_x(p, g, ((long)n * p.C + gci) * p.D * p.H * p.W, vd0 + d, vr0 + r, vc0 + c);
      s_in[i] = v;
    }
    const int nw4 = g.CI_T * taps * (kCoT / 4);
    for (int i = tid; i < nw4; i += 256) {
      const int c4 = i % (kCoT / 4), t = (i / (kCoT / 4)) % taps, ci = i / (taps * (kCoT / 4));
      const float4 *src = reinterpret_cast<const float4 *>(
          wp + ((long)(ci0 + ci) * taps + t) * COp + cb * kCoT);
      reinterpret_cast<float4 *>(s_w + ((long)ci * taps + t) * kCoT)[c4] = __ldg(src + c4);
    }
    __syncthreads();

    for (int ci = 0; ci < g.CI_T; ++ci) {
      const float *xin = s_in + (long)ci * plane_in;
      for (int kd = 0; kd < g.KD; ++kd)
        for (int kh = 0; kh < g.KH; ++kh)
          for (int kw = 0; kw < g.KW; ++kw) {
            const int t = (kd * g.KH + kh) * g.KW + kw;
            const float4 *ws4 = reinterpret_cast<const float4 *>(s_w + ((long)ci * taps + t) * kCoT + cg * 8);
            const float4 w0 = ws4[0], w1 = ws4[1];
            const float *xd = xin + (kd * g.DL) * g.SH * g.SW;
#pragma unroll
            for (int a = 0; a < NA; ++a)
#pragma unroll
              for (int c = 0; c < NB; ++c) {
                int rr, cc;
                if constexpr (PK == 0) {
                  rr = gr * g.S + kh * g.DL;
                  cc = (gc * 4 + c) * g.S + kw * g.DL;
                } else {
                  rr = gr * g.ps + a + kh;
                  cc = gc * g.ps + c + kw;
                }
                const float xv = xd[rr * g.SW + cc];
                acc[a][c][0] = fmaf(xv, w0.x, acc[a][c][0]);
                acc[a][c][1] = fmaf(xv, w0.y, acc[a][c][1]);
                acc[a][c][2] = fmaf(xv, w0.z, acc[a][c][2]);
                acc[a][c][3] = fmaf(xv, w0.w, acc[a][c][3]);
                acc[a][c][4] = fmaf(xv, w1.x, acc[a][c][4]);
                acc[a][c][5] = fmaf(xv, w1.y, acc[a][c][5]);
                acc[a][c][6] = fmaf(xv, w1.z, acc[a][c][6]);
                acc[a][c][7] = fmaf(xv, w1.w, acc[a][c][7]);
              }
          }
    }
  }

  const int co0 = cb * kCoT + cg * 8;
  if constexpr (PK == 0) {
    const long plane = (long)p.Do * p.Ho * p.Wo;
    const int oh = r0 + gr;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int co = co0 + j;
      if (co >= p.CO || oh >= p.Ho) break;
      const float bias = p.epi.bias ? __ldg(p.epi.bias + co) : 0.0f;
      const float add = chain_addend<CHAIN>(p.epi, co);
      float *yc = p.y + ((long)n * p.CO + co) * plane + ((long)od * p.Ho + oh) * p.Wo;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int ow = c0 + gc * 4 + c;
        if (ow < p.Wo) yc[ow] = apply_chain<CHAIN>(p.epi, co, acc[0][c][j] + bias, add);
      }
    }
  } else {
    const bool valid = (th * kGenPH + gr < g.Hp) && (tw * kGenPW + gc < g.Wp);
    float part[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int co = co0 + j;
      const float bias = (co < p.CO && p.epi.bias) ? __ldg(p.epi.bias + co) : 0.0f;
      float m = acc[0][0][j];
#pragma unroll
      for (int a = 0; a < PK; ++a)
#pragma unroll
        for (int c = 0; c < PK; ++c) m = fmaxf(m, acc[a][c][j]);
      m = fminf(fmaxf(m + bias, p.ht_lo), p.ht_hi);
      part[j] = valid ? m : 0.0f;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int j = 0; j < 8; ++j) part[j] += __shfl_xor_sync(0xffffffffu, part[j], off);
    if (pg == 0) {
      const int T = g.tiles_h * g.tiles_w;
      float *dst = partial + ((long)n * T + th * g.tiles_w + tw) * p.CO;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (co0 + j < p.CO) dst[co0 + j] = part[j];
    }
  }
}

// Geometry for a problem; returns false if no chunk size fits shared memory.
bool gen_geom(const ConvProblem &p, GenGeom &g, size_t *smem) {
  g.KD = p.KD; g.KH = p.KH; g.KW = p.KW;
  g.taps = p.KD * p.KH * p.KW;
  if (p.pool) {  // transposed conv over the zero-inserted input, stride 1
    g.S = 1; g.DL = 1;
    g.ST = p.tstride;
    g.pd = 0;
    g.ph = p.KH - 1 - p.tpad;
    g.pw = p.KW - 1 - p.tpad;
    g.XD = 1;
    g.XH = (p.H - 1) * g.ST + 1;
    g.XW = (p.W - 1) * g.ST + 1;
    g.pk = p.pk; g.ps = p.ps;
    g.Hp = (p.Ho - p.pk) / p.ps + 1;
    g.Wp = (p.Wo - p.pk) / p.ps + 1;
    g.tiles_h = cdiv(g.Hp, kGenPH);
    g.tiles_w = cdiv(g.Wp, kGenPW);
    const int rows = (kGenPH - 1) * g.ps + g.pk, cols = (kGenPW - 1) * g.ps + g.pk;
    g.SD = 1;
    g.SH = rows + p.KH - 1;
    g.SW = cols + p.KW - 1;
  } else {
    g.S = p.stride; g.DL = p.dil; g.ST = 1;
    g.pd = p.pad_d; g.ph = g.pw = p.pad;
    g.XD = p.D; g.XH = p.H; g.XW = p.W;
    g.pk = g.ps = 1; g.Hp = g.Wp = 0;
    g.tiles_h = cdiv(p.Ho, kGenTH);
    g.tiles_w = cdiv(p.Wo, kGenTW);
    g.SD = (p.KD - 1) * p.dil + 1;
    g.SH = (kGenTH - 1) * p.stride + (p.KH - 1) * p.dil + 1;
    g.SW = (kGenTW - 1) * p.stride + (p.KW - 1) * p.dil + 1;
  }
  const size_t per_ci = sizeof(float) * ((size_t)g.taps * kCoT + (size_t)g.SD * g.SH * g.SW);
  int ci_t = 8;
  while (ci_t > 1 && per_ci * ci_t > (size_t)kGenSmemMax) ci_t >>= 1;
  if (per_ci * ci_t > (size_t)kGenSmemMax) return false;
  g.CI_T = ci_t;
  *smem = per_ci * ci_t;
  return true;
}

template <int CHAIN, int PK>
cudaError_t launch_gen(const ConvProblem &p, const GenGeom &g, size_t smem, const float *wp,
                       int Cp, int COp, float *partial, cudaStream_t s) {
  const long blocks = (long)(COp / kCoT) * p.N * p.Do * g.tiles_h * g.tiles_w;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
  auto kern = ffma_gen_kernel<CHAIN, PK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  prof_begin(s);
  kern<<<(unsigned)blocks, 256, smem, s>>>(p, g, wp, Cp, COp, partial);
  prof_end(s, p.entry);
  return cudaGetLastError();
}

}  // namespace

int ffma_gen_channel_chunk(const ConvProblem &p) {
  GenGeom g{};
  size_t smem = 0;
  return gen_geom(p, g, &smem) ? g.CI_T : 0;
}

int ffma_gen_tiles_per_image(const ConvProblem &p) {
  GenGeom g{};
  size_t smem = 0;
  if (!gen_geom(p, g, &smem)) return 0;
  return g.tiles_h * g.tiles_w;
}

// The general kernel; wp holds the packed weights [Cp][taps][COp] (Cp a
// multiple of 8, so of every chunk size).
cudaError_t ffma_gen_launch(const ConvProblem &p, const float *wp, int Cp, int COp, float *partial,
                            cudaStream_t s, int *launches) {
  GenGeom g{};
  size_t smem = 0;
  if (!gen_geom(p, g, &smem)) return cudaErrorNotSupported;
  cudaError_t e;
  if (p.pool) {
    switch (p.pk) {
      case 1: e = launch_gen<CHAIN_NONE, 1>(p, g, smem, wp, Cp, COp, partial, s); break;
      case 2: e = launch_gen<CHAIN_NONE, 2>(p, g, smem, wp, Cp, COp, partial, s); break;
      case 3: e = launch_gen<CHAIN_NONE, 3>(p, g, smem, wp, Cp, COp, partial, s); break;
      default: e = launch_gen<CHAIN_NONE, 4>(p, g, smem, wp, Cp, COp, partial, s); break;
    }
    if (e != cudaSuccess) return e;
    *launches += 1;
    e = pool_finish_launch(p, partial, g.tiles_h * g.tiles_w, s);
    *launches += 1;
    return e;
  }
  switch (p.chain) {
    case CHAIN_NONE: e = launch_gen<CHAIN_NONE, 0>(p, g, smem, wp, Cp, COp, nullptr, s); break;
    case CHAIN_RELU_HARDSWISH:
      e = launch_gen<CHAIN_RELU_HARDSWISH, 0>(p, g, smem, wp, Cp, COp, nullptr, s); break;
    case CHAIN_LEAKY_ADD_CLAMP_GELU:
      e = launch_gen<CHAIN_LEAKY_ADD_CLAMP_GELU, 0>(p, g, smem, wp, Cp, COp, nullptr, s); break;
    case CHAIN_LEAKY_ADD_CLAMP1_GELU:
      e = launch_gen<CHAIN_LEAKY_ADD_CLAMP1_GELU, 0>(p, g, smem, wp, Cp, COp, nullptr, s); break;
    default: e = launch_gen<CHAIN_GENERIC, 0>(p, g, smem, wp, Cp, COp, nullptr, s); break;
  }
  *launches += 1;
  return e;
}

}  // namespace fc
