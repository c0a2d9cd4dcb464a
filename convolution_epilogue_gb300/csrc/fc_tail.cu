// fc_tail.cu -- the standalone pooled-mean tail on a materialised conv
// output: y[n][c] = tanh(mean_{i,j} hardtanh(max_{a,b<k} x[n][c][i*s+a][j*s+b]))
// with the floor output extent (H - k) / s + 1 (Kimi-K2.6__l2_p10 trace:
// the tail kernel and its general max-pool paragraphs).  The fused entry
// fc_convT2d_pool_mean never writes the conv output; this kernel exists to
// measure what that fusion saves and for callers that already hold a conv
// output.
//
// One block of kTailThreads per (n, c) plane.  Thread t takes the pooled
// pixels t, t + kTailThreads, ... in row-major order (consecutive threads
// read consecutive input columns) and keeps an fp32 sum; the block adds the
// per-thread sums in double in a fixed order (warp shuffle tree, then the
// warps in index order), so the result does not depend on scheduling.
#include "fc_internal.h"

namespace fc {
namespace {

constexpr int kTailThreads = 256;

template <bool K2S2>
__global__ void __launch_bounds__(kTailThreads)
tail_kernel(const float *__restrict__ x, int H, int W, int k, int s, int Hp, int Wp, float lo,
            float hi, double inv_count, float *__restrict__ y) {
  const long plane = blockIdx.x;
  const float *xp = x + plane * (long)H * W;
  const int np = Hp * Wp;
  float acc = 0.0f;
  for (int pix = threadIdx.x; pix < np; pix += kTailThreads) {
    const int i = pix / Wp, j = pix - i * Wp;
    float m;
    if constexpr (K2S2) {  // 2x2 window at (2i, 2j): two 8-byte loads
      const float2 a = __ldg(reinterpret_cast<const float2 *>(xp + (long)(2 * i) * W + 2 * j));
      const float2 b = __ldg(reinterpret_cast<const float2 *>(xp + (long)(2 * i + 1) * W + 2 * j));
      m = fmaxf(fmaxf(a.x, a.y), fmaxf(b.x, b.y));
    } else {
      const float *w0 = xp + (long)(i * s) * W + j * s;
      m = __ldg(w0);
      for (int a = 0; a < k; ++a)
        for (int b = 0; b < k; ++b) m = fmaxf(m, __ldg(w0 + (long)a * W + b));
    }
    acc += fminf(fmaxf(m, lo), hi);
  }
  double d = (double)acc;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
  __shared__ double ws[kTailThreads / 32];
  if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = d;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = ws[0];
    for (int w = 1; w < kTailThreads / 32; ++w) t += ws[w];
    y[plane] = (float)tanh(t * inv_count);
  }
}

}  // namespace

cudaError_t tail_launch(const float *x, long planes, int H, int W, int k, int s, float lo,
                        float hi, float *y, cudaStream_t st, int *launches) {
  const int Hp = (H - k) / s + 1, Wp = (W - k) / s + 1;
  const double inv = 1.0 / ((double)Hp * Wp);
  const bool fast = k == 2 && s == 2 && (W % 2) == 0 &&
                    (reinterpret_cast<uintptr_t>(x) % 8) == 0;
  prof_begin(st);
  if (fast)
    tail_kernel<true><<<(unsigned)planes, kTailThreads, 0, st>>>(x, H, W, k, s, Hp, Wp, lo, hi,
                                                                 inv, y);
  else
    tail_kernel<false><<<(unsigned)planes, kTailThreads, 0, st>>>(x, H, W, k, s, Hp, Wp, lo, hi,
                                                                  inv, y);
  prof_end(st, 3);
  *launches = 1;
  return cudaGetLastError();
}

}  // namespace fc
