// fc_epi.cuh -- the elementwise epilogue ops, applied in registers to a conv
// output that already carries its bias.
//
// Each op is written from its definition in the traces:
//   HardSwish x * clamp((x + 3) / 6, 0, 1)   (Kimi-K2.6__l2_p57, problem)
//   LeakyReLU(a), + per-channel tensor, clamp, exact GELU
//   0.5 x (1 + erf(x / sqrt 2))               (Kimi-K2.6__l2_p90, problem and
//                                              GELU accuracy paragraph)
//   Hardtanh, tanh                            (Kimi-K2.6__l2_p10, problem)
// erff / tanhf are CUDA's own functions (no fast-math approximations).
#pragma once
#include "fc_internal.h"
#include "fc_tc_ptx.cuh"

namespace fc {

// x * clamp((x + 3) / 6, 0, 1), the gate as one saturated multiply-add.
__device__ __forceinline__ float op_hardswish(float v) {
  return v * __saturatef(fmaf(v, 1.0f / 6.0f, 0.5f));
}

// GELU for |v| <= 1 (the fused conv3d chain clamps to [-1, 1] first):
//   GELU(v) = v/2 + v/2 erf(v / sqrt 2) = v/2 + s R(s),   s = v^2,
// with R(s) = (GELU(v) - v/2) / s an even, entire function of v, replaced on
// s in [0, 1] by the degree-4 polynomial below: the minimax fit of the GELU
// error s (R(s) - p(s)) by weighted least squares with Lawson's iteration,
// computed by gen_gelu_poly.py next to this file.  Fit error 4e-9; in fp32
// Horner form within 1e-7 of GELU on [-1, 1] (the result's own rounding
// level), far inside the 1e-4 tolerance.
constexpr float kGeluR0 = 0.39894208f, kGeluR1 = -0.06648772f, kGeluR2 = 0.00996112f,
                kGeluR3 = -0.0011617212f, kGeluR4 = 9.097826e-05f;  // s^0 .. s^4

__device__ __forceinline__ float op_gelu_small(float v) {
  const float s = v * v;
  float r = fmaf(kGeluR4, s, kGeluR3);
  r = fmaf(r, s, kGeluR2);
  r = fmaf(r, s, kGeluR1);
  r = fmaf(r, s, kGeluR0);
  return fmaf(s, r, 0.5f * v);
}

// The same for two values on the paired fp32 pipe (bit-identical per lane).
__device__ __forceinline__ uint64_t op_gelu_small2(uint64_t v) {
  const uint64_t s = ptx::mul2(v, v);
  uint64_t r = ptx::fma2(ptx::pk2(kGeluR4, kGeluR4), s, ptx::pk2(kGeluR3, kGeluR3));
  r = ptx::fma2(r, s, ptx::pk2(kGeluR2, kGeluR2));
  r = ptx::fma2(r, s, ptx::pk2(kGeluR1, kGeluR1));
  r = ptx::fma2(r, s, ptx::pk2(kGeluR0, kGeluR0));
  return ptx::fma2(s, r, ptx::mul2(v, ptx::pk2(0.5f, 0.5f)));
}

__device__ __forceinline__ float op_gelu_erf(float v) {
  return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
}

__device__ __forceinline__ float apply_op(int kind, float a, float b,
                                          const float *chan, int co, float v) {
  switch (kind) {
    case FC_EPI_RELU: return fmaxf(v, 0.0f);
    case FC_EPI_HARDSWISH: return op_hardswish(v);
    case FC_EPI_LEAKY_RELU: return v > 0.0f ? v : a * v;
    case FC_EPI_ADD_CHANNEL: return v + __ldg(chan + co);
    case FC_EPI_CLAMP:
    case FC_EPI_HARDTANH: return fminf(fmaxf(v, a), b);
    case FC_EPI_GELU_ERF: return op_gelu_erf(v);
    case FC_EPI_TANH: return tanhf(v);
    default: return v;
  }
}

// v already includes the bias.  `add` is the per-channel value of the
// ADD_CHANNEL op for the fused chain (pre-loaded by the caller).
template <int CHAIN>
__device__ __forceinline__ float apply_chain(const EpiDev &e, int co, float v,
                                             float add) {
  if constexpr (CHAIN == CHAIN_NONE) {
    return v;
  } else if constexpr (CHAIN == CHAIN_RELU_HARDSWISH) {
    return op_hardswish(fmaxf(v, 0.0f));
  } else if constexpr (CHAIN == CHAIN_LEAKY_ADD_CLAMP_GELU) {
    v = v > 0.0f ? v : e.a[0] * v;
    v = v + add;
    v = fminf(fmaxf(v, e.a[2]), e.b[2]);
    return op_gelu_erf(v);
  } else if constexpr (CHAIN == CHAIN_LEAKY_ADD_CLAMP1_GELU) {
    v = fmaxf(v, e.a[0] * v);  // LeakyReLU for a slope in [0, 1]
    v = v + add;
    v = fminf(fmaxf(v, e.a[2]), e.b[2]);  // inside [-1, 1]
    return op_gelu_small(v);
  } else {
    for (int i = 0; i < e.n_ops; ++i)
      v = apply_op(e.kind[i], e.a[i], e.b[i], e.chan[i], co, v);
    return v;
  }
}

// The general chain on N consecutive output channels co0 .. co0 + N - 1 of
// one pixel, v already carrying the bias.  The op loop is outside and the
// values inside, so each op's kind and parameters are read and dispatched
// once per N outputs instead of once per output.  Every value sees the same
// ops in the same order as in apply_chain<CHAIN_GENERIC> (bit-identical
// results).  Only the first `nco` channels exist (ADD_CHANNEL reads only
// those; the caller stores only those).
template <int N>
__device__ __forceinline__ void apply_chain_generic_n(const EpiDev &e, int co0, int nco,
                                                      float (&v)[N]) {
#pragma unroll 1
  for (int i = 0; i < e.n_ops; ++i) {
    const float a = e.a[i], b = e.b[i];
    switch (e.kind[i]) {
      case FC_EPI_RELU:
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] = fmaxf(v[j], 0.0f);
        break;
      case FC_EPI_HARDSWISH:
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] = op_hardswish(v[j]);
        break;
      case FC_EPI_LEAKY_RELU:
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] = v[j] > 0.0f ? v[j] : a * v[j];
        break;
      case FC_EPI_ADD_CHANNEL: {
        const float *ch = e.chan[i] + co0;
#pragma unroll
        for (int j = 0; j < N; ++j)
          if (j < nco) v[j] = v[j] + __ldg(ch + j);
        break;
      }
      case FC_EPI_CLAMP:
      case FC_EPI_HARDTANH:
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] = fminf(fmaxf(v[j], a), b);
        break;
      case FC_EPI_GELU_ERF:
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] = op_gelu_erf(v[j]);
        break;
      case FC_EPI_TANH:
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] = tanhf(v[j]);
        break;
      default:
        break;
    }
  }
}

// Two adjacent channels of one pixel through the fused chains on the paired
// fp32 pipe, from conv sums already combined (hi + scale lo) in registers:
// y = chain(x + bias).  Bit-identical to apply_chain on each lane (the
// paired ops round per lane like the scalar ones).  Only the two fixed
// chains.
template <int CHAIN>
__device__ __forceinline__ void apply_chain2x(const EpiDev &e, float v0, float v1, float b0,
                                              float b1, float a0, float a1, float &o0,
                                              float &o1) {
  uint64_t x = ptx::add2(ptx::pk2(v0, v1), ptx::pk2(b0, b1));
  float x0, x1;
  if constexpr (CHAIN == CHAIN_RELU_HARDSWISH) {
    ptx::upk2(x, x0, x1);
    x0 = fmaxf(x0, 0.0f);
    x1 = fmaxf(x1, 0.0f);
    const float g0 = __saturatef(fmaf(x0, 1.0f / 6.0f, 0.5f));
    const float g1 = __saturatef(fmaf(x1, 1.0f / 6.0f, 0.5f));
    ptx::upk2(ptx::mul2(ptx::pk2(x0, x1), ptx::pk2(g0, g1)), o0, o1);
  } else {  // CHAIN_LEAKY_ADD_CLAMP1_GELU
    float t0, t1;
    ptx::upk2(x, x0, x1);
    ptx::upk2(ptx::mul2(x, ptx::pk2(e.a[0], e.a[0])), t0, t1);
    x = ptx::add2(ptx::pk2(fmaxf(x0, t0), fmaxf(x1, t1)), ptx::pk2(a0, a1));
    ptx::upk2(x, x0, x1);
    x0 = fminf(fmaxf(x0, e.a[2]), e.b[2]);
    x1 = fminf(fmaxf(x1, e.a[2]), e.b[2]);
    ptx::upk2(op_gelu_small2(ptx::pk2(x0, x1)), o0, o1);
  }
}

// Per-channel addend used by CHAIN_LEAKY_ADD_CLAMP_GELU (op 1).
template <int CHAIN>
__device__ __forceinline__ float chain_addend(const EpiDev &e, int co) {
  if constexpr (CHAIN == CHAIN_LEAKY_ADD_CLAMP_GELU || CHAIN == CHAIN_LEAKY_ADD_CLAMP1_GELU)
    return __ldg(e.chan[1] + co);
  else return 0.0f;
}

}  // namespace fc
