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

namespace fc {

// x * clamp((x + 3) / 6, 0, 1), the gate as one saturated multiply-add.
__device__ __forceinline__ float op_hardswish(float v) {
  return v * __saturatef(fmaf(v, 1.0f / 6.0f, 0.5f));
}

// erf(z) by its Maclaurin series, erf(z) = 2/sqrt(pi) sum_n (-1)^n
// z^(2n+1) / (n! (2n+1)), truncated after n = 8 (Horner in z^2).  For
// |z| <= 1/sqrt(2) the first omitted term is below 3e-10, far under fp32
// rounding; used only where the argument is known to be that small.
__device__ __forceinline__ float erf_maclaurin(float z) {
  constexpr float c[9] = {1.128379167e+00f, -3.761263890e-01f, 1.128379167e-01f, -2.686617065e-02f, 5.223977625e-03f, -8.548327023e-04f, 1.205533298e-04f, -1.492565036e-05f, 1.646211437e-06f};
  const float z2 = z * z;
  float p = c[8];
#pragma unroll
  for (int n = 7; n >= 0; --n) p = fmaf(p, z2, c[n]);
  return z * p;
}

// GELU for |v| <= 1 (its argument v / sqrt 2 is then within the series'
// range).
__device__ __forceinline__ float op_gelu_small(float v) {
  const float h = 0.5f * v;
  return fmaf(h, erf_maclaurin(v * 0.70710678118654752f), h);
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
    v = v > 0.0f ? v : e.a[0] * v;
    v = v + add;
    v = fminf(fmaxf(v, e.a[2]), e.b[2]);  // inside [-1, 1]
    return op_gelu_small(v);
  } else {
    for (int i = 0; i < e.n_ops; ++i)
      v = apply_op(e.kind[i], e.a[i], e.b[i], e.chan[i], co, v);
    return v;
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
