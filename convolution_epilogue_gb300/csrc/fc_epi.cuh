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

__device__ __forceinline__ float op_hardswish(float v) {
  float g = fminf(fmaxf((v + 3.0f) * (1.0f / 6.0f), 0.0f), 1.0f);
  return v * g;
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
  } else {
    for (int i = 0; i < e.n_ops; ++i)
      v = apply_op(e.kind[i], e.a[i], e.b[i], e.chan[i], co, v);
    return v;
  }
}

// Per-channel addend used by CHAIN_LEAKY_ADD_CLAMP_GELU (op 1).
template <int CHAIN>
__device__ __forceinline__ float chain_addend(const EpiDev &e, int co) {
  if constexpr (CHAIN == CHAIN_LEAKY_ADD_CLAMP_GELU) return __ldg(e.chan[1] + co);
  else return 0.0f;
}

}  // namespace fc
