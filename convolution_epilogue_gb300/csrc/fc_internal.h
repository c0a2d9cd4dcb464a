// fc_internal.h -- host/device shared declarations of libfusedconv (not part
// of the public ABI).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fusedconv.h"

namespace fc {

// Elementwise chains with a specialised fast path; anything else runs the
// generic op interpreter.
enum ChainId : int {
  CHAIN_GENERIC = 0,
  CHAIN_NONE = 1,             // no op after the bias
  CHAIN_RELU_HARDSWISH = 2,   // relu -> hardswish
  CHAIN_LEAKY_ADD_CLAMP_GELU = 3,  // leaky(a) -> + chan -> clamp[a,b] -> gelu
  CHAIN_LEAKY_ADD_CLAMP1_GELU = 4  // the same with [a,b] inside [-1,1]
};

// Epilogue as the kernels see it (passed by value).
struct EpiDev {
  const float *bias;
  int n_ops;
  int kind[FC_MAX_EPI_OPS];
  float a[FC_MAX_EPI_OPS];
  float b[FC_MAX_EPI_OPS];
  const float *chan[FC_MAX_EPI_OPS];
};

// One conv problem after the host has validated it.  2-D problems have
// D = Do = KD = 1 and pad_d = 0.  Transposed convs arrive here already
// rewritten as a conv (swapped + flipped weights, pad k - 1 - p).
struct ConvProblem {
  const float *x;
  const float *w;  // caller layout (see wlayout)
  float *y;        // eltwise: [N][CO][Do][Ho][Wo]; pool: [N][CO]
  int N, C, D, H, W;
  int CO, KD, KH, KW;
  int pad_d, pad;  // zero padding on D and on H/W
  int stride;      // conv stride on every spatial axis (1 or 2)
  int dil;         // conv dilation on every spatial axis (1 or 2)
  int Do, Ho, Wo;
  int wlayout;     // 0: conv [CO][C][KD][KH][KW]; 1: convT [C][CO][KH][KW]
  int pool;        // 1: 2x2 maxpool -> hardtanh -> mean -> tanh
  // 1: stride-2 transposed conv (k 3, pad 1) computed per output parity
  // class on the input grid (x, w in transposed-conv form, no rewrite);
  // Ho, Wo are then the transposed conv's output extents.
  int subpix;
  int pk, ps;      // pooled entry: max-pool window and stride (floor extent)
  // pooled entry: the transposed conv's own stride, padding and output
  // padding (the fields above describe the kernels' rewritten form)
  int tstride, tpad, top;
  // 1: only the general CUDA-core kernel (fc_ffma_gen.cu) computes this
  // problem (kernel sizes, strides, dilations or transposed-conv
  // parameters outside the fixed-size kernels)
  int gen;
  int staging;     // tensor-core input staging: 1 tensor copies where possible, 0 loads
  int cl;          // 1: x is N(D)HWC and y is N(Do)(Ho)(Wo)C_out (channels last)
  float ht_lo, ht_hi;
  int chain;       // ChainId
  int entry;       // 0 conv2d, 1 conv3d, 2 convT-pool-mean (for profiling)
  EpiDev epi;
  unsigned int *status;  // device status word
  // per-block maxima of |w| written by the fp16-split weight pack (wmax_n
  // floats in the workspace), read back by the main kernel's range check
  float *wmax;
  int wmax_n;
};

// Status bits written by kernels.
// ST_PLAN: a kernel met a plan it cannot run (a defect of the library, not
// of the inputs); it stopped without touching memory and reports FC_ERR_CUDA.
enum : unsigned int { ST_TIMEOUT = 1u, ST_RANGE = 2u, ST_PLAN = 4u };

// Workspace regions (byte offsets, all 256-aligned).
struct WsLayout {
  size_t ffma_w, ffma_w_bytes;
  size_t tc_w, tc_w_bytes;
  size_t partial, partial_bytes;
  size_t wmax, wmax_bytes;  // per-block maxima of |w| (fp16-split range check)
  size_t total;
};

WsLayout ws_layout(const ConvProblem &p);
// Most blocks the tensor-core weight pack launches (one |w| maximum each).
constexpr int kMaxPackBlocks = 2048;

// Event pair around a main kernel (no-ops unless fc_profile_enable(1)).
void prof_begin(cudaStream_t s);
void prof_end(cudaStream_t s, int entry);

// Launchers (each returns cudaSuccess or the launch error) and the number of
// kernels they launched through *launches.
cudaError_t ffma_launch(const ConvProblem &p, void *ws, const WsLayout &L,
                        cudaStream_t s, int *launches);
cudaError_t pool_finish_launch(const ConvProblem &p, const float *partials,
                               int tiles_per_image, cudaStream_t s);
int ffma_pool_tiles_per_image(const ConvProblem &p);
// General CUDA-core kernel: launch (pack already done), channels staged per
// chunk (0: the problem does not fit its shared memory) and pooled tiles.
cudaError_t ffma_gen_launch(const ConvProblem &p, const float *wp, int Cp, int COp, float *partial,
                            cudaStream_t s, int *launches);
int ffma_gen_channel_chunk(const ConvProblem &p);
int ffma_gen_tiles_per_image(const ConvProblem &p);
// Whether the fixed-size CUDA-core kernels of fc_ffma.cu take this problem.
bool ffma_fixed_supported(const ConvProblem &p);

// Tensor-core path.  prec: 0 = tf32x3, 1 = f16x3.
bool tc_supported(const ConvProblem &p, int prec);
// Whether a tensor-core plan for the problem (with its `staging` field)
// stages the input with tensor copies.
int tc_uses_tma(const ConvProblem &p, int prec);
cudaError_t tc_launch(const ConvProblem &p, int prec, void *ws,
                      const WsLayout &L, cudaStream_t s, int *launches);
int tc_pool_tiles_per_image(const ConvProblem &p);
size_t tc_weight_bytes(const ConvProblem &p);
cudaError_t selftest_wait_launch(unsigned int *status, uint64_t limit_ns, cudaStream_t s);

// Standalone pooled-mean tail over `planes` H x W planes (fc_tail.cu).
cudaError_t tail_launch(const float *x, long planes, int H, int W, int k, int s, float lo,
                        float hi, float *y, cudaStream_t st, int *launches);

}  // namespace fc
