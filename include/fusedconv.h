/*
 * fusedconv.h -- C ABI of libfusedconv: dense 2-D / 3-D convolutions
 * (kernel sizes 1-7, strides and dilations 1-4, any padding up to 64) and a
 * transposed convolution (kernel sizes 1-7, strides 1-4) with their
 * elementwise and reduction epilogues fused into the same kernel, for one
 * NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (three POPCORNBENCH reasoning traces):
 *  - fc_conv2d_epi: trace "Kimi-K2.6__l2_p57", problem statement and
 *    "simplest kernel" paragraph: Conv2d (bias, stride 1, padding 0) ->
 *    ReLU -> HardSwish x * clamp((x + 3) / 6, 0, 1).
 *  - fc_conv3d_epi: trace "Kimi-K2.6__l2_p90", problem statement: Conv3d
 *    (bias) -> LeakyReLU(0.2) -> + sum_tensor[C_out,1,1,1] -> clamp[-1, 1]
 *    -> GELU 0.5 x (1 + erf(x / sqrt 2)) (exact form, GELU accuracy
 *    paragraph).
 *  - fc_convT2d_pool_mean: trace "Kimi-K2.6__l2_p10", problem statement:
 *    ConvTranspose2d(k 3, stride 1, padding 1) (bias) -> MaxPool2d(2, 2) ->
 *    Hardtanh[-1, 1] -> mean over (H, W) keepdim -> tanh.  Computed as a
 *    plain convolution with swapped channel axes, both taps flipped and
 *    padding k - 1 - p (the trace's transposed-conv equivalence paragraph);
 *    at stride 2 per output parity class (the taps each class reads) on the
 *    input grid; the trace's general max-pool paragraph for other pool
 *    windows.
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers to contiguous fp32 arrays in
 *    PyTorch's default layouts: x NCHW / NCDHW (NHWC / NDHWC for the
 *    _nhwc / _ndhwc entry points, which also write y channels-last); conv weights
 *    [C_out][C_in][kD][kH][kW]; transposed-conv weights [C_in][C_out][k][k];
 *    bias [C_out]; per-channel tensors of epilogue ops [C_out].  The caller
 *    owns every buffer; the library allocates nothing.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous: they enqueue kernels and return.
 *  - `ws` is a caller-owned device workspace of at least
 *    fc_workspace_bytes(...) bytes, 256-byte aligned, that must not be used
 *    by another call in flight on another stream.  It holds the packed
 *    weights and (for the pooled entry point) the per-tile partial sums.
 *  - Invalid shapes, NULL or misaligned pointers, unsupported parameters or
 *    epilogue chains and a too-small workspace are rejected on the host
 *    before anything is launched, and the call returns a non-zero
 *    fc_status.  No exception ever crosses this boundary.  There is no CPU
 *    fallback: without a usable sm_103a device the calls return
 *    FC_ERR_CUDA.
 *  - Kernel-side failures (a bounded wait that ran out, an input value
 *    outside the range of the fp16-split variant) are recorded in a
 *    per-device status word that fc_get_last_device_error() reads.
 */
#ifndef FUSEDCONV_H
#define FUSEDCONV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FC_API __attribute__((visibility("default")))
#else
#define FC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FC_OK = 0,
  FC_ERR_INVALID_ARG = 1, /* bad shape, NULL pointer, bad op parameter */
  FC_ERR_UNSUPPORTED = 2, /* valid but not implemented (stride, pad, chain) */
  FC_ERR_ALIGNMENT = 3,   /* a pointer is not 16-byte aligned */
  FC_ERR_WORKSPACE = 4,   /* ws is NULL/misaligned or ws_bytes too small */
  FC_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
  FC_ERR_TIMEOUT = 6,     /* a kernel's bounded wait ran out (device) */
  FC_ERR_RANGE = 7        /* x or w outside the fp16-split range (device) */
} fc_status;

/* Epilogue ops, applied in order to the conv output (bias already added). */
typedef enum {
  FC_EPI_RELU = 1,        /* max(x, 0) */
  FC_EPI_HARDSWISH = 2,   /* x * clamp((x + 3) / 6, 0, 1) */
  FC_EPI_LEAKY_RELU = 3,  /* x > 0 ? x : a * x */
  FC_EPI_ADD_CHANNEL = 4, /* x + chan[c_out] (device pointer, C_out floats) */
  FC_EPI_CLAMP = 5,       /* min(max(x, a), b) */
  FC_EPI_GELU_ERF = 6,    /* 0.5 x (1 + erf(x / sqrt 2)) */
  FC_EPI_MAXPOOL2X2 = 7,  /* 2x2 window, stride 2, floor extent */
  FC_EPI_HARDTANH = 8,    /* min(max(x, a), b) */
  FC_EPI_MEAN_HW = 9,     /* mean over the (pooled) H x W plane */
  FC_EPI_TANH = 10,       /* tanh(x) */
  FC_EPI_MAXPOOL = 11     /* window a x a, stride b (integers 1 .. 4), floor extent
                             (H - a) / b + 1; pooled entry only */
} fc_epi_kind;

typedef struct {
  int kind;          /* fc_epi_kind */
  float a, b;        /* parameters, see fc_epi_kind */
  const float *chan; /* FC_EPI_ADD_CHANNEL only: device pointer [C_out] */
} fc_epi_op;

#define FC_MAX_EPI_OPS 8

typedef struct {
  const float *bias; /* device pointer [C_out] or NULL (no bias) */
  int n_ops;         /* 0 .. FC_MAX_EPI_OPS */
  fc_epi_op ops[FC_MAX_EPI_OPS];
} fc_epilogue;

/* How the contraction is computed.  AUTO picks per shape from a table of
 * measured times (fc_select_variant).  FFMA: fp32 CUDA-core
 * register-blocked direct conv (fixed-size kernels for 3 x 3 (x 3) at
 * stride / dilation 1-2, a general kernel for every other parameter).
 * TC_TF32X3: tcgen05 tensor cores, each fp32 operand split into a tf32
 * high part and a tf32 remainder, three products (hi*hi + hi*lo + lo*hi)
 * accumulated in fp32 in tensor memory.  TC_F16X3: the same split with fp16
 * parts (the remainder scaled by 2^11): same accuracy as TC_TF32X3 for
 * |x| < 65520 and |w| <= 65504 (fp16's largest finite value) as long as the
 * data is not tiny throughout -- the largest |w|, and the largest |x| that a
 * CTA stages, at least 2^-12 (below 2^-14 fp16 parts turn subnormal) --
 * twice the tensor rate; data outside that range sets FC_ERR_RANGE in the
 * device status word (run TC_TF32X3 or FFMA for it).  The tensor-core
 * variants take square odd kernels up to 7 x 7 (cubic up to 5 x 5 x 5) at
 * stride / dilation 1-2 where the plan fits shared memory. */
typedef enum {
  FC_VARIANT_AUTO = 0,
  FC_VARIANT_FFMA = 1,
  FC_VARIANT_TC_TF32X3 = 2,
  FC_VARIANT_TC_F16X3 = 3
} fc_variant;

/* Conv2d + bias + elementwise epilogue chain (any sequence of RELU,
 * HARDSWISH, LEAKY_RELU, ADD_CHANNEL, CLAMP, GELU_ERF, HARDTANH, TANH).
 * x [N][C_in][H][W]; w [C_out][C_in][kH][kW]; y [N][C_out][Ho][Wo] with
 * Ho = (H + 2 pad - dilation (kH - 1) - 1) / stride + 1 and Wo likewise
 * (floor), output (oh, ow) reading input row oh*stride + kh*dilation - pad
 * and column ow*stride + kw*dilation - pad (the dilated extent is the one
 * trace "Kimi-K2.6__l2_p10" states for pooling windows; its l2_p57 trace
 * names the layer's stride / padding / dilation defaults 1 / 0 / 1).
 * Supported: kH, kW 1..7, stride 1..4, dilation 1..4, 0 <= pad <= 64,
 * 1 <= C_in, 1 <= C_out, H + 2 pad and W + 2 pad at least the dilated
 * window, fewer than 2^31 elements per image of x, of y and in w (whole
 * tensors may be larger: offsets are 64-bit).  FFMA takes all of it;
 * the tensor-core variants the square odd kernels at stride / dilation
 * 1-2 whose plan fits (they stage stride 2 as even/odd row x column
 * sub-planes).  N = 0 is a valid empty call (nothing is launched).
 * Argument order: the boundary's base form is (..., stride, pad, epi, ...);
 * `dilation` is inserted after `pad` (every variant takes it). */
FC_API fc_status fc_conv2d_epi(const float *x, int N, int C_in, int H, int W,
                        const float *w, int C_out, int kH, int kW, int stride,
                        int pad, int dilation, const fc_epilogue *epi, float *y,
                        void *ws, size_t ws_bytes, void *stream);

/* fc_conv2d_epi for callers that cannot allocate device memory (code run
 * from a host callback or an allocator hook, allocation-free real-time or
 * certified paths, plug-ins whose host owns the memory pool).  The pages
 * have no counterpart to this call; it exists for those callers.
 * Same arguments and results as fc_conv2d_epi minus ws / ws_bytes: the
 * workspace is a fixed 1 MiB device array inside the library (held on every
 * GPU that loads the library until the process exits).  The caller still
 * passes x, w, the epilogue tensors and y.  Shapes whose workspace
 * (fc_workspace_bytes(0, dims)) exceeds 1 MiB are refused with
 * FC_ERR_WORKSPACE.  Nothing is allocated: no cudaMalloc / cudaFree and no
 * allocating library routine (keep fc_profile_enable off).
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * All calls on a device share the array and it keeps the last call's
 * contents (each call rewrites what it reads first); calls that overlap on
 * the GPU -- on different streams or host threads -- race on it. */
FC_API fc_status fc_conv2d_epi_noalloc(const float *x, int N, int C_in, int H, int W,
                                       const float *w, int C_out, int kH, int kW,
                                       int stride, int pad, int dilation,
                                       const fc_epilogue *epi, float *y, void *stream);

/* Conv3d + bias + elementwise epilogue chain; same ops as fc_conv2d_epi.
 * x [N][C_in][D][H][W]; w [C_out][C_in][kD][kH][kW];
 * y [N][C_out][Do][Ho][Wo], each extent
 * (in + 2 pad - dilation (k - 1) - 1) / stride + 1, output (od, oh, ow)
 * reading input od*stride + kd*dilation - pad on each axis.
 * Supported: kD, kH, kW 1..7, stride 1..4, dilation 1..4, pad 0..64 (the
 * same padding on every axis), as for fc_conv2d_epi; the general
 * CUDA-core kernel refuses (FC_ERR_UNSUPPORTED) a layer whose staged window
 * for one input channel exceeds its shared memory (large kernels at large
 * strides and dilations). */
FC_API fc_status fc_conv3d_epi(const float *x, int N, int C_in, int D, int H, int W,
                        const float *w, int C_out, int kD, int kH, int kW,
                        int stride, int pad, int dilation, const fc_epilogue *epi,
                        float *y, void *ws, size_t ws_bytes, void *stream);

/* Channels-last forms of fc_conv2d_epi / fc_conv3d_epi: the same
 * arguments (sizes as N, C_in, [D,] H, W; weights [C_out][C_in][k...] as
 * there), but x is [N][H][W][C_in] ([N][D][H][W][C_in]) and y is
 * [N][Ho][Wo][C_out] ([N][Do][Ho][Wo][C_out]).  A pixel's channels are then
 * adjacent: with C_in a multiple of 4 a tiled tensor copy (TMA) brings each
 * channel chunk's input halo -- rows of pixels of chunk_ci channels -- into
 * shared memory in one operation (fc_set_staging), else the producers read
 * pixels as 16-byte vectors; outputs are written as 16-byte vectors when
 * C_out is a multiple of 4.  Tensor-core variants only (FC_VARIANT_FFMA
 * returns FC_ERR_UNSUPPORTED; AUTO picks the tensor cores): stride 1, the
 * kernels and dilations the tensor-core variants take; other parameters
 * return FC_ERR_UNSUPPORTED.  Workspace: fc_workspace_bytes(0 or 1, ...) as
 * for the channels-first calls. */
FC_API fc_status fc_conv2d_epi_nhwc(const float *x, int N, int C_in, int H, int W,
                                    const float *w, int C_out, int kH, int kW, int stride,
                                    int pad, int dilation, const fc_epilogue *epi, float *y,
                                    void *ws, size_t ws_bytes, void *stream);
FC_API fc_status fc_conv3d_epi_ndhwc(const float *x, int N, int C_in, int D, int H, int W,
                                     const float *w, int C_out, int kD, int kH, int kW,
                                     int stride, int pad, int dilation, const fc_epilogue *epi,
                                     float *y, void *ws, size_t ws_bytes, void *stream);

/* ConvTranspose2d + bias -> MaxPool2d -> Hardtanh[a,b] -> mean(H,W)
 * -> tanh.  x [N][C_in][H][W]; w [C_in][C_out][k][k];
 * y [N][C_out][1][1].  The epilogue chain must be exactly
 * MAXPOOL2X2 (or MAXPOOL(k_p, s_p), window and stride 1..4), HARDTANH(a, b),
 * MEAN_HW, TANH.  Transposed-conv output extent Ho = (H - 1) stride -
 * 2 pad + k + out_pad (likewise Wo; the output-size formula of trace
 * "Kimi-K2.6__l2_p10"), pooled with the floor extent (Ho - k_p) / s_p + 1.
 * Supported: k 1..7, stride 1..4, 0 <= pad <= 64, 0 <= out_pad < stride,
 * Ho, Wo >= k_p.  How each form runs:
 *   stride 1, pad <= k - 1: the equivalent conv (swapped channel axes,
 *     flipped taps, padding k - 1 - pad) -- tensor cores for odd k (2x2/2
 *     pool: two conv rows per unit; other windows: one tile per window row,
 *     windows taken in shared memory), CUDA cores for every k;
 *   stride 2, k 3, pad 1, 2x2/2 pool: per output parity class on the input
 *     grid (tensor cores); the general CUDA-core kernel for FFMA;
 *   anything else: the general CUDA-core kernel (the zero-inserted input
 *     staged in shared memory), FFMA only.
 * The conv output never leaves the kernel.  The mean is reduced in a fixed
 * order (per-tile partials, then a second kernel sums them in index order),
 * so results are bitwise reproducible. */
FC_API fc_status fc_convT2d_pool_mean(const float *x, int N, int C_in, int H, int W,
                               const float *w, int C_out, int k, int stride,
                               int pad, int out_pad, const fc_epilogue *epi,
                               float *y, void *ws, size_t ws_bytes,
                               void *stream);

/* Workspace bytes needed by one call.  entry: 0 = fc_conv2d_epi (and the
 * _nhwc / _noalloc forms), 1 = fc_conv3d_epi (and _ndhwc),
 * 2 = fc_convT2d_pool_mean with the 2x2 pool (any supported stride and
 * out_pad), 3 = fc_convT2d_pool_mean with a general pool window.
 * dims:
 *   entry 0: {N, C_in, H, W, C_out, k, pad}
 *   entry 1: {N, C_in, D, H, W, C_out, k, pad}
 *   entry 2: {N, C_in, H, W, C_out, k, pad}
 *   entry 3: {N, C_in, H, W, C_out, k, pad, stride, out_pad,
 *             pool window, pool stride}
 * The size covers every variant, so it does not depend on the selection.
 * Returns 0 for an invalid entry or NULL dims. */
FC_API size_t fc_workspace_bytes(int entry, const int *dims);

/* The variant a call would run (FC_VARIANT_AUTO's choice, or the override
 * set by fc_set_variant), without a device and without running anything:
 * the automatic choice takes, among the shapes of a table of kernel times
 * measured per variant on a GB300 (same entry point, kernel size, stride,
 * dilation, layout and pool window), the one nearest in log2 of the MAC
 * count and of the channel counts, and its fastest variant this problem
 * supports.  entry / dims:
 *   0 fc_conv2d_epi, 4 fc_conv2d_epi_nhwc:
 *     {N, C_in, H, W, C_out, k, stride, pad, dilation}
 *   1 fc_conv3d_epi, 5 fc_conv3d_epi_ndhwc:
 *     {N, C_in, D, H, W, C_out, k, stride, pad, dilation}
 *   2 fc_convT2d_pool_mean:
 *     {N, C_in, H, W, C_out, k, stride, pad, out_pad, pool window, pool stride}
 * Returns an fc_variant (1 .. 3), or -1 for an invalid or unsupported
 * problem (or an override the problem does not support).  The pages have
 * no counterpart: it exposes the library's own selection. */
FC_API int fc_select_variant(int entry, const int *dims);

/* Process-wide variant override (FC_VARIANT_AUTO restores the automatic
 * choice).  Returns FC_ERR_INVALID_ARG for an unknown value.  Not
 * synchronised with calls running on other host threads. */
FC_API fc_status fc_set_variant(int variant);

/* How the tensor-core variants bring x into shared memory (process-wide,
 * like fc_set_variant).  1: tiled tensor copies (TMA) of the input halo --
 * one copy per channel chunk and depth slice into a ring of raw fp32 slots,
 * zeros outside the tensor supplied by the copy -- which producer warps then
 * split into the hi / lo operand slices; used where the plan allows it
 * (stride 1, channels-first W or channels-last C_in a multiple of 4, room
 * in shared memory), register loads elsewhere.  0: register loads by the
 * producer warps everywhere.  -1 (the default): chosen per shape together
 * with the variant, from the measured table (see fc_select_variant).  All
 * give the same results.  FC_ERR_INVALID_ARG for another value. */
FC_API fc_status fc_set_staging(int mode);

/* The input staging the calling thread's last successful entry-point call
 * used: 1 tensor copies, 0 register loads (and the CUDA-core variant). */
FC_API int fc_last_staging(void);

/* The variant the calling thread's last successful entry-point call used. */
FC_API int fc_last_variant(void);

/* Number of kernels the calling thread's last successful entry-point call
 * launched. */
FC_API int fc_last_launch_count(void);

/* Human-readable name of a status code (static string). */
FC_API const char *fc_status_string(fc_status s);

/* The pooled-mean tail alone, on a conv output the caller already holds
 * (trace "Kimi-K2.6__l2_p10", tail-kernel and general max-pool paragraphs):
 *   y[n][c] = tanh( mean_{i<Hp, j<Wp} clamp( max_{a,b<k} x[n][c][i*s+a][j*s+b],
 *                                             ht_lo, ht_hi ) ),
 *   Hp = (H - k) / s + 1, Wp = (W - k) / s + 1 (floor; rows/columns past the
 *   last whole window are dropped).
 * x: device, contiguous fp32 [N][C][H][W], 4-byte aligned.  y: device fp32
 * [N][C] (the [N][C][1][1] of the pooled entry), written in full.  Any
 * k >= 1, s >= 1 with k <= H, W (overlapping windows and gaps allowed).
 * Deterministic: per-plane sums in a fixed order.  Asynchronous on `stream`.
 * Errors: FC_ERR_INVALID_ARG (extents, k, s, ht_lo > ht_hi, null pointers
 * with N > 0), FC_ERR_ALIGNMENT, FC_ERR_UNSUPPORTED (N*C or H*W beyond
 * 2^31 - 1), FC_ERR_CUDA (launch failure).  fc_convT2d_pool_mean fuses this
 * tail into the conv and never writes x; this call serves callers with a
 * materialised conv output and measures what the fusion saves.  Its kernel
 * time is profiled under entry 3 by fc_profile_read. */
FC_API fc_status fc_pool_mean_tail(const float *x, int N, int C, int H, int W, int k, int s,
                                   float ht_lo, float ht_hi, float *y, void *stream);

/* Self-test of the kernels' bounded waits (failure detection without a GPU
 * fault).  Launches one block on `stream` in which one warp waits, with the
 * bounded-wait routine the conv kernels use and a limit of `limit_us`
 * microseconds, on an mbarrier that nothing completes: it gives up, records
 * the wait and raises the block's abort flag.  A second warp, waiting on
 * another such barrier under the kernels' normal 4 s limit, sees the flag
 * and gives up at once.  Afterwards fc_get_last_device_error returns
 * FC_ERR_TIMEOUT and fc_wait_report lists both waits (role tags 0x71000001,
 * and 0x79000002 for the one ended by the flag).  limit_us in
 * [1, 1000000], else FC_ERR_INVALID_ARG; FC_ERR_CUDA if the launch fails.
 * The pages have no counterpart: it tests this library's failure path. */
FC_API fc_status fc_selftest_wait_timeout(unsigned int limit_us, void *stream);

/* Synchronises `stream`, then reads and clears the current device's status
 * word.  Returns FC_OK, FC_ERR_TIMEOUT, FC_ERR_RANGE or FC_ERR_CUDA. */
FC_API fc_status fc_get_last_device_error(void *stream);

/* Kernel timing for benchmarks.  While enabled, every entry-point call
 * records a pair of CUDA events on its stream around its main (contraction
 * + epilogue) kernel; pack and finishing kernels are outside the pair.
 * fc_profile_read synchronises on the recorded events and returns, for one
 * entry (0 conv2d, 1 conv3d, 2 convT-pool-mean, 3 pool-mean tail), the summed milliseconds and
 * the number of timed launches since the last fc_profile_reset.  At most
 * 4096 pairs are kept; later launches are not timed.  Host-thread safe only
 * when one thread uses it at a time. */
FC_API fc_status fc_profile_enable(int on);
FC_API fc_status fc_profile_read(int entry, double *total_ms, int *launches);
FC_API void fc_profile_reset(void);

/* Diagnostics for FC_ERR_TIMEOUT.  Synchronises `stream`, copies the
 * current device's record of timed-out kernel waits into `out` (word 0:
 * number of timeouts since the last call; then 8 words per record, at most
 * 32 records: block, thread, barrier index, phase parity, the waiting
 * role's tag, the raw 64-bit barrier word (low, high), and the marker
 * 0x5afe), clears it, and returns the number of timeouts (-1 on error).
 * No counterpart on the pages: this is the failure-detection side of the
 * bounded waits. */
FC_API int fc_wait_report(void *stream, unsigned int *out, int max_words);

/* Library version (major * 10000 + minor * 100 + patch). */
FC_API int fc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FUSEDCONV_H */
