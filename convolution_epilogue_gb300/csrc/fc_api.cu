// fc_api.cu -- the C ABI of libfusedconv: validation, epilogue decoding,
// variant selection, workspace layout and launches.  Nothing here computes
// a conv value; every step of the path runs in the kernels.
#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "fc_internal.h"
#include "fc_variant_table.h"

namespace fc {

namespace {

// Per-device status area: word 0 is the status word (kernels OR bits into
// it; fc_get_last_device_error reads and clears it); word 1 counts
// timed-out waits and words 2.. hold up to 32 records of 8 words each
// describing where those waits gave up (read by fc_wait_report).
constexpr int kStatusWords = 2 + 32 * 8;
__device__ unsigned int g_status_word[kStatusWords];

constexpr int kMaxDevices = 64;
unsigned int *g_status_ptr[kMaxDevices];

int g_variant_override = FC_VARIANT_AUTO;
// Input staging of the tensor-core variants: -1 chosen per shape with the
// variant (measured table), 0 register loads, 1 tensor copies where the
// plan allows them.
int g_staging_override = -1;
thread_local int t_last_variant = 0;
thread_local int t_last_launches = 0;
thread_local int t_last_staging = 0;

// ---- benchmark profiling: event pairs around main kernels
constexpr int kMaxProf = 4096;
bool g_prof_on = false;
cudaEvent_t g_prof_ev[kMaxProf][2];
int g_prof_entry[kMaxProf];
int g_prof_n = 0;       // pairs recorded since reset
int g_prof_created = 0; // pairs whose events exist
bool g_prof_open = false;

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

fc_status status_ptr(unsigned int **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return FC_ERR_CUDA;
  if (!g_status_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return FC_ERR_CUDA;
    g_status_ptr[dev] = static_cast<unsigned int *>(p);
  }
  *out = g_status_ptr[dev];
  return FC_OK;
}

bool elementwise_kind(int k) {
  return k == FC_EPI_RELU || k == FC_EPI_HARDSWISH || k == FC_EPI_LEAKY_RELU ||
         k == FC_EPI_ADD_CHANNEL || k == FC_EPI_CLAMP || k == FC_EPI_GELU_ERF ||
         k == FC_EPI_HARDTANH || k == FC_EPI_TANH;
}

// Decode an elementwise chain into EpiDev + a ChainId.
fc_status decode_eltwise(const fc_epilogue *epi, EpiDev *e, int *chain) {
  memset(e, 0, sizeof(*e));
  if (!epi) {
    *chain = CHAIN_NONE;
    return FC_OK;
  }
  if (epi->bias && !aligned16(epi->bias)) return FC_ERR_ALIGNMENT;
  if (epi->n_ops < 0 || epi->n_ops > FC_MAX_EPI_OPS) return FC_ERR_INVALID_ARG;
  e->bias = epi->bias;
  e->n_ops = epi->n_ops;
  for (int i = 0; i < epi->n_ops; ++i) {
    const fc_epi_op &o = epi->ops[i];
    if (!elementwise_kind(o.kind)) return FC_ERR_UNSUPPORTED;
    if (o.kind == FC_EPI_ADD_CHANNEL && !o.chan) return FC_ERR_INVALID_ARG;
    if ((o.kind == FC_EPI_CLAMP || o.kind == FC_EPI_HARDTANH) && !(o.a <= o.b))
      return FC_ERR_INVALID_ARG;
    e->kind[i] = o.kind;
    e->a[i] = o.a;
    e->b[i] = o.b;
    e->chan[i] = o.chan;
  }
  const int n = epi->n_ops;
  if (n == 0) *chain = CHAIN_NONE;
  else if (n == 2 && e->kind[0] == FC_EPI_RELU && e->kind[1] == FC_EPI_HARDSWISH)
    *chain = CHAIN_RELU_HARDSWISH;
  else if (n == 4 && e->kind[0] == FC_EPI_LEAKY_RELU &&
           e->kind[1] == FC_EPI_ADD_CHANNEL &&
           (e->kind[2] == FC_EPI_CLAMP || e->kind[2] == FC_EPI_HARDTANH) &&
           e->kind[3] == FC_EPI_GELU_ERF)
    // GELU's argument within [-1, 1] and a slope in [0, 1]: the polynomial
    // GELU and LeakyReLU as max(v, a v)
    *chain = (e->a[2] >= -1.0f && e->b[2] <= 1.0f && e->a[0] >= 0.0f && e->a[0] <= 1.0f)
                 ? CHAIN_LEAKY_ADD_CLAMP1_GELU
                 : CHAIN_LEAKY_ADD_CLAMP_GELU;
  else
    *chain = CHAIN_GENERIC;
  return FC_OK;
}

// The pooled entry point accepts exactly MAXPOOL2X2 (or MAXPOOL(k, s)),
// HARDTANH, MEAN_HW, TANH.
fc_status decode_pool(const fc_epilogue *epi, EpiDev *e, float *lo, float *hi, int *pk,
                      int *ps) {
  memset(e, 0, sizeof(*e));
  if (!epi) return FC_ERR_INVALID_ARG;
  if (epi->bias && !aligned16(epi->bias)) return FC_ERR_ALIGNMENT;
  if (epi->n_ops != 4) return FC_ERR_UNSUPPORTED;
  const int want[4] = {FC_EPI_MAXPOOL2X2, FC_EPI_HARDTANH, FC_EPI_MEAN_HW, FC_EPI_TANH};
  for (int i = 1; i < 4; ++i)
    if (epi->ops[i].kind != want[i]) return FC_ERR_UNSUPPORTED;
  if (epi->ops[0].kind == FC_EPI_MAXPOOL2X2) {
    *pk = *ps = 2;
  } else if (epi->ops[0].kind == FC_EPI_MAXPOOL) {
    const float a = epi->ops[0].a, b = epi->ops[0].b;
    if (!(a >= 1.0f && a <= 4.0f && b >= 1.0f && b <= 4.0f) || a != (float)(int)a ||
        b != (float)(int)b)
      return FC_ERR_UNSUPPORTED;  // window and stride: integers 1 .. 4
    *pk = (int)a;
    *ps = (int)b;
  } else {
    return FC_ERR_UNSUPPORTED;
  }
  if (!(epi->ops[1].a <= epi->ops[1].b)) return FC_ERR_INVALID_ARG;
  e->bias = epi->bias;
  *lo = epi->ops[1].a;
  *hi = epi->ops[1].b;
  return FC_OK;
}

bool fits_int32(long long v) { return v >= 0 && v < (1LL << 31); }

bool variant_supported(const ConvProblem &p, int v) {
  if (v == FC_VARIANT_TC_TF32X3) return !p.gen && tc_supported(p, 0);
  if (v == FC_VARIANT_TC_F16X3) return !p.gen && tc_supported(p, 1);
  if (v == FC_VARIANT_FFMA)  // the fixed-size kernels, else the general one (no channels-last form)
    return !p.cl && (ffma_fixed_supported(p) || ffma_gen_channel_chunk(p) > 0);
  return false;
}

// Built-in rule, used when the measured table has no row of the problem's
// category: the tensor-core f16-split path once there is enough work.
int rule_variant(const ConvProblem &p) {
  if (p.gen) return FC_VARIANT_FFMA;
  if (p.subpix || p.cl) return tc_supported(p, 1) ? FC_VARIANT_TC_F16X3 : FC_VARIANT_TC_TF32X3;
  if (p.pool && (p.pk != 2 || p.ps != 2)) return FC_VARIANT_FFMA;  // general pool windows
  const double macs = (double)p.N * p.CO * p.Do * p.Ho * p.Wo * p.C * p.KD * p.KH * p.KW;
  if (tc_supported(p, 1) && macs >= 4.0e8) return FC_VARIANT_TC_F16X3;
  if (tc_supported(p, 0) && macs >= 4.0e8) return FC_VARIANT_TC_TF32X3;
  return FC_VARIANT_FFMA;
}

double problem_macs(const ConvProblem &p) {
  if (p.subpix)  // stride-2 transposed conv: each input pixel meets each tap once
    return (double)p.N * p.C * p.CO * p.H * p.W * p.KH * p.KW;
  return (double)p.N * p.CO * p.Do * p.Ho * p.Wo * p.C * p.KD * p.KH * p.KW;
}

// Automatic choice from measured times (fc_variant_table.h): among the
// table rows of the problem's category (entry point, kernel size, stride,
// dilation, layout, pool window), the one nearest in log2 MACs and log2
// channel counts; its (variant, staging) pairs in order of measured time,
// the first the problem supports.  Returns the variant and sets *staging.
int auto_choice(const ConvProblem &p, int *staging) {
  *staging = 1;
  if (p.gen) return FC_VARIANT_FFMA;  // only the general kernel computes it
  const int entry = p.pool ? 2 : p.entry;  // 0 conv2d, 1 conv3d, 2 pooled
  const int stride = p.pool ? p.tstride : p.stride;
  const int pgen = p.pool && (p.pk != 2 || p.ps != 2);
  const double lm = log2(problem_macs(p) + 1.0), lc = log2((double)p.C), lco = log2((double)p.CO);
  int best = -1;
  double bd = 0.0;
  const int nrows = (int)(sizeof(kVariantTable) / sizeof(kVariantTable[0]));
  for (int i = 0; i < nrows; ++i) {
    const VariantRow &r = kVariantTable[i];
    if (r.entry != entry || r.stride != stride || r.dil != p.dil || r.cl != p.cl ||
        r.pool_general != pgen || r.k != p.KH)
      continue;
    const double d = fabs(lm - log2(r.macs + 1.0)) + 0.5 * fabs(lc - log2((double)r.C)) +
                     0.5 * fabs(lco - log2((double)r.CO));
    if (best < 0 || d < bd) { best = i; bd = d; }
  }
  if (best < 0) return rule_variant(p);
  const VariantRow &r = kVariantTable[best];
  // candidates: (FFMA), (TF32, loads), (TF32, tensor copies), (F16, loads), (F16, copies)
  const int cv[kTableCols] = {FC_VARIANT_FFMA, FC_VARIANT_TC_TF32X3, FC_VARIANT_TC_TF32X3,
                              FC_VARIANT_TC_F16X3, FC_VARIANT_TC_F16X3};
  const int cs[kTableCols] = {1, 0, 1, 0, 1};
  int pick = -1;
  for (int i = 0; i < kTableCols; ++i) {
    if (r.ms[i] < 0.f) continue;  // refused when measured
    ConvProblem q = p;
    q.staging = cs[i];
    if (!variant_supported(q, cv[i])) continue;
    if (pick < 0 || r.ms[i] < r.ms[pick]) pick = i;
  }
  if (pick < 0) return rule_variant(p);
  *staging = cs[pick];
  return cv[pick];
}

fc_status run(ConvProblem &p, void *ws, size_t ws_bytes, void *stream) {
  t_last_launches = 0;
  unsigned int *st = nullptr;
  fc_status s = status_ptr(&st);
  if (s != FC_OK) return s;
  p.status = st;
  WsLayout L = ws_layout(p);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) != 0 || ws_bytes < L.total)
    return FC_ERR_WORKSPACE;
  int staging = 1;
  const int va = auto_choice(p, &staging);
  const int v = g_variant_override != FC_VARIANT_AUTO ? g_variant_override : va;
  if (g_variant_override != FC_VARIANT_AUTO && v != va) staging = 1;  // the override's own default
  p.staging = g_staging_override >= 0 ? g_staging_override : staging;
  if (!variant_supported(p, v)) return FC_ERR_UNSUPPORTED;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  int launches = 0;
  cudaError_t e;
  if (v == FC_VARIANT_FFMA) e = ffma_launch(p, ws, L, cs, &launches);
  else e = tc_launch(p, v == FC_VARIANT_TC_F16X3 ? 1 : 0, ws, L, cs, &launches);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FC_ERR_CUDA;
  }
  t_last_variant = v;
  t_last_launches = launches;
  t_last_staging = (v != FC_VARIANT_FFMA && tc_uses_tma(p, v == FC_VARIANT_TC_F16X3 ? 1 : 0)) ? 1 : 0;
  return FC_OK;
}

}  // namespace

void prof_begin(cudaStream_t s) {
  if (!g_prof_on || g_prof_n >= kMaxProf) return;
  if (g_prof_n >= g_prof_created) {
    if (cudaEventCreate(&g_prof_ev[g_prof_n][0]) != cudaSuccess) return;
    if (cudaEventCreate(&g_prof_ev[g_prof_n][1]) != cudaSuccess) {
      cudaEventDestroy(g_prof_ev[g_prof_n][0]);
      return;
    }
    g_prof_created = g_prof_n + 1;
  }
  if (cudaEventRecord(g_prof_ev[g_prof_n][0], s) == cudaSuccess) g_prof_open = true;
}

void prof_end(cudaStream_t s, int entry) {
  if (!g_prof_open) return;
  g_prof_open = false;
  if (cudaEventRecord(g_prof_ev[g_prof_n][1], s) != cudaSuccess) return;
  g_prof_entry[g_prof_n] = entry;
  ++g_prof_n;
}

WsLayout ws_layout(const ConvProblem &p) {
  WsLayout L{};
  const long Cp = (p.C + 7) / 8 * 8, COp = (p.CO + 63) / 64 * 64;
  const long taps = (long)p.KD * p.KH * p.KW;
  size_t off = 0;
  L.ffma_w = off;
  L.ffma_w_bytes = sizeof(float) * Cp * taps * COp;
  off = align256(off + L.ffma_w_bytes);
  L.tc_w = off;
  L.tc_w_bytes = tc_weight_bytes(p);
  off = align256(off + L.tc_w_bytes);
  L.partial = off;
  if (p.pool) {
    long T = ffma_pool_tiles_per_image(p);
    long T2 = tc_pool_tiles_per_image(p);
    if (T2 > T) T = T2;
    L.partial_bytes = sizeof(float) * (size_t)p.N * T * p.CO;
  }
  off = align256(off + L.partial_bytes);
  L.wmax = off;
  L.wmax_bytes = sizeof(float) * kMaxPackBlocks;
  off = align256(off + L.wmax_bytes);
  L.total = off;
  return L;
}

}  // namespace fc

using namespace fc;

// ---------------------------------------------------------------------------
// Workspace for fc_conv2d_epi_noalloc.  Some callers cannot allocate device
// memory at all: code running inside a host-side callback or a custom
// allocator hook, real-time or safety-certified paths that forbid allocation
// after start-up, and plug-in hosts that own the device memory pool.  For
// them the library keeps this fixed array in device memory; it exists on
// every GPU that loads the library, until the process exits.
static constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB
static __device__ __align__(256) unsigned char fc_noalloc_scratch[kNoAllocScratchBytes];
// In host code `fc_noalloc_scratch` names a host-side stand-in, not device
// memory: kernels must get the address cudaGetSymbolAddress returns, looked
// up once per device (with that device current) and cached here.
static unsigned char *g_noalloc_ptr[64];

static fc_status noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FC_ERR_CUDA;
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, fc_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FC_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = static_cast<unsigned char *>(p);
  }
  *out = g_noalloc_ptr[dev];
  return FC_OK;
}

extern "C" {

fc_status fc_conv2d_epi_noalloc(const float *x, int N, int C_in, int H, int W,
                                const float *w, int C_out, int kH, int kW, int stride,
                                int pad, int dilation, const fc_epilogue *epi, float *y,
                                void *stream) {
  // The shapes' workspace must fit the fixed array; anything larger is
  // refused before touching the device.
  const int dims[7] = {N, C_in, H, W, C_out, kH, pad};
  if (kH == kW && N >= 0 && C_in >= 1 && C_out >= 1 && H >= 1 && W >= 1 && pad >= 0) {
    const size_t need = fc_workspace_bytes(0, dims);
    if (need > kNoAllocScratchBytes) return FC_ERR_WORKSPACE;
  }
  void *scratch = nullptr;
  const fc_status s = noalloc_scratch(&scratch);
  if (s != FC_OK) return s;
  // The packed weights are rewritten in the array by every call before use,
  // so nothing in it has to start at zero.
  return fc_conv2d_epi(x, N, C_in, H, W, w, C_out, kH, kW, stride, pad, dilation, epi, y,
                       scratch, kNoAllocScratchBytes, stream);
}

// Layer parameters the entry points accept (every variant that supports a
// shape computes the same values; the fixed-size kernels take kernel size 3,
// stride and dilation 1 or 2, the general CUDA-core kernel the rest).
static constexpr int kMaxK = 7, kMaxStride = 4, kMaxDil = 4, kMaxPad = 64;

// Elements per image must stay below 2^31 (per-image offsets are 32-bit in
// places); whole tensors may be larger (64-bit offsets).
static bool image_fits(long long v) { return v >= 0 && v < (1LL << 31); }

// Validates a conv2d / conv3d call and fills the problem.  `check_ptrs`:
// also the pointers (a real call, not a query).
static fc_status conv_problem(const float *x, int N, int C_in, int D, int H, int W, const float *w,
                       int C_out, int kD, int kH, int kW, int stride, int pad, int dilation,
                       const fc_epilogue *epi, float *y, int cl, int d3, bool check_ptrs,
                       ConvProblem *out) {
  if (N < 0 || C_in < 1 || C_out < 1 || D < 1 || H < 1 || W < 1 || kD < 1 || kH < 1 ||
      kW < 1 || stride < 1 || pad < 0 || dilation < 1)
    return FC_ERR_INVALID_ARG;
  if (stride > kMaxStride || dilation > kMaxDil || kD > kMaxK || kH > kMaxK || kW > kMaxK ||
      pad > kMaxPad)
    return FC_ERR_UNSUPPORTED;
  const int pd = d3 ? pad : 0;
  const int spanD = dilation * (kD - 1) + 1, spanH = dilation * (kH - 1) + 1,
            spanW = dilation * (kW - 1) + 1;
  if (D + 2 * pd < spanD || H + 2 * pad < spanH || W + 2 * pad < spanW) return FC_ERR_INVALID_ARG;
  const int Do = (D + 2 * pd - spanD) / stride + 1, Ho = (H + 2 * pad - spanH) / stride + 1,
            Wo = (W + 2 * pad - spanW) / stride + 1;
  if (Do < 1 || Ho < 1 || Wo < 1) return FC_ERR_INVALID_ARG;
  if (!image_fits((long long)C_in * D * H * W) || !image_fits((long long)C_out * Do * Ho * Wo) ||
      !image_fits((long long)C_out * C_in * kD * kH * kW))
    return FC_ERR_UNSUPPORTED;
  ConvProblem &p = *out;
  p = ConvProblem{};
  fc_status s = decode_eltwise(epi, &p.epi, &p.chain);
  if (s != FC_OK) return s;
  if (check_ptrs && N > 0) {
    if (!x || !w || !y) return FC_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return FC_ERR_ALIGNMENT;
  }
  p.x = x; p.w = w; p.y = y;
  p.N = N; p.C = C_in; p.D = D; p.H = H; p.W = W;
  p.CO = C_out; p.KD = kD; p.KH = kH; p.KW = kW;
  p.pad_d = pd; p.pad = pad;
  p.stride = stride;
  p.dil = dilation;
  p.cl = cl;
  p.Do = Do; p.Ho = Ho; p.Wo = Wo;
  p.wlayout = 0;
  p.entry = d3 ? 1 : 0;
  p.tstride = 1;
  // the tensor-core kernel takes square odd kernels up to 7 (3D: cubic up
  // to 5) at stride / dilation <= 2; the rest only the general CUDA-core one
  p.gen = !(kH == kW && (kH & 1) && (d3 ? (kD == kH && kD <= 5) : kD == 1) && stride <= 2 &&
            dilation <= 2);
  return FC_OK;
}

static fc_status conv2d_impl(const float *x, int N, int C_in, int H, int W, const float *w,
                             int C_out, int kH, int kW, int stride, int pad, int dilation,
                             const fc_epilogue *epi, float *y, void *ws, size_t ws_bytes,
                             void *stream, int cl) {
  ConvProblem p;
  const fc_status s = conv_problem(x, N, C_in, 1, H, W, w, C_out, 1, kH, kW, stride, pad,
                                   dilation, epi, y, cl, 0, true, &p);
  if (s != FC_OK) return s;
  if (N == 0) return FC_OK;
  return run(p, ws, ws_bytes, stream);
}

fc_status fc_conv2d_epi(const float *x, int N, int C_in, int H, int W, const float *w, int C_out,
                        int kH, int kW, int stride, int pad, int dilation, const fc_epilogue *epi,
                        float *y, void *ws, size_t ws_bytes, void *stream) {
  return conv2d_impl(x, N, C_in, H, W, w, C_out, kH, kW, stride, pad, dilation, epi, y, ws,
                     ws_bytes, stream, 0);
}

fc_status fc_conv2d_epi_nhwc(const float *x, int N, int C_in, int H, int W, const float *w,
                             int C_out, int kH, int kW, int stride, int pad, int dilation,
                             const fc_epilogue *epi, float *y, void *ws, size_t ws_bytes,
                             void *stream) {
  return conv2d_impl(x, N, C_in, H, W, w, C_out, kH, kW, stride, pad, dilation, epi, y, ws,
                     ws_bytes, stream, 1);
}

static fc_status conv3d_impl(const float *x, int N, int C_in, int D, int H, int W,
                             const float *w, int C_out, int kD, int kH, int kW, int stride,
                             int pad, int dilation, const fc_epilogue *epi, float *y, void *ws,
                             size_t ws_bytes, void *stream, int cl) {
  ConvProblem p;
  const fc_status s = conv_problem(x, N, C_in, D, H, W, w, C_out, kD, kH, kW, stride, pad,
                                   dilation, epi, y, cl, 1, true, &p);
  if (s != FC_OK) return s;
  if (N == 0) return FC_OK;
  return run(p, ws, ws_bytes, stream);
}

fc_status fc_conv3d_epi(const float *x, int N, int C_in, int D, int H, int W, const float *w,
                        int C_out, int kD, int kH, int kW, int stride, int pad, int dilation,
                        const fc_epilogue *epi, float *y, void *ws, size_t ws_bytes,
                        void *stream) {
  return conv3d_impl(x, N, C_in, D, H, W, w, C_out, kD, kH, kW, stride, pad, dilation, epi, y,
                     ws, ws_bytes, stream, 0);
}

fc_status fc_conv3d_epi_ndhwc(const float *x, int N, int C_in, int D, int H, int W,
                              const float *w, int C_out, int kD, int kH, int kW, int stride,
                              int pad, int dilation, const fc_epilogue *epi, float *y, void *ws,
                              size_t ws_bytes, void *stream) {
  return conv3d_impl(x, N, C_in, D, H, W, w, C_out, kD, kH, kW, stride, pad, dilation, epi, y,
                     ws, ws_bytes, stream, 1);
}

static fc_status convT_problem(const float *x, int N, int C_in, int H, int W, const float *w,
                        int C_out, int k, int stride, int pad, int out_pad, const fc_epilogue *epi,
                        float *y, bool check_ptrs, ConvProblem *out) {
  if (N < 0 || C_in < 1 || C_out < 1 || H < 1 || W < 1 || k < 1 || stride < 1 || pad < 0 ||
      out_pad < 0)
    return FC_ERR_INVALID_ARG;
  // output padding below the stride (it selects among the output sizes a
  // stride > 1 allows)
  if (out_pad >= stride) return FC_ERR_INVALID_ARG;
  if (k > kMaxK || stride > kMaxStride || pad > kMaxPad) return FC_ERR_UNSUPPORTED;
  // transposed-conv output extent (H-1)*s - 2p + k + op
  const long long Hl = (long long)(H - 1) * stride - 2LL * pad + k + out_pad;
  const long long Wl = (long long)(W - 1) * stride - 2LL * pad + k + out_pad;
  if (Hl < 1 || Wl < 1) return FC_ERR_INVALID_ARG;
  if (!image_fits((long long)C_in * H * W) || !image_fits(Hl * Wl) ||
      !image_fits((long long)C_out * C_in * k * k))
    return FC_ERR_UNSUPPORTED;
  const int Ho = (int)Hl, Wo = (int)Wl;
  ConvProblem &p = *out;
  p = ConvProblem{};
  float lo = 0.f, hi = 0.f;
  int pk = 2, ps = 2;
  fc_status s = decode_pool(epi, &p.epi, &lo, &hi, &pk, &ps);
  if (s != FC_OK) return s;
  if (Ho < pk || Wo < pk) return FC_ERR_INVALID_ARG;  // no full pooling window
  if (check_ptrs && N > 0) {
    if (!x || !w || !y) return FC_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return FC_ERR_ALIGNMENT;
  }
  p.pk = pk;
  p.ps = ps;
  p.x = x; p.w = w; p.y = y;
  p.N = N; p.C = C_in; p.D = 1; p.H = H; p.W = W;
  p.CO = C_out; p.KD = 1; p.KH = k; p.KW = k;
  p.tstride = stride; p.tpad = pad; p.top = out_pad;
  p.pad_d = 0;
  p.stride = 1;
  p.dil = 1;
  p.Do = 1; p.Ho = Ho; p.Wo = Wo;
  p.wlayout = 1;
  p.pool = 1;
  p.ht_lo = lo; p.ht_hi = hi;
  p.chain = CHAIN_NONE;
  p.entry = 2;
  if (stride == 1 && pad <= k - 1) {
    // the equivalent conv: swapped + flipped weights, padding k - 1 - p
    p.pad = k - 1 - pad;
    p.gen = (k & 1) == 0;  // the tensor-core kernel takes odd kernel sizes
  } else if (stride == 2 && k == 3 && pad == 1 && pk == 2 && ps == 2) {
    // per output parity class on the input grid (tensor cores); the
    // general CUDA-core kernel for the CUDA-core variant
    p.pad = 0;
    p.subpix = 1;
  } else {
    p.gen = 1;
  }
  return FC_OK;
}

fc_status fc_convT2d_pool_mean(const float *x, int N, int C_in, int H, int W,
                               const float *w, int C_out, int k, int stride,
                               int pad, int out_pad, const fc_epilogue *epi,
                               float *y, void *ws, size_t ws_bytes,
                               void *stream) {
  ConvProblem p;
  const fc_status s = convT_problem(x, N, C_in, H, W, w, C_out, k, stride, pad, out_pad, epi, y,
                                    true, &p);
  if (s != FC_OK) return s;
  if (N == 0) return FC_OK;
  return run(p, ws, ws_bytes, stream);
}

fc_status fc_pool_mean_tail(const float *x, int N, int C, int H, int W, int k, int s,
                            float ht_lo, float ht_hi, float *y, void *stream) {
  if (N < 0 || C < 1 || H < 1 || W < 1 || k < 1 || s < 1 || k > H || k > W ||
      !(ht_lo <= ht_hi))
    return FC_ERR_INVALID_ARG;
  if (!fits_int32((long long)N * C) || !fits_int32((long long)H * W)) return FC_ERR_UNSUPPORTED;
  t_last_variant = 0;
  t_last_launches = 0;
  if (N == 0) return FC_OK;
  if (!x || !y) return FC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) % 4) || (reinterpret_cast<uintptr_t>(y) % 4))
    return FC_ERR_ALIGNMENT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FC_ERR_CUDA;
  int launches = 0;
  if (tail_launch(x, (long)N * C, H, W, k, s, ht_lo, ht_hi, y,
                  static_cast<cudaStream_t>(stream), &launches) != cudaSuccess)
    return FC_ERR_CUDA;
  t_last_launches = launches;
  return FC_OK;
}

// An epilogue holding the pooled entry's chain for a window / stride.
static fc_epilogue pool_chain(int pk, int ps) {
  fc_epilogue e;
  memset(&e, 0, sizeof(e));
  e.n_ops = 4;
  if (pk == 2 && ps == 2) {
    e.ops[0].kind = FC_EPI_MAXPOOL2X2;
  } else {
    e.ops[0].kind = FC_EPI_MAXPOOL;
    e.ops[0].a = (float)pk;
    e.ops[0].b = (float)ps;
  }
  e.ops[1].kind = FC_EPI_HARDTANH;
  e.ops[1].a = -1.0f;
  e.ops[1].b = 1.0f;
  e.ops[2].kind = FC_EPI_MEAN_HW;
  e.ops[3].kind = FC_EPI_TANH;
  return e;
}

size_t fc_workspace_bytes(int entry, const int *d) {
  if (!d) return 0;
  ConvProblem p;
  switch (entry) {
    case 0:  // {N, C_in, H, W, C_out, k, pad}: independent of stride and dilation
      if (conv_problem(nullptr, d[0], d[1], 1, d[2], d[3], nullptr, d[4], 1, d[5], d[5], 1, d[6],
                       1, nullptr, nullptr, 0, 0, false, &p) != FC_OK)
        return 0;
      return ws_layout(p).total;
    case 1:  // {N, C_in, D, H, W, C_out, k, pad}
      if (conv_problem(nullptr, d[0], d[1], d[2], d[3], d[4], nullptr, d[5], d[6], d[6], d[6], 1,
                       d[7], 1, nullptr, nullptr, 0, 1, false, &p) != FC_OK)
        return 0;
      return ws_layout(p).total;
    case 2: {  // {N, C_in, H, W, C_out, k, pad}, 2x2 pool: covers every stride / output padding
      const fc_epilogue e = pool_chain(2, 2);
      size_t total = 0;
      for (int st = 1; st <= kMaxStride; ++st)
        for (int op = 0; op < st; ++op)
          if (convT_problem(nullptr, d[0], d[1], d[2], d[3], nullptr, d[4], d[5], st, d[6], op,
                            &e, nullptr, false, &p) == FC_OK) {
            const size_t t = ws_layout(p).total;
            if (t > total) total = t;
          }
      return total;
    }
    case 3: {  // {N, C_in, H, W, C_out, k, pad, stride, out_pad, pool k, pool s}
      if (d[9] < 1 || d[10] < 1 || d[9] > 4 || d[10] > 4) return 0;
      const fc_epilogue e = pool_chain(d[9], d[10]);
      if (convT_problem(nullptr, d[0], d[1], d[2], d[3], nullptr, d[4], d[5], d[7], d[6], d[8], &e,
                        nullptr, false, &p) != FC_OK)
        return 0;
      return ws_layout(p).total;
    }
    default:
      return 0;
  }
}

int fc_select_variant(int entry, const int *d) {
  if (!d) return -1;
  ConvProblem p;
  fc_status s;
  switch (entry) {
    case 0:
    case 4:  // {N, C_in, H, W, C_out, k, stride, pad, dilation}
      s = conv_problem(nullptr, d[0], d[1], 1, d[2], d[3], nullptr, d[4], 1, d[5], d[5], d[6],
                       d[7], d[8], nullptr, nullptr, entry == 4, 0, false, &p);
      break;
    case 1:
    case 5:  // {N, C_in, D, H, W, C_out, k, stride, pad, dilation}
      s = conv_problem(nullptr, d[0], d[1], d[2], d[3], d[4], nullptr, d[5], d[6], d[6], d[6],
                       d[7], d[8], d[9], nullptr, nullptr, entry == 5, 1, false, &p);
      break;
    case 2: {  // {N, C_in, H, W, C_out, k, stride, pad, out_pad, pool k, pool s}
      if (d[9] < 1 || d[10] < 1 || d[9] > 4 || d[10] > 4) return -1;
      const fc_epilogue e = pool_chain(d[9], d[10]);
      s = convT_problem(nullptr, d[0], d[1], d[2], d[3], nullptr, d[4], d[5], d[6], d[7], d[8], &e,
                        nullptr, false, &p);
      break;
    }
    default:
      return -1;
  }
  if (s != FC_OK) return -1;
  int staging = 1;
  const int va = auto_choice(p, &staging);
  const int v = g_variant_override != FC_VARIANT_AUTO ? g_variant_override : va;
  p.staging = g_staging_override >= 0 ? g_staging_override : staging;
  return variant_supported(p, v) ? v : -1;
}

fc_status fc_set_variant(int v) {
  if (v < FC_VARIANT_AUTO || v > FC_VARIANT_TC_F16X3) return FC_ERR_INVALID_ARG;
  g_variant_override = v;
  return FC_OK;
}

fc_status fc_set_staging(int mode) {
  if (mode < -1 || mode > 1) return FC_ERR_INVALID_ARG;
  g_staging_override = mode;
  return FC_OK;
}

int fc_last_staging(void) { return t_last_staging; }

int fc_last_variant(void) { return t_last_variant; }

int fc_last_launch_count(void) { return t_last_launches; }

const char *fc_status_string(fc_status s) {
  switch (s) {
    case FC_OK: return "FC_OK";
    case FC_ERR_INVALID_ARG: return "FC_ERR_INVALID_ARG: invalid argument";
    case FC_ERR_UNSUPPORTED: return "FC_ERR_UNSUPPORTED: parameters or epilogue chain not supported";
    case FC_ERR_ALIGNMENT: return "FC_ERR_ALIGNMENT: pointer not 16-byte aligned";
    case FC_ERR_WORKSPACE: return "FC_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case FC_ERR_CUDA: return "FC_ERR_CUDA: CUDA runtime or launch failure";
    case FC_ERR_TIMEOUT: return "FC_ERR_TIMEOUT: a kernel's bounded wait ran out";
    case FC_ERR_RANGE: return "FC_ERR_RANGE: input beyond the fp16-split range";
    default: return "unknown fc_status";
  }
}

fc_status fc_get_last_device_error(void *stream) {
  unsigned int *st = nullptr;
  fc_status s = status_ptr(&st);
  if (s != FC_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(cs) != cudaSuccess) return FC_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, st, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FC_ERR_CUDA;
  if (word) {
    unsigned int zero = 0;
    if (cudaMemcpy(st, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return FC_ERR_CUDA;
  }
  if (word & ST_PLAN) return FC_ERR_CUDA;
  if (word & ST_TIMEOUT) return FC_ERR_TIMEOUT;
  if (word & ST_RANGE) return FC_ERR_RANGE;
  return FC_OK;
}

int fc_version(void) { return 100; }

fc_status fc_selftest_wait_timeout(unsigned int limit_us, void *stream) {
  if (limit_us < 1 || limit_us > 1000000) return FC_ERR_INVALID_ARG;
  unsigned int *st = nullptr;
  fc_status s = status_ptr(&st);
  if (s != FC_OK) return s;
  if (selftest_wait_launch(st, (uint64_t)limit_us * 1000ull, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return FC_ERR_CUDA;
  return FC_OK;
}

int fc_wait_report(void *stream, unsigned int *out, int max_words) {
  unsigned int *st = nullptr;
  if (status_ptr(&st) != FC_OK || !out || max_words < 1) return -1;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return -1;
  unsigned int buf[kStatusWords];
  if (cudaMemcpy(buf, st, sizeof(buf), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  const int n = (int)(buf[1] < 32u ? buf[1] : 32u);
  const int words = 1 + 8 * n;
  for (int i = 0; i < words && i < max_words; ++i) out[i] = buf[1 + i];
  if (buf[1]) {
    unsigned int zero[kStatusWords - 1] = {0};
    if (cudaMemcpy(st + 1, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return -1;
  }
  return (int)buf[1];
}

fc_status fc_profile_enable(int on) {
  g_prof_on = on != 0;
  return FC_OK;
}

fc_status fc_profile_read(int entry, double *total_ms, int *launches) {
  if (!total_ms || !launches) return FC_ERR_INVALID_ARG;
  double tot = 0.0;
  int cnt = 0;
  for (int i = 0; i < g_prof_n; ++i) {
    if (g_prof_entry[i] != entry) continue;
    if (cudaEventSynchronize(g_prof_ev[i][1]) != cudaSuccess) return FC_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_prof_ev[i][0], g_prof_ev[i][1]) != cudaSuccess)
      return FC_ERR_CUDA;
    tot += ms;
    ++cnt;
  }
  *total_ms = tot;
  *launches = cnt;
  return FC_OK;
}

void fc_profile_reset(void) {
  g_prof_n = 0;
  g_prof_open = false;
}

}  // extern "C"
