// fc_tc.cu -- tcgen05 tensor-core path: implicit-GEMM convolution with the
// epilogue fused, persistent and warp-specialised, for sm_103a.
//
// GEMM view (the implicit-GEMM reading of the Kimi-K2.6__l2_p57 and
// Kimi-K2.6__l2_p90 traces, GEMM-shape paragraphs):
//   M = output pixels (128 per MMA, one TMEM lane each), N = output channels
//   (64), K = C_in x taps.
// fp32 accuracy from 11-bit-significand tensor formats: every operand v is
// split into v_hi (rounded to the tensor format) and a remainder v_lo; the
// sum x_hi w_hi + x_hi w_lo + x_lo w_hi is exact up to the x_lo w_lo term
// (~2^-22 relative).  The B operand is stored as [W_hi | W_lo] (N = 128), so
// the three products take two MMAs per K step:
//   D[:, 0:128]  += A_hi * [W_hi | W_lo]     (N = 128)
//   D[:, 64:128] += A_lo * W_hi              (N = 64)
//   y = D[:, c] + scale * D[:, 64 + c]
// tf32 mode (kind::tf32): scale 1.  f16 mode (kind::f16, twice the rate):
// the remainders are stored multiplied by 2^11 so they stay normal in fp16,
// and scale = 2^-11; |x|, |w| must stay within 65504 (checked, status bit).
//
// Operand layout (no swizzle, K-major): a "slice" is 16 bytes per row (4
// tf32 or 8 fp16 values of consecutive input channels).  Staged input
// pixels sit 16 bytes apart in each slice plane, in the same raster order
// (rows RS pixels apart) as the M tile's output pixels, so the A operand of
// tap (kd, kh, kw) is the stage shifted by ((kd*RIN + kh)*RS + kw) pixels:
// a different descriptor start address, no data movement per tap.  This is
// the GB300 form of the traces' shared-memory halo tile.
//
// Roles (512 threads): warps 0-7 epilogue (warp w: TMEM lanes 32(w%4)..+31,
// channels 32(w/4)..+31), warp 8
// TMEM allocation + MMA issue (the warp runs converged; each burst of MMAs
// and each commit is issued by the lane elect.sync picks, the same lowest
// lane every time), warps 9-15 producers (one staged input row per warp
// pass, lanes across its pixels: global loads, hi/lo split, st.shared into
// the stage ring; one producer lane also streams packed weights with bulk
// copies).  All waits are
// bounded (4 s on %globaltimer) and warp-uniform; a timeout sets a status
// bit, every role drains, and the CTA frees its tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#include "fc_epi.cuh"
#include "fc_internal.h"
#include "fc_tc_ptx.cuh"

namespace fc {

namespace {

constexpr int kThreads = 512;
// Warp roles of the 16 warps: kEpi epilogue warps (two per TMEM lane
// quadrant, 32 channels each; with FEW_EPI one per quadrant taking all 64
// channels -- the 2x2-pooled entry, whose epilogue is light and whose
// stages want more loading warps), one MMA warp, the rest producers.
template <bool FEW_EPI>
struct Roles {
  static constexpr int kEpi = FEW_EPI ? 4 : 8;
  static constexpr int kMma = kEpi;
  static constexpr int kProd0 = kEpi + 1;
  static constexpr int kProd = 16 - kProd0;
  static constexpr int kProdT = 32 * kProd;
};
constexpr int kBStep = 4096;                  // one K step of B: 2 slices x 128 rows x 16 B
constexpr int kMaxSmem = 227 * 1024 - 1024;   // minus the 1 KB alignment slack
constexpr uint64_t kWaitNs = 4000000000ull;
constexpr uint32_t kSleepHintNs = 20000;  // hardware sleep per poll while waiting
constexpr float kF16SplitMin = 1.0f / 4096.0f;  // 2^-12: smallest data maximum of the fp16 split
constexpr unsigned int kWaitRecords = 32;  // diagnostic records kept after the status word
// Kernel sizes the tensor-core plans take: odd, up to 7 x 7 in 2-D and
// 5 x 5 x 5 in 3-D (125 taps); K-step tables hold kMaxTaps + 2 entries.
constexpr int kMaxTaps = 126;

// Division of 0 <= n < 2^31 by a divisor fixed at plan time, as a
// multiply-high, add and shift (the round-up method of Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994):
// with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (umulhi(m, n) + n) >> l.
struct FastDiv {
  uint32_t d, m, l;
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  f.l = 0;
  while ((1ull << f.l) < d) ++f.l;
  f.m = (uint32_t)(((1ull << 32) * ((1ull << f.l) - d)) / d + 1);
  return f;
}

__host__ __device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
#ifdef __CUDA_ARCH__
  const uint32_t hi = __umulhi(n, f.m);
#else
  const uint32_t hi = (uint32_t)(((uint64_t)n * f.m) >> 32);
#endif
  return (hi + n) >> f.l;
}

struct TcPlan {
  int ok;
  int prec;       // 0 tf32, 1 f16
  int E;          // values per 16-byte slice
  int chunk_ci;   // input channels per stage
  int P;          // slice planes per stage
  int NCH;        // stages per unit (chunks of C_in)
  int KS;         // K steps per chunk
  int TAPS;
  int KH, KW;     // kernel rows / columns (odd; 3-D kernels are KH x KH x KH)
  int pairtaps;   // f16 with one plane per chunk: a K step spans two taps
  int U, R, RS, WT, RIN;
  // Staging geometry.  RS is the pitch (pixels) between the M tile's output
  // rows in a staged plane; RIN the input rows loaded per depth slice; LW
  // the input pixels loaded per row; DSL the staged pixels per depth slice.
  // Stride 2 (S2) stages each input slice deinterleaved into four
  // sub-planes (even/odd rows x even/odd columns) of SR x RS pixels (SUB
  // each), so that tap (kh, kw) at input offset (a, b) = (kh, kw) * DIL
  // reads sub-plane (a & 1, b & 1) at a shift of (a >> 1, b >> 1) -- again
  // one shifted descriptor start per tap.  DIL is the dilation.
  int S2, DIL, LW, SR, SUB, DSL;
  uint8_t perm[kMaxTaps + 2];  // K order of the taps (paired taps: increasing shifts)
  // Stride-2 transposed conv by output parity class (SP): K step ks feeds
  // class kcls[ks] & 3 (accumulator (kcls & 3) x 128 columns); bit 7 marks
  // the class's first K step of a chunk.  skd[ks] is the step's A start |
  // slice distance << 16 (16-byte units), computed here on the host.
  int SP;
  uint8_t kcls[28];
  uint32_t skd[28];
  // SP with a unit's chunks and weights all resident (NCH <= S): the MMAs
  // of classes (0,0), (0,1) (half A, TMEM columns 0-255) run over every
  // chunk before those of (1,0), (1,1) (half B, 256-511), each half with its
  // own accumulator barriers, so the epilogue's work on one half overlaps
  // the MMAs of the other.  KA = the K steps of half A.
  int SPLIT, KA;
  int NPIX;
  int plane_bytes;
  int a_stage_bytes;
  int S;
  int COB;
  int b_chunk_bytes;
  int b_resident;
  int SB;
  // CTA pairs (2x2-pooled plans): a cluster of two CTAs, the even one
  // issuing M = 256 MMAs over both CTAs' tiles, each CTA holding half of B
  // (b_kstep = 3072 bytes a K step: 64 rows of [W_hi | W_lo], 32 of W_hi)
  int PAIR;
  int b_kstep;
  int NACC;
  int tmem_cols;
  int n_rt, n_ct;
  long units;
  FastDiv fd_ct, fd_rt, fd_do, fd_n, fd_cb;  // unit index -> position
  int smem_bytes;
  int off_b, off_bar, off_misc;
  // Tensor-copy staging (TMA, stride 1): one producer warp loads the raw
  // fp32 input of each (chunk, depth slice) -- RIN rows of LW pixels, all
  // chunk channels, zeros outside the tensor -- with one tiled tensor copy
  // into a ring of TR slots (raw_bytes each, raw_tx bytes per copy); the
  // other producer warps split it into the stage's hi / lo slices.
  // Channels-first slots are [chunk_ci][RIN][BW] (BW = LW + coff rounded up
  // to 4: the copy starts coff columns early so that its first column is
  // 16-byte aligned); channels-last slots [RIN][LW][chunk_ci].
  int TMA, TR, raw_bytes, raw_tx, off_raw, BW, coff;
  FastDiv fd_lw;
  FastDiv fd_rin;  // division by RIN (depth slice of a staged row)
  // Unit origin: input rows / columns advance by ROWSTEP / COLSTEP conv
  // outputs per unit row / column index (U R and WT, except for the general
  // max pool).  General max pool (GP, window pk, stride ps other than 2 / 2):
  // a unit is one pooled row -- U = pk conv rows, one tile each -- of PJ
  // pooled columns; the epilogue writes each lane's row maximum to XB bytes
  // of shared memory at off_xb and takes the windows there.
  int ROWSTEP, COLSTEP, GP, PJ, off_xb, XB;
};

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

constexpr int kMaxCoTc = 512;  // output channels the tensor-core path stages in smem
// General max pool: channel rows of the row-maxima buffer are 129 floats
// apart, so the 32 channels a warp reads at one column fall in 32 banks
// (at 128 they all fell in one: 51 M conflicted loads in a 3x3/2 pool of
// 16x64x256x256).
constexpr int kXbPitch = 129;

struct SmemCtl {
  uint32_t tmem_base;
  int abort;
  uint32_t amax_bits;  // largest |x| the producers staged (fp32 bits)
  uint32_t kdelta[kMaxTaps + 2];  // per K step: A start (16-byte units) | slice distance << 16
  uint32_t kcls[28];    // per K step (stride-2 transposed conv): class | first << 7
  alignas(16) float red[4][64];          // pool: per-warp partial sums
  alignas(16) float bias[kMaxCoTc];      // bias per output channel (0 without bias)
  alignas(16) float addend[kMaxCoTc];    // per-channel addend of the fused GELU chain
};
// The epilogue reads bias / addend as float4.
static_assert(offsetof(SmemCtl, bias) % 16 == 0 && offsetof(SmemCtl, addend) % 16 == 0,
              "16-byte aligned per-channel arrays");
static_assert(sizeof(SmemCtl) % 16 == 0, "SmemCtl size");

// Staged-pixel shift of tap t = (kd, kh, kw) from an M tile's first
// pixel, with input offsets a = kh * DIL, b = kw * DIL: stride 1
// kd*DSL + a*RS + b; stride 2 sub-plane (a & 1, b & 1) of depth slice kd,
// then (a >> 1) rows and (b >> 1) columns.  (Depth slice kd is staged input
// depth od*stride + kd*DIL - pad.)
__host__ __device__ __forceinline__ int tap_shift(int t, const TcPlan &q) {
  const int kd = t / (q.KH * q.KW), a = ((t / q.KW) % q.KH) * q.DIL, b = (t % q.KW) * q.DIL;
  if (!q.S2) return kd * q.DSL + a * q.RS + b;
  return kd * q.DSL + (2 * (a & 1) + (b & 1)) * q.SUB + (a >> 1) * q.RS + (b >> 1);
}


// Channel chunks and K steps of a plan.  They do not depend on the
// geometry, so neither does the weight image (nor the workspace): stride,
// dilation and the spatial extents change only the staging.
void plan_chunks(const ConvProblem &p, int prec, TcPlan &q) {
  q.prec = prec;
  q.E = prec ? 8 : 4;
  const int Cp8 = cdiv(p.C, 8) * 8;
  q.chunk_ci = (prec && Cp8 > 8) ? 16 : 8;
  const int Cp = cdiv(p.C, q.chunk_ci) * q.chunk_ci;
  q.P = q.chunk_ci / q.E;
  q.NCH = Cp / q.chunk_ci;
  q.KH = p.KH;
  q.KW = p.KW;
  q.TAPS = p.KD * p.KH * p.KW;
  q.pairtaps = (q.P == 1);
  q.KS = q.pairtaps ? cdiv(q.TAPS, 2) : q.TAPS;
  q.COB = cdiv(p.CO, 64);
  q.b_chunk_bytes = q.KS * kBStep;
}

// Plan with `U` M tiles per unit (pooling needs 2).
// Kernel shapes the tensor-core plans take: square, odd, 1..7 in 2-D and
// cubic, odd, 1..5 in 3-D.
bool tc_kernel_ok(const ConvProblem &p) {
  if (p.KH != p.KW || (p.KH & 1) == 0 || p.KH > 7) return false;
  if (p.KD > 1) return p.KD == p.KH && p.KD <= 5;
  return p.entry != 1 || p.KH == 1;
}

TcPlan make_plan_u(const ConvProblem &p, int prec, int U, bool allow_pair = true) {
  TcPlan q{};
  if (!tc_kernel_ok(p)) return q;
  if (p.stride > 2 || p.dil > 2 || ((p.stride > 1 || p.dil > 1) && p.pool)) return q;
  if (p.cl && (p.pool || p.stride != 1)) return q;  // channels-last: stride 1, no pool
  const bool gp = p.pool && (p.pk != 2 || p.ps != 2);
  // 2x2 pool: one row pair per unit; general pool: one tile per window row
  if (p.pool && U != (gp ? p.pk : 2)) return q;
  if (p.pool && p.KD != 1) return q;
  if (gp && (p.pk < 1 || p.pk > 4 || p.ps < 1 || p.ps > 4)) return q;
  plan_chunks(p, prec, q);
  q.GP = gp;
  q.S2 = p.stride == 2;
  q.DIL = p.dil;
  // staged columns past the tile's outputs: the last tap's column offset
  // (KW - 1) DIL (stride 2: half of it, in the half-width sub-planes)
  const int span = (p.KW - 1) * q.DIL, spanh = (p.KH - 1) * q.DIL;
  const int halo = q.S2 ? span / 2 : span;
  const bool rowpack = (p.Wo + halo <= 128);
  if (rowpack) {
    q.RS = p.Wo + halo;
    q.WT = p.Wo;
    q.n_ct = 1;
    q.R = p.pool ? 1 : 128 / q.RS;
  } else {
    q.RS = 128 + halo;
    q.WT = 128;
    q.n_ct = cdiv(p.Wo, 128);
    q.R = 1;
  }
  q.U = U;
  q.ROWSTEP = q.U * q.R;
  q.COLSTEP = q.WT;
  if (gp) {
    // pooled columns per tile: the windows wholly inside its WT columns
    const int Wp = (p.Wo - p.pk) / p.ps + 1;
    q.PJ = (q.WT - p.pk) / p.ps + 1;
    if (q.PJ > Wp) q.PJ = Wp;
    // strips advance by PJ ps columns: keep that a multiple of 4 so every
    // strip's first staged column stays 16-byte aligned for tensor copies
    if (q.PJ < Wp)
      while (q.PJ > 1 && (q.PJ * p.ps) % 4 != 0) --q.PJ;
    if (q.PJ < 1) return q;
    q.COLSTEP = q.PJ * p.ps;
    q.n_ct = cdiv(Wp, q.PJ);
    q.ROWSTEP = p.ps;
    q.XB = 64 * kXbPitch * 4;  // row maxima of 64 channels x 128 columns
  }
  if (!q.S2) {  // output rows u read input rows u + kh DIL: UR + (KH - 1) DIL rows
    q.RIN = q.U * q.R + spanh;
    q.LW = q.RS;
    q.DSL = q.RIN * q.RS;
  } else {  // output rows u read input rows 2u + kh DIL: 2UR - 1 + (KH - 1) DIL rows
    q.RIN = 2 * q.U * q.R - 1 + spanh;
    q.LW = 2 * q.RS;  // of 2 RS columns
    q.SR = q.U * q.R + spanh / 2;  // even input rows (odd rows: one fewer)
    q.SUB = q.SR * q.RS;
    q.DSL = 4 * q.SUB;
  }
  // K order of the taps: by increasing shift, so a K step's two paired taps
  // are one positive LBO apart (stride 1: the natural order)
  int shift[kMaxTaps];
  for (int t = 0; t < q.TAPS; ++t) {
    shift[t] = tap_shift(t, q);
    q.perm[t] = (uint8_t)t;
  }
  for (int i = 1; i < q.TAPS; ++i)  // insertion sort by shift
    for (int j = i; j > 0 && shift[q.perm[j]] < shift[q.perm[j - 1]]; --j) {
      const uint8_t tmp = q.perm[j];
      q.perm[j] = q.perm[j - 1];
      q.perm[j - 1] = tmp;
    }
  for (int t = q.TAPS; t < kMaxTaps + 2; ++t) q.perm[t] = 255;  // zero-weight padding slot
  // last staged pixel any MMA can touch: the largest tap shift (+1 for the
  // paired zero-weight slice), the last tile, 128 rows
  int maxshift = 0;
  for (int t = 0; t < q.TAPS; ++t) maxshift = shift[t] > maxshift ? shift[t] : maxshift;
  const int maxread = maxshift + 1 + (q.U - 1) * q.R * q.RS + 127;
  int npix = maxread + 1;
  if (npix < p.KD * q.DSL) npix = p.KD * q.DSL;
  q.NPIX = cdiv(npix, 8) * 8;
  q.plane_bytes = q.NPIX * 16;
  q.a_stage_bytes = 2 * q.P * q.plane_bytes;
  if (q.COB * 64 > kMaxCoTc) return q;
  q.n_rt = gp ? (p.Ho - p.pk) / p.ps + 1 : p.pool ? p.Ho / 2 : cdiv(p.Ho, q.U * q.R);
  q.units = (long)q.COB * p.N * p.Do * q.n_rt * q.n_ct;
  if (q.units >= (1L << 31)) return q;  // unit indices are 32-bit
  q.fd_ct = make_fastdiv((uint32_t)q.n_ct);
  q.fd_rt = make_fastdiv((uint32_t)q.n_rt);
  q.fd_do = make_fastdiv((uint32_t)p.Do);
  q.fd_n = make_fastdiv((uint32_t)p.N);
  q.fd_cb = make_fastdiv((uint32_t)((long)p.N * p.Do * q.n_rt * q.n_ct));
  q.NACC = q.U == 1 ? 4 : q.U == 2 ? 2 : 1;
  q.tmem_cols = q.U == 3 ? 512 : q.NACC * q.U * 128;  // allocations are powers of two
  if (q.tmem_cols > 512) return q;
  // shared memory: A stages + raw slots (tensor-copy staging) + B (resident
  // or a ring) + barriers/misc (+ the general pool's row maxima)
  const int misc = 512 + (int)sizeof(SmemCtl) + 256 + q.XB;
  q.b_kstep = kBStep;
  // 2x2 pool: CTA pairs when the units pair up, there are enough of them
  // to amortise the pair's start (its weight half loads completely before
  // the first MMA; measured: 16 x 64 x 64 x 64 0.033 -> 0.037 ms on pairs,
  // 128 x 64 x 128 x 128 (8192 units) 0.565 -> 0.561, 128 x 64 x 256 x 256
  // 1.24 -> 1.16) and the pair's smaller weight half stays resident beside
  // two or more stages
  if (allow_pair && p.pool && !gp && q.U == 2 && q.units >= 8192 && q.units % 2 == 0) {
    const long b_pair = (long)q.COB * q.NCH * q.KS * 3072;
    if (2L * q.a_stage_bytes + b_pair + misc <= kMaxSmem) {
      q.PAIR = 1;
      q.b_kstep = 3072;
      q.b_chunk_bytes = q.KS * 3072;
    }
  }
  const long b_all = (long)q.COB * q.NCH * q.b_chunk_bytes;
  // Tensor-copy staging needs 16-byte multiples for the tensor's strides
  // (channels-first: W % 4 == 0; channels-last: C_in % 4 == 0) and box
  // extents of at most 256.
  q.coff = p.cl ? 0 : (((-p.pad) % 4) + 4) % 4;
  q.BW = p.cl ? q.LW : (q.LW + q.coff + 3) / 4 * 4;
  // (channels-first: every unit's first column iw0 - coff a multiple of 4,
  // so the strips must advance by a multiple of 4 columns)
  const bool tma_ok = p.staging && !q.S2 && !p.pool && (p.cl ? (p.C % 4 == 0) : (p.W % 4 == 0)) &&
                      (p.cl || q.n_ct == 1 || q.COLSTEP % 4 == 0) && q.BW <= 256 &&
                      q.RIN <= 256;
  q.raw_tx = q.chunk_ci * q.RIN * q.BW * 4;
  q.raw_bytes = (q.raw_tx + 127) / 128 * 128;
  int S = 0, resident = 0, SB = 0, TR = 0;
  if (tma_ok) {  // at least two stages and two slots (a stage's depth slices + 1 in 3D)
    const int tr_min = p.KD > 1 ? p.KD + 1 : 2;
    for (int s = 4; s >= 2 && !S; --s)
      for (int tr = 4; tr >= tr_min && !S; --tr)
        if ((long)s * q.a_stage_bytes + (long)tr * q.raw_bytes + b_all + misc <= kMaxSmem) {
          S = s; TR = tr; resident = 1;
        }
  }
  for (int s = 4; s >= 2 && !S; --s)
    if ((long)s * q.a_stage_bytes + b_all + misc <= kMaxSmem) { S = s; resident = 1; }
  if (!S)
    for (int s = 4; s >= 1 && !S; --s)
      if ((long)s * q.a_stage_bytes + 2L * q.b_chunk_bytes + misc <= kMaxSmem) { S = s; SB = 2; }
  if (!S)
    for (int s = 2; s >= 1 && !S; --s)
      if ((long)s * q.a_stage_bytes + 1L * q.b_chunk_bytes + misc <= kMaxSmem) { S = s; SB = 1; }
  if (!S) return q;
  q.S = S;
  q.TMA = TR > 0;
  q.TR = TR;
  q.fd_lw = make_fastdiv((uint32_t)q.LW);
  q.fd_rin = make_fastdiv((uint32_t)q.RIN);
  q.b_resident = resident;
  q.SB = resident ? 1 : SB;
  q.off_raw = S * q.a_stage_bytes;  // 128-byte aligned (NPIX is a multiple of 8)
  q.off_b = q.off_raw + TR * q.raw_bytes;
  q.off_bar = q.off_b + (int)(resident ? b_all : (long)q.SB * q.b_chunk_bytes);
  q.off_misc = q.off_bar + 512;  // 16-byte aligned: off_b and the B region are
  q.off_xb = q.off_misc + (int)sizeof(SmemCtl);
  q.smem_bytes = q.off_bar + misc;
  if (q.smem_bytes < 120 * 1024) q.smem_bytes = 120 * 1024;  // one CTA per SM
  q.ok = 1;
  return q;
}

// Stride-2 transposed conv (k 3, pad 1) + pool by output parity class.
// Output (2i + a, 2j + b) of the transposed conv sums the taps (kh, kw)
// with a + 1 - kh and b + 1 - kw even, each reading input
// (i + (a + 1 - kh) / 2, j + (b + 1 - kw) / 2): class (0,0) has tap (1,1);
// (0,1) taps (1,2), (1,0); (1,0) taps (2,1), (0,1); (1,1) the four corners.
// The 2x2 pool window at (i, j) holds exactly the four classes at (i, j),
// so a unit is one M tile of pooled pixels (R rows of WT pooled columns on
// the input grid) with one accumulator per class, and the epilogue takes
// the max over the four accumulators lane by lane.  Staging is a stride-1
// input tile with a one-pixel halo (R + 1 rows, WT + 1 columns).
TcPlan make_plan_subpix(const ConvProblem &p, int prec) {
  TcPlan q{};
  if (!p.pool || p.KH != 3 || p.KW != 3 || p.KD != 1 || p.wlayout != 1) return q;
  if (p.pk != 2 || p.ps != 2) return q;
  plan_chunks(p, prec, q);
  q.SP = 1;
  q.DIL = 1;
  const int Hp = p.Ho / 2, Wp = p.Wo / 2;  // pooled extents
  const bool rowpack = Wp + 1 <= 128;
  if (rowpack) {
    q.RS = Wp + 1;
    q.WT = Wp;
    q.n_ct = 1;
    q.R = 128 / q.RS;
  } else {
    q.RS = 129;
    q.WT = 128;
    q.n_ct = cdiv(Wp, 128);
    q.R = 1;
  }
  q.U = 1;
  q.ROWSTEP = q.R;
  q.COLSTEP = q.WT;
  q.RIN = q.R + 1;
  q.fd_rin = make_fastdiv((uint32_t)q.RIN);
  q.LW = q.RS;
  q.DSL = q.RIN * q.RS;
  // K slots class by class, each class's taps by increasing shift; with
  // paired taps class (0,0) takes a zero-weight slot so no pair straddles
  // two classes.  10 (paired) or 9 slots.
  static const int kTaps[4][4] = {{4, -1, -1, -1}, {5, 3, -1, -1}, {7, 1, -1, -1}, {8, 6, 2, 0}};
  static const int kNTaps[4] = {1, 2, 2, 4};
  int slot = 0, shift[28];
  int slot_cls[28];
  for (int cls = 0; cls < 4; ++cls) {
    const int a = cls >> 1, b = cls & 1;
    for (int k = 0; k < kNTaps[cls]; ++k) {
      const int tap = kTaps[cls][k], kh = tap / 3, kw = tap % 3;
      q.perm[slot] = (uint8_t)tap;
      shift[slot] = ((a + 1 - kh) / 2) * q.RS + (b + 1 - kw) / 2;
      slot_cls[slot++] = cls;
    }
    if (q.pairtaps && (kNTaps[cls] & 1)) {
      q.perm[slot] = 255;
      shift[slot] = shift[slot - 1] + 1;  // any staged data: zero weights
      slot_cls[slot++] = cls;
    }
  }
  const int nslots = slot;
  if (q.KS != (q.pairtaps ? nslots / 2 : nslots)) return q;
  for (int t = nslots; t < kMaxTaps + 2; ++t) q.perm[t] = 255;
  int prev = -1;
  for (int ks = 0; ks < q.KS; ++ks) {
    const int s0 = q.pairtaps ? 2 * ks : ks;
    const int cls = slot_cls[s0];
    q.kcls[ks] = (uint8_t)(cls | (cls != prev ? 0x80 : 0));
    prev = cls;
    uint32_t lbo;
    if (q.pairtaps) {
      lbo = (uint32_t)(shift[s0 + 1] - shift[s0]);  // > 0 (increasing shifts)
    } else {
      lbo = 0;  // filled in below once the plane size is known
    }
    q.skd[ks] = (uint32_t)shift[s0] | (lbo << 16);
  }
  int maxshift = 0;
  for (int t = 0; t < nslots; ++t) maxshift = shift[t] > maxshift ? shift[t] : maxshift;
  int npix = maxshift + 1 + 127 + 1;
  if (npix < q.RIN * q.RS) npix = q.RIN * q.RS;
  q.NPIX = cdiv(npix, 8) * 8;
  q.plane_bytes = q.NPIX * 16;
  if (!q.pairtaps)
    for (int ks = 0; ks < q.KS; ++ks) q.skd[ks] |= (uint32_t)(q.plane_bytes >> 4) << 16;
  q.a_stage_bytes = 2 * q.P * q.plane_bytes;
  if (q.COB * 64 > kMaxCoTc) return q;
  q.n_rt = cdiv(Hp, q.R);
  q.units = (long)q.COB * p.N * q.n_rt * q.n_ct;
  if (q.units >= (1L << 31)) return q;
  q.fd_ct = make_fastdiv((uint32_t)q.n_ct);
  q.fd_rt = make_fastdiv((uint32_t)q.n_rt);
  q.fd_do = make_fastdiv(1u);
  q.fd_n = make_fastdiv((uint32_t)p.N);
  q.fd_cb = make_fastdiv((uint32_t)((long)p.N * q.n_rt * q.n_ct));
  q.NACC = 1;
  q.tmem_cols = 512;  // four class accumulators of 128 columns
  const int misc = 512 + (int)sizeof(SmemCtl) + 256;
  const long b_all = (long)q.COB * q.NCH * q.b_chunk_bytes;
  int S = 0, resident = 0, SB = 0;
  for (int s = 4; s >= 2 && !S; --s)
    if ((long)s * q.a_stage_bytes + b_all + misc <= kMaxSmem) { S = s; resident = 1; }
  if (!S)
    for (int s = 4; s >= 1 && !S; --s)
      if ((long)s * q.a_stage_bytes + 2L * q.b_chunk_bytes + misc <= kMaxSmem) { S = s; SB = 2; }
  if (!S)
    for (int s = 2; s >= 1 && !S; --s)
      if ((long)s * q.a_stage_bytes + 1L * q.b_chunk_bytes + misc <= kMaxSmem) { S = s; SB = 1; }
  if (!S) return q;
  q.S = S;
  q.b_resident = resident;
  q.SB = resident ? 1 : SB;
  q.off_raw = S * q.a_stage_bytes;
  q.off_b = S * q.a_stage_bytes;
  q.off_bar = q.off_b + (int)(resident ? b_all : (long)q.SB * q.b_chunk_bytes);
  q.off_misc = q.off_bar + 512;
  q.smem_bytes = q.off_bar + misc;
  if (q.smem_bytes < 120 * 1024) q.smem_bytes = 120 * 1024;
  q.KA = q.pairtaps ? 2 : 3;  // classes (0,0), (0,1): 1 + 2 taps
  q.SPLIT = (q.b_resident && q.NCH <= q.S) ? 1 : 0;
  q.ok = 1;
  return q;
}

// Pooling pairs two output rows per unit.  Without pooling a unit also
// takes two M tiles (half the barrier hand-offs per MMA, fewer re-staged
// halo rows) when the image has rows for both and shared memory still holds
// at least three stages; otherwise one.
TcPlan make_plan(const ConvProblem &p, int prec, bool allow_pair = true) {
  if (p.subpix) return make_plan_subpix(p, prec);
  // 2x2 pool: one row pair per unit.  (Two pairs, four tiles per K step,
  // issue faster but hold one accumulator and stream the weights: measured
  // 1.52 against 1.45 ms on the pooled workload.)
  if (p.pool) return make_plan_u(p, prec, (p.pk == 2 && p.ps == 2) ? 2 : p.pk, allow_pair);
  TcPlan q2 = make_plan_u(p, prec, 2);
  if (q2.ok && q2.S >= 3 && p.Ho > q2.R) return q2;
  TcPlan q1 = make_plan_u(p, prec, 1);
  return q1.ok ? q1 : q2;
}

// --------------------------------------------------------------- device


// Bounded wait on phase `parity` of `bar`.  On timeout: sets the status
// bit, records where it gave up (block, thread, barrier index, parity, the
// caller's tag and the raw barrier word) in the diagnostic area that
// follows the status word, raises the CTA's abort flag and returns false.
__device__ __noinline__ void record_timeout(unsigned int *status, const uint64_t *bar,
                                            int bar_idx, uint32_t parity, uint32_t tag) {
  if (!(tag & 0x08000000u)) atomicOr(status, ST_TIMEOUT);
  const unsigned int i = atomicAdd(status + 1, 1u);
  if (i < kWaitRecords) {
    unsigned int *r = status + 2 + i * 8;
    uint64_t word;
    asm volatile("ld.shared.b64 %0, [%1];" : "=l"(word) : "r"(ptx::smem_u32(bar)));
    r[0] = blockIdx.x;
    r[1] = threadIdx.x;
    r[2] = (unsigned)bar_idx;
    r[3] = parity;
    r[4] = tag;
    r[5] = (unsigned)word;
    r[6] = (unsigned)(word >> 32);
    r[7] = 0x5afeu;
  }
}

__device__ __forceinline__ bool wait_bar(uint64_t *bars, int idx, uint32_t parity,
                                         volatile int *abort, unsigned int *status,
                                         uint32_t tag, uint64_t limit_ns = kWaitNs) {
  uint64_t *bar = bars + idx;
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if ((i & 7u) == 0) {
      if (*abort) {
        record_timeout(status, bar, idx, parity, tag | 0x08000000u);
        return false;
      }
      if (ptx::globaltimer_ns() - t0 > limit_ns) {
        record_timeout(status, bar, idx, parity, tag);
        *abort = 1;
        return false;
      }
    }
  }
}

// Warp-uniform bounded wait.  Every lane tests the barrier once (a phase
// that has already completed costs one instruction and a vote); otherwise
// lane 0 polls and the verdict is broadcast, so a warp never splits around
// .sync.aligned instructions or named barriers.
__device__ __forceinline__ bool wait_bar_warp(uint64_t *bars, int idx, uint32_t parity,
                                              volatile int *abort, unsigned int *status,
                                              uint32_t tag, uint64_t limit_ns = kWaitNs) {
  if (__all_sync(0xffffffffu, ptx::mbar_test_wait(bars + idx, parity))) return true;
  int ok = 1;
  if ((threadIdx.x & 31) == 0)
    ok = wait_bar(bars, idx, parity, abort, status, tag, limit_ns) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Weight-ring slot of chunk g.
__device__ __forceinline__ int psb_tma_slot(uint32_t g, int SB) { return (int)(g % (uint32_t)SB); }

// AND of a predicate over the NT epilogue threads (named barrier 1).
template <int NT>
__device__ __forceinline__ bool epi_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(NT)
      : "memory");
  return r != 0;
}

template <int NT>
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory"); }

struct UnitPos {
  int cb, n, od, rt, ct;
};

__device__ __forceinline__ UnitPos decode_unit(long unit, const TcPlan &q) {
  UnitPos r;
  uint32_t u = (uint32_t)unit, t;
  t = fdiv(u, q.fd_ct); r.ct = (int)(u - t * q.fd_ct.d); u = t;
  t = fdiv(u, q.fd_rt); r.rt = (int)(u - t * q.fd_rt.d); u = t;
  t = fdiv(u, q.fd_do); r.od = (int)(u - t * q.fd_do.d); u = t;
  t = fdiv(u, q.fd_n); r.n = (int)(u - t * q.fd_n.d); r.cb = (int)t;
  return r;
}

__device__ __forceinline__ uint32_t tf32_rna(float v) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ bool f16_out_of_range(float v) {
  return !(fabsf(v) <= 65504.0f) && v == v;  // NaN propagates, not flagged
}

// Packs the B image: for each (channel block, chunk, K step) a 4 KB block
// of 2 slices x 128 rows x 16 bytes; rows 0-63 hold W_hi of the block's
// output channels, rows 64-127 W_lo (zero rows past C_out).
__global__ void tc_pack_weights(ConvProblem p, TcPlan q, uint8_t *__restrict__ out) {
  const long nelem = (long)q.COB * q.NCH * q.KS * 2 * 128 * q.E;
  float wmx = 0.0f;  // largest |w| this thread packs (fp16 split: range check)
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < nelem;
       i += (long)gridDim.x * blockDim.x) {
    const int e = (int)(i % q.E);
    long t = i / q.E;
    const int row = (int)(t % 128); t /= 128;
    const int k = (int)(t % 2); t /= 2;
    const int ks = (int)(t % q.KS); t /= q.KS;
    const int c = (int)(t % q.NCH);
    const int cb = (int)(t / q.NCH);
    int tap, ci;
    if (q.pairtaps) {
      tap = q.perm[2 * ks + k];
      ci = c * q.chunk_ci + e;
    } else {
      tap = q.perm[ks];
      ci = c * q.chunk_ci + k * q.E + e;
    }
    const int co = cb * 64 + (row & 63);
    float w = 0.0f;
    if (tap < q.TAPS && ci < p.C && co < p.CO) {
      if (p.wlayout == 0) {
        w = p.w[((long)co * p.C + ci) * q.TAPS + tap];
      } else if (q.SP) {  // transposed conv by parity class: W[ci][co][kh][kw] as is
        w = p.w[((long)ci * p.CO + co) * 9 + tap];
      } else {  // transposed conv as a conv: swap channel axes, flip both taps
        const int kh = tap / q.KW, kw = tap % q.KW;
        w = p.w[(((long)ci * p.CO + co) * q.KH + (q.KH - 1 - kh)) * q.KW + (q.KW - 1 - kw)];
      }
    }
    const bool lo = row >= 64;
    const long base = ((((long)cb * q.NCH + c) * q.KS + ks) * kBStep) + k * 2048 + row * 16;
    if (q.prec == 0) {
      const uint32_t hi = tf32_rna(w);
      const uint32_t v = lo ? tf32_rna(w - __uint_as_float(hi)) : hi;
      reinterpret_cast<uint32_t *>(out + base)[e] = v;
    } else {
      if (f16_out_of_range(w)) atomicOr(p.status, ST_RANGE);
      wmx = fmaxf(wmx, fabsf(w));
      const __half hi = __float2half_rn(w);
      const __half v = lo ? __float2half_rn((w - __half2float(hi)) * 2048.0f) : hi;
      reinterpret_cast<__half *>(out + base)[e] = v;
    }
  }
  if (q.prec == 1 && p.wmax) {  // the block's maximum, for the main kernel's check
    __shared__ float red[8];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wmx = fmaxf(wmx, __shfl_xor_sync(0xffffffffu, wmx, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = wmx;
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = 0.0f;
      for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
      p.wmax[blockIdx.x] = m;
    }
  }
}

// Splits E input channels of one pixel into hi / lo parts and stores the
// two 16-byte slices.  fp16: hi = rn(v), lo = rn((v - hi) * 2^11), and |v|
// is folded into the running maximum `amax` for the range check (hi is
// infinite once |v| >= 65520); tf32: hi = rna(v), lo = rna(v - hi).
template <int PREC, int E>
__device__ __forceinline__ void store_slice(uint8_t *hi_dst, uint8_t *lo_dst, const float (&v)[E],
                                            float &amax) {
  uint32_t h[4], l[4];
  if constexpr (PREC == 0) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      h[e] = tf32_rna(v[e]);
      l[e] = tf32_rna(v[e] - __uint_as_float(h[e]));
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = v[2 * e], b = v[2 * e + 1];
      amax = fmaxf(amax, fmaxf(fabsf(a), fabsf(b)));  // NaN is not flagged
      h[e] = ptx::cvt_f16x2(a, b);
      float ha, hb, da, db;
      ptx::f16x2_to_f32(h[e], ha, hb);
      ptx::sub_mul_f32x2(a, b, ha, hb, 2048.0f, da, db);
      l[e] = ptx::cvt_f16x2(da, db);
    }
  }
  *reinterpret_cast<uint4 *>(hi_dst) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4 *>(lo_dst) = make_uint4(l[0], l[1], l[2], l[3]);
}



// One staged row of one slice plane.
struct RowJob {
  long rowbase;   // element index of (n, channel 0, id, ih, iw0)
  int cbase;      // first input channel of the slice plane
  uint32_t dst;   // byte offset of the row in the hi planes of the stage
  bool ok;        // the input row exists (else zeros)
};

// Where the stage's rows come from: unit position, first channel of the
// chunk and the staging geometry.
struct StageSrc {
  long xn;        // element index of image n
  int id0, ih0, iw0, ci0;  // first input depth, row, column; first channel
};

// Input row `job` of a stage: slice plane, depth slice, then the row r of
// the RIN loaded per depth.  Its staged pixels start at jb.dst; the input
// column cc lands at staged column col_px(cc) of that row.
__host__ __device__ __forceinline__ RowJob row_job(int job, const StageSrc &ss, const TcPlan &q,
                                                   const ConvProblem &p, int nrows, int E, bool s2,
                                                   bool cl = false) {
  RowJob jb;
  // a stage holds at most 2 slice planes of KD depth slices
  const int plane = job >= nrows ? 1 : 0;
  const int sr = job - plane * nrows;
  const int kdp = (int)fdiv((uint32_t)sr, q.fd_rin);  // no division routine in the loop
  const int r = sr - kdp * q.RIN;
  const int id = ss.id0 + kdp * q.DIL, ih = ss.ih0 + r;
  jb.ok = id >= 0 && id < p.D && ih >= 0 && ih < p.H;
  // channels-last input: pixels C floats apart, channels adjacent
  jb.rowbase = ss.xn + (((long)id * p.H + ih) * p.W + ss.iw0) * (cl ? p.C : 1);
  jb.cbase = ss.ci0 + plane * E;
  // stride 2: even / odd rows go to sub-plane row r >> 1 of their parity
  const int row_px = s2 ? 2 * (r & 1) * q.SUB + (r >> 1) * q.RS : r * q.RS;
  jb.dst = (uint32_t)(plane * q.plane_bytes + (kdp * q.DSL + row_px) * 16);
  return jb;
}

// Staged column of input column cc of a loaded row (stride 2: even / odd
// columns to their sub-planes).
__host__ __device__ __forceinline__ int col_px(int cc, int s2sub) {
  return s2sub ? (cc & 1) * s2sub + (cc >> 1) : cc;
}

// Loads E channels of staged pixel cc of a row (zero outside the image).
// Channels-first input: one load per channel plane (cstride apart).
// Channels-last (CL): the E channels are adjacent, read as float4 vectors
// when C is a multiple of 4 (then every slice starts 16-byte aligned).
template <int E, bool CL = false>
__device__ __forceinline__ void load_pixel(const float *__restrict__ x, const RowJob &jb, int cc,
                                           long cstride, int iw0, int W, int C, float (&v)[E]) {
  const bool colok = jb.ok && iw0 + cc >= 0 && iw0 + cc < W;
  if constexpr (CL) {
    const float *px = x + jb.rowbase + (long)cc * C + jb.cbase;
    if ((C & 3) == 0 && jb.cbase + E <= C) {
#pragma unroll
      for (int e = 0; e < E; e += 4) {
        const float4 f = colok ? __ldg(reinterpret_cast<const float4 *>(px + e))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        v[e] = f.x; v[e + 1] = f.y; v[e + 2] = f.z; v[e + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = (colok && jb.cbase + e < C) ? __ldg(px + e) : 0.0f;
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e)
      v[e] = (colok && jb.cbase + e < C) ? __ldg(x + jb.rowbase + cc + (long)(jb.cbase + e) * cstride)
                                          : 0.0f;
  }
}

// A loaded row of LW pixels has G = LW / 32 full 32-pixel groups, taken by
// ceil(G / 4) main jobs of at most 4 groups each (stride-2 column strips
// load 258 pixels a row: two main jobs); the LW - 32 G pixels left over go
// to tail jobs.  Main job J covers row J / parts, groups 4 (J % parts) on.
struct MainJob { int row, c0, ngroups; };
__host__ __device__ __forceinline__ MainJob main_job(int J, int parts, int G) {
  MainJob m;
  m.row = J / parts;
  const int part = J - m.row * parts;
  m.c0 = 128 * part;
  m.ngroups = G - 4 * part < 4 ? G - 4 * part : 4;
  return m;
}

// Main job: pixels cc = c0 + lane + 32k (k < NCOL) of one row, all loads in
// flight before the first store.  `wait_stage` runs between the loads and
// the stores (the stage may still be in use while the loads travel).
template <int PREC, int E, int NCOL, bool CL, class Wait>
__device__ __forceinline__ bool fill_row(const float *__restrict__ x, const RowJob &jb, int c0,
                                         long cstride, int iw0, int W, int C, uint8_t *stage,
                                         int lo_off, int lane, float &amax, int s2sub,
                                         Wait &&wait_stage) {
  float v[NCOL][E];
#pragma unroll
  for (int k = 0; k < NCOL; ++k)
    load_pixel<E, CL>(x, jb, c0 + lane + 32 * k, cstride, iw0, W, C, v[k]);
  if (!wait_stage()) return false;
#pragma unroll
  for (int k = 0; k < NCOL; ++k) {
    const uint32_t o = jb.dst + (uint32_t)col_px(c0 + lane + 32 * k, s2sub) * 16u;
    store_slice<PREC, E>(stage + o, stage + lo_off + o, v[k], amax);
  }
  return true;
}

// One M tile's KS K steps (elementwise units), unrolled: every step's
// shared-memory delta and weight offset at a constant address, the next
// step's delta read while this step's MMAs issue (few registers, no loop
// control between two MMA pairs); `look` runs before the last step when
// `lk`.
template <int PREC, int KS, class F>
__device__ __forceinline__ void issue_tile_fixed(const volatile uint32_t *kt, uint32_t at,
                                                 uint32_t b_lo, uint32_t d, uint32_t lo_delta,
                                                 int c, bool lk, F &&look) {
  constexpr uint32_t fmt = PREC ? 0u : 2u;
  constexpr uint32_t idesc1 = ptx::instr_desc(fmt, 128, 128);
  constexpr uint32_t idesc2 = ptx::instr_desc(fmt, 128, 64);
  constexpr uint64_t desc_hi = (uint64_t)((128u >> 4) | (1u << 14)) << 32;
  uint32_t kd_next = kt[0];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const uint32_t kd_cur = kd_next;
    if (ks + 1 < KS) kd_next = kt[ks + 1];
    if (ks == KS - 1 && lk) look();
    const uint32_t ah = at + kd_cur;
    const uint64_t bd = desc_hi | (b_lo + (uint32_t)(ks * (kBStep >> 4)));
    const uint32_t accum = (ks | c) ? 1u : 0u;
    if constexpr (PREC == 0) {
      ptx::mma_tf32(d, desc_hi | ah, bd, idesc1, accum);
      ptx::mma_tf32(d + 64, desc_hi | (ah + lo_delta), bd, idesc2, 1u);
    } else {
      ptx::mma_f16(d, desc_hi | ah, bd, idesc1, accum);
      ptx::mma_f16(d + 64, desc_hi | (ah + lo_delta), bd, idesc2, 1u);
    }
  }
}

// One K step's two products of an M tile: A_hi x [W_hi | W_lo] (N = 128)
// into columns d .. d + 127 and A_lo x W_hi (N = 64) into d + 64 .. d + 127.
// bk1 / bk2: low descriptor words of the two B operands (the same operand
// in one CTA; with CTA pairs this CTA's halves, M = 256 over both CTAs).
template <int PREC, bool PAIR>
__device__ __forceinline__ void mma_k_step(uint32_t d, uint32_t ah, uint32_t lo_delta,
                                           uint32_t bk1, uint32_t bk2, uint32_t accum) {
  constexpr uint32_t fmt = PREC ? 0u : 2u;
  constexpr uint32_t M = PAIR ? 256u : 128u;
  constexpr uint32_t idesc1 = ptx::instr_desc(fmt, M, 128), idesc2 = ptx::instr_desc(fmt, M, 64);
  constexpr uint64_t desc_hi = (uint64_t)((128u >> 4) | (1u << 14)) << 32;  // SBO 128 B, version 1
  const uint64_t a1 = desc_hi | ah, a2 = desc_hi | (ah + lo_delta);
  const uint64_t b1 = desc_hi | bk1, b2 = desc_hi | bk2;
  if constexpr (PAIR) {
    if constexpr (PREC == 0) {
      ptx::mma2_tf32(d, a1, b1, idesc1, accum);
      ptx::mma2_tf32(d + 64, a2, b2, idesc2, 1u);
    } else {
      ptx::mma2_f16(d, a1, b1, idesc1, accum);
      ptx::mma2_f16(d + 64, a2, b2, idesc2, 1u);
    }
  } else {
    if constexpr (PREC == 0) {
      ptx::mma_tf32(d, a1, b1, idesc1, accum);
      ptx::mma_tf32(d + 64, a2, b2, idesc2, 1u);
    } else {
      ptx::mma_f16(d, a1, b1, idesc1, accum);
      ptx::mma_f16(d + 64, a2, b2, idesc2, 1u);
    }
  }
}

// A pooled chunk of KS K steps, every one of the U tiles per step,
// unrolled (same reads as issue_tile_fixed); `look` runs before the last
// step.
template <int PREC, int U, int KS, bool PAIR, class F>
__device__ __forceinline__ void issue_pool_fixed(const volatile uint32_t *kt, uint32_t a_lo,
                                                 uint32_t b_lo, uint32_t b_lo2, uint32_t dacc,
                                                 uint32_t lo_delta, uint32_t tile_delta, int c,
                                                 F &&look) {
  constexpr uint32_t kStep16 = (PAIR ? 3072u : (uint32_t)kBStep) >> 4;
  uint32_t kd_next = kt[0];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const uint32_t kd_cur = kd_next;
    if (ks + 1 < KS) kd_next = kt[ks + 1];
    if (ks == KS - 1) look();
    const uint32_t ah = a_lo + kd_cur;
    const uint32_t accum = (ks | c) ? 1u : 0u;
#pragma unroll
    for (int t = 0; t < U; ++t)
      mma_k_step<PREC, PAIR>(dacc + (uint32_t)(t * 128), ah + (uint32_t)t * tile_delta, lo_delta,
                             b_lo + (uint32_t)ks * kStep16, b_lo2 + (uint32_t)ks * kStep16, accum);
  }
}

// Every MMA of a CTA's units issued by one thread (all entries but the
// parity-class pooled one).  The tensor pipe runs at most about one MMA
// ahead of the issuing thread (measured: a pause of n clocks between two
// chunks lengthens the chunk by about n), so the work between two chunks is
// kept to commits and a fence: the next chunk's stage (with streamed
// weights also the next weight slot, and in a unit's last chunk the next
// accumulator) is tested before the chunk's last K step, while its MMAs
// run; no warp vote, no per-step elect; addresses from counters.
// Pooled units (POOL) issue every tile per K step and complete the unit's
// accumulator at once; elementwise units go tile by tile, each tile's
// accumulator completed by its own commit in the unit's last chunk, so the
// epilogue can start on it.  UNROLL: 14-step tiles unrolled (off for the
// channels-last instances, where it spilled registers).  Returns false
// when a wait gave up (the abort flag is then set).
template <int PREC, int U, bool POOL, bool UNROLL, bool PAIR>
__device__ __forceinline__ bool issue_units(const TcPlan &q, long units, uint32_t sbase,
                                            uint32_t tmem, uint64_t *bars, const uint32_t *kd_smem,
                                            uint32_t lo_delta, uint32_t tile_delta,
                                            volatile int *abort, unsigned int *status) {
  constexpr int A_FULL = 0, A_EMPTY = 4, B_FULL = 8, B_EMPTY = 10, ACC_FULL = 12, ACC_EMPTY = 16;
  constexpr uint32_t fmt = PREC ? 0u : 2u;
  constexpr uint32_t idesc1 = ptx::instr_desc(fmt, 128, 128);
  constexpr uint32_t idesc2 = ptx::instr_desc(fmt, 128, 64);
  constexpr uint64_t desc_hi = (uint64_t)((128u >> 4) | (1u << 14)) << 32;  // SBO 128 B, version 1
  const volatile uint32_t *kt = kd_smem;
  const uint32_t a_base = (sbase >> 4) & 0x3FFFu, a_step = (uint32_t)(q.a_stage_bytes >> 4);
  const uint32_t b_base = ((sbase + (uint32_t)q.off_b) >> 4) & 0x3FFFu;
  const uint32_t b_step = (uint32_t)(q.b_chunk_bytes >> 4);
  const bool resident = q.b_resident != 0;
  // commits reach both CTAs of a pair (each has its stage and accumulator
  // barriers at the same offsets)
  auto commit = [](uint64_t *bar) {
    if constexpr (PAIR) ptx::tc_commit2(bar, 3);
    else ptx::tc_commit(bar);
  };
  int ms = 0, macc = 0, msb = 0;
  uint32_t mph = 0, mpar = 0, msbph = 0, g = 0, it = 0;
  // seen complete by the look-ahead tests
  bool full_ok = false, acc_ok = false, wfull_ok = false;
  for (long u = blockIdx.x; u < units; u += gridDim.x, ++it) {
    const uint32_t cb = fdiv((uint32_t)u, q.fd_cb);
    const int acc = macc;
    const uint32_t acc_par = mpar ^ 1;
    if (++macc == q.NACC) { macc = 0; mpar ^= 1; }
    // one wait for the whole accumulator: the epilogue frees a unit's tiles
    // in order, so the last tile's barrier implies the others
    if (!acc_ok && !wait_bar(bars, ACC_EMPTY + (POOL ? acc : acc * U + U - 1), acc_par, abort,
                             status, 0x21000000u | it))
      return false;
    ptx::tc_fence_after();
    const uint32_t dacc = tmem + (uint32_t)(acc * U * 128);
    // B descriptors' low words: start | slice distance (LBO) << 16; with
    // CTA pairs this CTA's 64 rows of [W_hi | W_lo] (slices 1 KB apart)
    // and, 2 KB further, its 32 rows of W_hi (slices 512 B apart)
    constexpr uint32_t kLbo1 = (PAIR ? 1024u : 2048u) >> 4;
    uint32_t b_res = (b_base + cb * (uint32_t)q.NCH * b_step) | (kLbo1 << 16);
    for (int c = 0; c < q.NCH; ++c, ++g, b_res += b_step) {
      const int s = ms, sb = msb;
      const uint32_t sph = mph, sbph = msbph;
      if (++ms == q.S) { ms = 0; mph ^= 1; }
      if (!full_ok && !wait_bar(bars, A_FULL + s, sph, abort, status, 0x22000000u | g))
        return false;
      uint32_t b_lo = b_res;
      if (!resident) {  // weight ring slot sb
        if (++msb == q.SB) { msb = 0; msbph ^= 1; }
        if (!wfull_ok && !wait_bar(bars, B_FULL + sb, sbph, abort, status, 0x23000000u | g))
          return false;
        b_lo = (b_base + (uint32_t)sb * b_step) | (kLbo1 << 16);
      }
      const uint32_t b_lo2 = PAIR ? (((b_lo & 0x3FFFu) + (2048u >> 4)) | ((512u >> 4) << 16)) : b_lo;
      ptx::tc_fence_after();
      const uint32_t a_lo = a_base + (uint32_t)s * a_step;
      const bool last = c == q.NCH - 1;
      auto look_ahead = [&]() {  // while this chunk's last MMAs run
        full_ok = ptx::mbar_test_wait(bars + A_FULL + ms, mph);
        if (!resident) wfull_ok = ptx::mbar_test_wait(bars + B_FULL + msb, msbph);
        if (last)
          acc_ok = ptx::mbar_test_wait(bars + ACC_EMPTY + (POOL ? macc : macc * U + U - 1),
                                       mpar ^ 1);
      };
      if (POOL && U == 2 && q.KS == 9) {
        uint32_t bt, bt2;  // opaque: keeps the steps' descriptors from being hoisted
        asm volatile("mov.b32 %0, %1;" : "=r"(bt) : "r"(b_lo));
        asm volatile("mov.b32 %0, %1;" : "=r"(bt2) : "r"(b_lo2));
        issue_pool_fixed<PREC, U, 9, PAIR>(kt, a_lo, bt, bt2, dacc, lo_delta, tile_delta, c,
                                           look_ahead);
      } else if constexpr (POOL) {
        uint32_t kd_next = kt[0];
        for (int ks = 0; ks < q.KS; ++ks) {
          const uint32_t kd_cur = kd_next;
          kd_next = kt[ks + 1];
          if (ks == q.KS - 1) look_ahead();
          const uint32_t ah = a_lo + kd_cur;
          const uint32_t kb = (uint32_t)ks * ((PAIR ? 3072u : (uint32_t)kBStep) >> 4);
          const uint32_t accum = (ks | c) ? 1u : 0u;
#pragma unroll
          for (int t = 0; t < U; ++t)
            mma_k_step<PREC, PAIR>(dacc + (uint32_t)(t * 128), ah + (uint32_t)t * tile_delta,
                                   lo_delta, b_lo + kb, b_lo2 + kb, accum);
        }
      } else {
#pragma unroll 1
        for (int t = 0; t < U; ++t) {
          const uint32_t at = a_lo + (uint32_t)t * tile_delta;
          const uint32_t d = dacc + (uint32_t)(t * 128);
          const bool lk = t == U - 1;
          // 3x3x3 with 8-channel chunks (14 paired K steps): unrolled
          // (0.653 -> 0.563 ms on the conv3d workload); the loop measured
          // faster for 5 steps (conv2d 0.135 unrolled against 0.114 ms)
          switch (UNROLL ? q.KS : 0) {
            case 14: {
              // the weight start as an opaque per-tile value: otherwise every
              // unrolled step's descriptor is hoisted out of the tile loop
              // and held in registers (spilled)
              uint32_t bt;
              asm volatile("mov.b32 %0, %1;" : "=r"(bt) : "r"(b_lo));
              issue_tile_fixed<PREC, 14>(kt, at, bt, d, lo_delta, c, lk, look_ahead);
            } break;
            default: {  // the K-step loop over the table in shared memory
          uint32_t kd_next = kt[0];
          for (int ks = 0; ks < q.KS; ++ks) {
            const uint32_t kd_cur = kd_next;
            kd_next = kt[ks + 1];
            if (lk && ks == q.KS - 1) look_ahead();
            const uint32_t ah = at + kd_cur;
            const uint64_t bd = desc_hi | (b_lo + (uint32_t)(ks * (kBStep >> 4)));
            const uint32_t accum = (ks | c) ? 1u : 0u;
            if constexpr (PREC == 0) {
              ptx::mma_tf32(d, desc_hi | ah, bd, idesc1, accum);
              ptx::mma_tf32(d + 64, desc_hi | (ah + lo_delta), bd, idesc2, 1u);
            } else {
              ptx::mma_f16(d, desc_hi | ah, bd, idesc1, accum);
              ptx::mma_f16(d + 64, desc_hi | (ah + lo_delta), bd, idesc2, 1u);
            }
          }
            } break;
          }
          if (last) commit(bars + ACC_FULL + acc * U + t);
        }
      }
      commit(bars + A_EMPTY + s);
      if (!resident) commit(bars + B_EMPTY + sb);
    }
    if constexpr (POOL) commit(bars + ACC_FULL + acc);
  }
  return true;
}

// Issues one chunk of the stride-2 transposed conv by parity class: K step
// ks adds into accumulator (kcls[ks] & 3) x 128 columns; the class's first
// K step of the unit's first chunk starts the accumulator (accumulate 0).
// Fully unrolled over KS (5 paired or 9 single K steps) with the step
// tables in registers, so no shared-memory load sits between two bursts.
template <int PREC, int K0, int K1>
__device__ __forceinline__ void issue_subpix(const uint32_t (&kt)[28], const uint32_t (&kc)[9],
                                             uint32_t a_lo, uint32_t b_lo, uint32_t dacc,
                                             uint32_t lo_delta, bool first_chunk) {
  constexpr uint32_t fmt = PREC ? 0u : 2u;
  constexpr uint32_t idesc1 = ptx::instr_desc(fmt, 128, 128);
  constexpr uint32_t idesc2 = ptx::instr_desc(fmt, 128, 64);
  constexpr uint64_t desc_hi = (uint64_t)((128u >> 4) | (1u << 14)) << 32;
#pragma unroll
  for (int ks = K0; ks < K1; ++ks) {
    const uint32_t ah = a_lo + kt[ks];
    const uint32_t cls = kc[ks];
    const uint64_t bd = desc_hi | (b_lo + (uint32_t)(ks * (kBStep >> 4)));
    const uint32_t accum = (first_chunk && (cls & 0x80u)) ? 0u : 1u;
    const uint32_t d = dacc + (cls & 3u) * 128u;
    if (ptx::elect_one()) {
      if constexpr (PREC == 0) {
        ptx::mma_tf32(d, desc_hi | ah, bd, idesc1, accum);
        ptx::mma_tf32(d + 64, desc_hi | (ah + lo_delta), bd, idesc2, 1u);
      } else {
        ptx::mma_f16(d, desc_hi | ah, bd, idesc1, accum);
        ptx::mma_f16(d + 64, desc_hi | (ah + lo_delta), bd, idesc2, 1u);
      }
    }
    __syncwarp();
  }
}

// Sums v[0..15] over the 32 lanes of a warp: after the call lane l holds in
// v[0] the total of the value v[(l >> 1) & 15] had on every lane.
__device__ __forceinline__ void lane_sum16(float (&v)[16], int lane) {
#pragma unroll
  for (int h = 8, o = 16; h >= 1; h >>= 1, o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = up ? v[i] : v[i + h];
      const float keep = up ? v[i + h] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
}

template <int PREC, int CHAIN, bool POOL, int U, bool S2, bool SP, bool CL, bool GP, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
tc_conv_kernel(ConvProblem p, TcPlan q, const uint8_t *__restrict__ bimg,
               float *__restrict__ partial, const __grid_constant__ CUtensorMap tmx) {
  constexpr int E = PREC ? 8 : 4;
  static_assert(U >= 1 && U <= 4, "one to four M tiles per unit");
  static_assert(!POOL || U == 2 || SP || GP, "the 2x2 pool takes two output rows per unit");
  static_assert(!GP || (POOL && !SP && !S2 && !CL), "general pool: stride-1 pooled entry");
  static_assert(!SP || (POOL && U == 1 && !S2), "parity classes: one pooled tile per unit");
  static_assert(!CL || (!POOL && !S2), "channels-last: stride-1 elementwise entries");
  static_assert(!PAIR || (POOL && U == 2 && !SP && !GP), "CTA pairs: the 2x2-pooled entry");
  using RL = Roles<POOL && !SP && !GP>;
  constexpr int kEpiWarps = RL::kEpi, kMmaWarp = RL::kMma, kProdWarp0 = RL::kProd0;
  constexpr int kProdWarps = RL::kProd, kProdThreads = RL::kProdT;
  constexpr int kEpiThreads = 32 * kEpiWarps;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + q.off_bar);
  constexpr int A_FULL = 0, A_EMPTY = 4, B_FULL = 8, B_EMPTY = 10, ACC_FULL = 12,
                ACC_EMPTY = 16, DRAIN = 20, RAW_FULL = 21, RAW_EMPTY = 25;
  uint64_t *a_full = bars + A_FULL;
  uint64_t *a_empty = bars + A_EMPTY;
  uint64_t *b_full = bars + B_FULL;
  uint64_t *b_empty = bars + B_EMPTY;
  uint64_t *acc_full = bars + ACC_FULL;
  uint64_t *acc_empty = bars + ACC_EMPTY;
  uint64_t *drain = bars + DRAIN;
  SmemCtl *ctl = reinterpret_cast<SmemCtl *>(smem + q.off_misc);
  volatile int *abort_flag = &ctl->abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    // (CTA pairs: the even CTA's stage-full and accumulator-empty barriers
    // also count the odd CTA's producer and epilogue warps)
    for (int s = 0; s < q.S; ++s) {  // tensor-copy staging: one warp loads, the rest convert
      ptx::mbar_init(&a_full[s], (uint32_t)((q.TMA ? kProdWarps - 1 : kProdWarps) * (PAIR ? 2 : 1)));
      ptx::mbar_init(&a_empty[s], 1);
    }
    for (int r = 0; r < q.TR; ++r) {
      ptx::mbar_init(&bars[RAW_FULL + r], 1);
      ptx::mbar_init(&bars[RAW_EMPTY + r], (uint32_t)(kProdWarps - 1));
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&b_full[s], 1);
      ptx::mbar_init(&b_empty[s], 1);
    }
    for (int a = 0; a < 4; ++a) {
      ptx::mbar_init(&acc_full[a], 1);
      ptx::mbar_init(&acc_empty[a], kEpiWarps * (PAIR ? 2 : 1));
    }
    ptx::mbar_init(drain, 1);
    ctl->abort = 0;
    ctl->amax_bits = 0;
    ptx::fence_mbar_init();
  }
  if (SP && tid < q.KS) {  // per-class K steps, laid out on the host
    ctl->kdelta[tid] = q.skd[tid];
    ctl->kcls[tid] = q.kcls[tid];
  } else if (tid < q.KS) {
    uint32_t off16, lbo16;
    if (q.pairtaps) {  // slices: taps 2ks and 2ks+1 (a zero-weight slice past the last)
      const int t0 = q.perm[2 * tid], t1 = q.perm[2 * tid + 1];
      const int s0 = tap_shift(t0, q);
      off16 = (uint32_t)s0;
      lbo16 = (t1 < q.TAPS) ? (uint32_t)(tap_shift(t1, q) - s0) : 1u;
    } else {           // slices: planes 0 and 1 of tap ks
      off16 = (uint32_t)tap_shift(q.perm[tid], q);
      lbo16 = (uint32_t)(q.plane_bytes >> 4);
    }
    ctl->kdelta[tid] = (off16 & 0x3FFFu) | ((lbo16 & 0x3FFFu) << 16);
  } else if (tid < kMaxTaps + 2) {
    ctl->kdelta[tid] = 0;  // read (unused) by the last step's prefetch
  }
  for (int c = tid; c < q.COB * 64; c += kThreads) {
    ctl->bias[c] = (c < p.CO && p.epi.bias) ? p.epi.bias[c] : 0.0f;
    ctl->addend[c] = ((CHAIN == CHAIN_LEAKY_ADD_CLAMP_GELU ||
                       CHAIN == CHAIN_LEAKY_ADD_CLAMP1_GELU) && c < p.CO)
                         ? p.epi.chan[1][c]
                         : 0.0f;
  }
  const uint32_t rank = PAIR ? ptx::cluster_rank() : 0u;
  if (warp == kMmaWarp) {
    if constexpr (PAIR) {  // one allocation spanning both CTAs, same address in each
      ptx::tmem_alloc2(&ctl->tmem_base, (uint32_t)q.tmem_cols);
      ptx::tmem_relinquish2();
    } else {
      ptx::tmem_alloc(&ctl->tmem_base, (uint32_t)q.tmem_cols);
      ptx::tmem_relinquish();
    }
  }
  if constexpr (PAIR) {
    // This CTA's half of B, resident: per K step of the packed image (2
    // slices x 128 rows of [W_hi | W_lo], 16 B a row) the rows 64 rank ..
    // 64 rank + 63 of each slice (the N = 128 product's columns of this
    // CTA) and the rows 32 rank .. 32 rank + 31 (of W_hi: the N = 64
    // product's), at 3072 bytes a K step.  Both CTAs' halves are in place
    // before the cluster barrier below, so the first MMA needs no wait.
    if (tid == 0) {
      const long ksteps = (long)q.COB * q.NCH * q.KS;
      ptx::mbar_arrive_expect_tx(&b_full[0], (uint32_t)(ksteps * 3072));
      for (long k = 0; k < ksteps; ++k) {
        const uint8_t *src = bimg + k * kBStep;
        uint8_t *dst = smem + q.off_b + k * 3072;
        for (int sl = 0; sl < 2; ++sl) {
          ptx::bulk_g2s(dst + sl * 1024, src + sl * 2048 + rank * 1024, 1024u, &b_full[0]);
          ptx::bulk_g2s(dst + 2048 + sl * 512, src + sl * 2048 + rank * 512, 512u, &b_full[0]);
        }
      }
      volatile int no_abort = 0;
      wait_bar(bars, B_FULL, 0, &no_abort, p.status, 0x17000000u);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) ptx::cluster_sync();  // barriers, TMEM and weights ready in both CTAs
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  const long units = q.units;
  const int HW = p.H * p.W;

  if (warp >= kProdWarp0) {
    // ------------------------------------------------------------ producers
    const int pt = tid - kProdWarp0 * 32;
    const int pw = warp - kProdWarp0;  // producer warp index
    float amax = 0.0f;                 // largest |x| staged (fp16 range check)
    uint32_t g = 0;
    bool ok = true;
    if (!PAIR && q.b_resident && pt == 0) {
      const long total = (long)q.COB * q.NCH * q.b_chunk_bytes;
      ptx::mbar_arrive_expect_tx(&b_full[0], (uint32_t)total);
      for (long off = 0; off < total; off += 16384) {
        const uint32_t nb = (uint32_t)((total - off) < 16384 ? (total - off) : 16384);
        ptx::bulk_g2s(smem + q.off_b + off, bimg + off, nb, &b_full[0]);
      }
    }
    const int nrows = p.KD * q.RIN;  // staged rows per slice plane
    const int jobs = q.P * nrows;     // (plane, staged row) pairs per stage
    const long cstride = (long)p.D * HW;
    // A stage is filled by main jobs (one row: its full 32-pixel column
    // groups) and tail jobs (32 of the rows' remaining pixels each).
    const int G = q.LW >> 5;
    // stride 1 loads at most 130 pixels a row: one main job, or none for
    // rows shorter than 32 pixels
    const int parts = S2 ? (G + 3) >> 2 : (G ? 1 : 0);
    const int tail = q.LW - 32 * G;
    const int mjobs = jobs * parts;
    const int njobs = mjobs + cdiv(jobs * tail, 32);
    const int s2sub = S2 ? q.SUB : 0;
    // Staged pixels no row job writes (past the staged rows; with stride 2
    // also the odd-row sub-planes' last row) are only read by discarded M
    // rows; zero them once so those rows stay finite.
    {
      const int tail0 = S2 ? 0 : nrows * q.RS;
      for (int st = 0; st < q.S; ++st)
        for (int pl = 0; pl < 2 * q.P; ++pl)
          for (int px = tail0 + pt; px < q.NPIX; px += kProdThreads)
            *reinterpret_cast<uint4 *>(smem + (long)st * q.a_stage_bytes + pl * q.plane_bytes +
                                       px * 16) = make_uint4(0, 0, 0, 0);
    }
    bool tma_done = false;
    if constexpr (!S2 && !SP && !POOL) {  // the pooled instances keep the smaller code
      if (q.TMA) {
        // ---- tensor-copy staging.  One producer warp (its first lane) issues
        // one tiled tensor copy per (chunk, depth slice) into the raw ring and
        // streams the weights; the others split each raw slice into the
        // stage's hi / lo slices (zeros outside the image come from the copy
        // itself).  The loader is the producer warp on the MMA warp's
        // scheduler (warp w issues on scheduler w % 4): its light work there
        // instead of a converter's.
        constexpr int kLoaderPw = ((kMmaWarp & 3) - (kProdWarp0 & 3) + 4) & 3;
        uint8_t *raw0 = smem + q.off_raw;
        int rs = 0;
        uint32_t rph = 0;
        const int iw_adj = CL ? 0 : q.coff;
        if (pw == kLoaderPw) {
          ptx::tma_prefetch_desc(&tmx);
          int last_rs = -1;
          uint32_t last_par = 0;  // bit r: phase parity of the last copy into slot r
          for (long u = blockIdx.x; ok && u < units; u += gridDim.x) {
            const UnitPos up = decode_unit(u, q);
            const int id0 = up.od - p.pad_d;
            const int ih0 = up.rt * q.ROWSTEP - p.pad;
            const int iw0 = up.ct * q.COLSTEP - p.pad - iw_adj;
            for (int c = 0; ok && c < q.NCH; ++c, ++g) {
              if (!q.b_resident) {
                const int sb = psb_tma_slot(g, q.SB);
                if (!wait_bar_warp(bars, B_EMPTY + sb, ((g / q.SB) & 1) ^ 1, abort_flag, p.status,
                                   0x11000000u | g)) {
                  ok = false;
                  break;
                }
                if (lane == 0) {
                  ptx::mbar_arrive_expect_tx(&b_full[sb], (uint32_t)q.b_chunk_bytes);
                  const uint8_t *src = bimg + ((long)up.cb * q.NCH + c) * q.b_chunk_bytes;
                  uint8_t *dst = smem + q.off_b + (long)sb * q.b_chunk_bytes;
                  for (int off = 0; off < q.b_chunk_bytes; off += 16384) {
                    const int nb = (q.b_chunk_bytes - off) < 16384 ? (q.b_chunk_bytes - off) : 16384;
                    ptx::bulk_g2s(dst + off, src + off, (uint32_t)nb, &b_full[sb]);
                  }
                }
                __syncwarp();
              }
              const int ci0 = c * q.chunk_ci;
              for (int kd = 0; kd < p.KD; ++kd) {
                if (!wait_bar_warp(bars, RAW_EMPTY + rs, rph ^ 1, abort_flag, p.status,
                                   0x14000000u | g)) {
                  ok = false;
                  break;
                }
                if (!CL && (iw0 & 3)) {
                  // a plan error (the copy's first column must be 16-byte
                  // aligned): report it and stop instead of issuing the copy
                  if (lane == 0) {
                    record_timeout(p.status, &bars[RAW_FULL + rs], RAW_FULL + rs, rph, 0x17000000u | g);
                    atomicOr(p.status, ST_PLAN);
                    *abort_flag = 1;
                  }
                  ok = false;
                  break;
                }
                if (lane == 0) {
                  uint64_t *bar = &bars[RAW_FULL + rs];
                  uint8_t *dst = raw0 + (long)rs * q.raw_bytes;
                  ptx::mbar_arrive_expect_tx(bar, (uint32_t)q.raw_tx);
                  const int id = id0 + kd * q.DIL;
                  // 3-D entry (any kernel depth): a rank-5 map with a depth axis
                  if constexpr (CL) {
                    if (p.entry != 1) ptx::tma_load_4d(dst, &tmx, ci0, iw0, ih0, up.n, bar);
                    else ptx::tma_load_5d(dst, &tmx, ci0, iw0, ih0, id, up.n, bar);
                  } else {
                    if (p.entry != 1) ptx::tma_load_4d(dst, &tmx, iw0, ih0, ci0, up.n, bar);
                    else ptx::tma_load_5d(dst, &tmx, iw0, ih0, id, ci0, up.n, bar);
                  }
                }
                __syncwarp();
                last_rs = rs > last_rs ? rs : last_rs;
                last_par = (last_par & ~(1u << rs)) | (rph << rs);
                if (++rs == q.TR) { rs = 0; rph ^= 1; }
              }
            }
          }
          // every issued copy has landed before the CTA can exit (waits bounded
          // by time only: they run even after an abort)
          if (lane == 0) {
            volatile int no_abort = 0;
            for (int r = 0; r <= last_rs; ++r)
              wait_bar(bars, RAW_FULL + r, (last_par >> r) & 1u, &no_abort, p.status,
                       0x15000000u | r);
          }
          if (lane == 0 && q.b_resident)  // the resident weights' copy (issued by pt 0)
            wait_bar(bars, B_FULL, 0, abort_flag, p.status, 0x12000000u);
          if (lane == 0 && !q.b_resident && g > 0) {
            const uint32_t lb = g - 1;
            wait_bar(bars, B_FULL + (int)(lb % q.SB), (lb / q.SB) & 1, abort_flag, p.status,
                     0x13000000u | lb);
          }
        } else {
          // converter thread, 0 .. 32 (kProdWarps - 1) - 1
          const int ct = (pw < kLoaderPw ? pw : pw - 1) * 32 + lane;
          constexpr int kConv = 32 * (kProdWarps - 1);
          const int lo_off = q.P * q.plane_bytes;
          const int items = q.P * q.RIN * q.LW;  // (plane, row, column) per depth slice
          const int chs = q.RIN * q.BW;          // channels-first: floats between channels
          int ps = 0;
          uint32_t pph = 0;
          for (long u = blockIdx.x; ok && u < units; u += gridDim.x) {
            for (int c = 0; ok && c < q.NCH; ++c, ++g) {
              const int s = ps;
              uint8_t *stage = smem + (long)s * q.a_stage_bytes;
              if (!wait_bar_warp(bars, A_EMPTY + s, pph ^ 1, abort_flag, p.status, 0x10000000u | g)) {
                ok = false;
                break;
              }
              for (int kd = 0; kd < p.KD; ++kd) {
                if (!wait_bar_warp(bars, RAW_FULL + rs, rph, abort_flag, p.status, 0x16000000u | g)) {
                  ok = false;
                  break;
                }
                const float *raw = reinterpret_cast<const float *>(raw0 + (long)rs * q.raw_bytes);
                for (int it = ct; it < items; it += kConv) {
                  const int row = (int)fdiv((uint32_t)it, q.fd_lw);
                  const int cc = it - row * q.LW;
                  const int pl = row >= q.RIN ? 1 : 0;
                  const int r = row - pl * q.RIN;
                  float v[E];
                  if constexpr (CL) {
                    const float4 *src = reinterpret_cast<const float4 *>(
                        raw + ((long)r * q.LW + cc) * q.chunk_ci + pl * E);
#pragma unroll
                    for (int e = 0; e < E; e += 4) {
                      const float4 f = src[e / 4];
                      v[e] = f.x; v[e + 1] = f.y; v[e + 2] = f.z; v[e + 3] = f.w;
                    }
                  } else {
                    const float *src = raw + ((long)pl * E * q.RIN + r) * q.BW + cc + q.coff;
#pragma unroll
                    for (int e = 0; e < E; ++e) v[e] = src[e * chs];
                  }
                  const uint32_t o = (uint32_t)(pl * q.plane_bytes + (kd * q.DSL + r * q.RS + cc) * 16);
                  store_slice<PREC, E>(stage + o, stage + lo_off + o, v, amax);
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bars[RAW_EMPTY + rs]);
                if (++rs == q.TR) { rs = 0; rph ^= 1; }
              }
              if (!ok) break;
              if (++ps == q.S) { ps = 0; pph ^= 1; }
              ptx::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive(&a_full[s]);
            }
          }
        }
        if (amax >= 65520.0f) atomicOr(p.status, ST_RANGE);  // some hi part overflowed
        atomicMax(&ctl->amax_bits, __float_as_uint(amax));    // |x| >= 0: bits order as values
        tma_done = true;
      }
    }
    if (!tma_done) {
    // 2x2-pooled stages of one job a warp at most (rows of 128..159 staged
    // columns, weights resident): each warp issues the loads of its job of
    // the NEXT stage before it waits for and fills the current one, so a
    // stage's loads are in flight for a whole stage period instead of being
    // waited for after the stage is free (two register buffers of 4 column
    // groups x E channels).  Jobs and their rotation as below.
    uint32_t last_b = 0xffffffffu;  // last chunk whose weights this warp streamed
    bool db_done = false;
    if constexpr (POOL && !SP && !GP && !S2 && !CL) {
      if (q.b_resident && njobs <= kProdWarps && G == 4 && parts == 1 && blockIdx.x < units) {
        db_done = true;
        auto stage_src = [&](long uu, int cc) {
          const UnitPos up = decode_unit(uu, q);
          StageSrc r;
          r.id0 = up.od * p.stride - p.pad_d;
          r.ih0 = up.rt * q.ROWSTEP * p.stride - p.pad;
          r.iw0 = up.ct * q.COLSTEP * p.stride - p.pad;
          r.xn = (long)up.n * p.C * p.D * HW;
          r.ci0 = cc * q.chunk_ci;
          return r;
        };
        // job J of the stage at `src` into v: a main job (row J, the row's 4
        // column groups) or a tail job (lane -> one of the rows' last
        // LW - 128 pixels); `dst` gets the byte offset of each loaded slice
        // in the hi planes (or ~0u: nothing to store)
        auto load_job = [&](int J, const StageSrc &src, float (&v)[4][E], uint32_t (&dst)[4]) {
          if (J < mjobs) {
            const RowJob jb = row_job(J, src, q, p, nrows, E, false);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              load_pixel<E, false>(p.x, jb, lane + 32 * k, cstride, src.iw0, p.W, p.C, v[k]);
              dst[k] = jb.dst + (uint32_t)(lane + 32 * k) * 16u;
            }
          } else {
            const int l = (J - mjobs) * 32 + lane;
            const int job = l / tail;
            const int cc = 32 * G + (l - job * tail);
#pragma unroll
            for (int k = 1; k < 4; ++k) dst[k] = ~0u;
            dst[0] = ~0u;
            if (job < jobs) {
              const RowJob jb = row_job(job, src, q, p, nrows, E, false);
              load_pixel<E, false>(p.x, jb, cc, cstride, src.iw0, p.W, p.C, v[0]);
              dst[0] = jb.dst + (uint32_t)cc * 16u;
            }
          }
        };
        const int lo_off = q.P * q.plane_bytes;
        long u = blockIdx.x;
        int c = 0, ps = 0, rot = 0;
        uint32_t pph = 0;
        StageSrc ss = stage_src(u, 0);
        float va[4][E], vb[4][E];
        uint32_t da[4], db[4];
        int JA = pw;  // rot = 0
        if (JA < njobs) load_job(JA, ss, va, da);
        for (;;) {
          long un = u;
          int cn = c + 1;
          if (cn == q.NCH) { cn = 0; un = u + gridDim.x; }
          int rotn = rot + njobs % kProdWarps;
          if (rotn >= kProdWarps) rotn -= kProdWarps;
          int JB = pw - rotn;
          if (JB < 0) JB += kProdWarps;
          StageSrc sn = ss;
          if (un < units) {
            if (un != u) sn = stage_src(un, 0);
            else sn.ci0 = cn * q.chunk_ci;
            if (JB < njobs) load_job(JB, sn, vb, db);
          }
          // the current stage: free once the MMAs that read it S chunks ago
          // are done; then the slices loaded one stage ago go in
          const int s = ps;
          if (!wait_bar_warp(bars, A_EMPTY + s, pph ^ 1, abort_flag, p.status, 0x10000000u | g)) {
            ok = false;
            break;
          }
          uint8_t *stage = smem + (long)s * q.a_stage_bytes;
          if (JA < njobs) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (da[k] != ~0u) store_slice<PREC, E>(stage + da[k], stage + lo_off + da[k], va[k], amax);
          }
          if (++ps == q.S) { ps = 0; pph ^= 1; }
          ++g;
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {  // (CTA pairs: the even CTA's barrier)
            if constexpr (PAIR) ptx::mbar_arrive_at(&a_full[s], 0);
            else ptx::mbar_arrive(&a_full[s]);
          }
          if (un >= units) break;
          u = un;
          c = cn;
          ss = sn;
          rot = rotn;
          JA = JB;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            da[k] = db[k];
#pragma unroll
            for (int e = 0; e < E; ++e) va[k][e] = vb[k][e];
          }
        }
      }
    }
    if (!db_done) {
    // Job J of a stage goes to producer warp (rot + J) % kProdWarps, where
    // rot counts the jobs of all earlier stages: the remainder of
    // njobs / kProdWarps moves round the warps instead of always landing on
    // the first ones.
    int rot = 0;
    // ring positions kept as counters (no integer division in the loop):
    // stage ps of phase pph; weight slot psb of phase psbph
    int ps = 0, psb = 0;
    uint32_t pph = 0, psbph = 0;
    for (long u = blockIdx.x; ok && u < units; u += gridDim.x) {
      const UnitPos up = decode_unit(u, q);
      StageSrc ss;
      const int st = p.stride;
      ss.id0 = up.od * st - p.pad_d;
      ss.ih0 = up.rt * q.ROWSTEP * st - p.pad;  // input row of the unit's first output row
      ss.iw0 = up.ct * q.COLSTEP * st - p.pad;
      ss.xn = (long)up.n * p.C * p.D * HW;
      for (int c = 0; c < q.NCH; ++c, ++g) {
        const int s = ps;
        if (!q.b_resident && pw == 0) {
          const int sb = psb;
          if (!wait_bar_warp(bars, B_EMPTY + sb, psbph ^ 1, abort_flag, p.status, 0x11000000u | g)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(&b_full[sb], (uint32_t)q.b_chunk_bytes);
            const uint8_t *src = bimg + ((long)up.cb * q.NCH + c) * q.b_chunk_bytes;
            uint8_t *dst = smem + q.off_b + (long)sb * q.b_chunk_bytes;
            for (int off = 0; off < q.b_chunk_bytes; off += 16384) {
              const int nb = (q.b_chunk_bytes - off) < 16384 ? (q.b_chunk_bytes - off) : 16384;
              ptx::bulk_g2s(dst + off, src + off, (uint32_t)nb, &b_full[sb]);
            }
          }
          last_b = g;
        }
        uint8_t *stage = smem + (long)s * q.a_stage_bytes;
        const int lo_off = q.P * q.plane_bytes;
        ss.ci0 = c * q.chunk_ci;
        // the stage is free once the MMAs that read it S chunks ago are done;
        // a warp's first loads of the stage are issued before it waits
        bool waited = false;
        auto wait_stage = [&]() -> bool {
          if (waited) return true;
          waited = true;
          const bool w = wait_bar_warp(bars, A_EMPTY + s, pph ^ 1, abort_flag,
                                       p.status, 0x10000000u | g);
          return w;
        };
        int J = pw - rot;
        if (J < 0) J += kProdWarps;
        for (; ok && J < njobs; J += kProdWarps) {
          if (J < mjobs) {
            const MainJob mj = main_job(J, parts, G);
            const RowJob jb = row_job(mj.row, ss, q, p, nrows, E, S2, CL);
            switch (mj.ngroups) {
              case 1: ok = fill_row<PREC, E, 1, CL>(p.x, jb, mj.c0, cstride, ss.iw0, p.W, p.C, stage, lo_off, lane, amax, s2sub, wait_stage); break;
              case 2: ok = fill_row<PREC, E, 2, CL>(p.x, jb, mj.c0, cstride, ss.iw0, p.W, p.C, stage, lo_off, lane, amax, s2sub, wait_stage); break;
              case 3: ok = fill_row<PREC, E, 3, CL>(p.x, jb, mj.c0, cstride, ss.iw0, p.W, p.C, stage, lo_off, lane, amax, s2sub, wait_stage); break;
              default: ok = fill_row<PREC, E, 4, CL>(p.x, jb, mj.c0, cstride, ss.iw0, p.W, p.C, stage, lo_off, lane, amax, s2sub, wait_stage); break;
            }
          } else {
            // lane -> (row job, tail pixel) pair
            const int l = (J - mjobs) * 32 + lane;
            const int job = l / tail;
            const int cc = 32 * G + (l - job * tail);
            float v[E];
            RowJob jb;
            if (job < jobs) {
              jb = row_job(job, ss, q, p, nrows, E, S2, CL);
              load_pixel<E, CL>(p.x, jb, cc, cstride, ss.iw0, p.W, p.C, v);
            }
            ok = wait_stage();
            if (ok && job < jobs) {
              const uint32_t o = jb.dst + (uint32_t)col_px(cc, s2sub) * 16u;
              store_slice<PREC, E>(stage + o, stage + lo_off + o, v, amax);
            }
          }
        }
        if (!ok || !wait_stage()) {
          ok = false;
          break;
        }
        rot += njobs % kProdWarps;
        if (rot >= kProdWarps) rot -= kProdWarps;
        if (++ps == q.S) { ps = 0; pph ^= 1; }
        if (++psb == q.SB) { psb = 0; psbph ^= 1; }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {  // (CTA pairs: the even CTA's barrier)
          if constexpr (PAIR) ptx::mbar_arrive_at(&a_full[s], 0);
          else ptx::mbar_arrive(&a_full[s]);
        }
      }
    }
    }  // !db_done
    if (amax >= 65520.0f) atomicOr(p.status, ST_RANGE);  // some hi part overflowed
    atomicMax(&ctl->amax_bits, __float_as_uint(amax));    // |x| >= 0: bits order as values
    // drain outstanding weight copies before the CTA can exit
    if (pt == 0 && q.b_resident) wait_bar(bars, B_FULL, 0, abort_flag, p.status, 0x12000000u);
    if (lane == 0 && last_b != 0xffffffffu)
      wait_bar(bars, B_FULL + (int)(last_b % q.SB), (last_b / q.SB) & 1, abort_flag, p.status,
               0x13000000u | last_b);
    }  // register-load producers
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issue
    // Every MMA and commit comes from the same (lowest) lane -- elect.sync
    // picks it each time -- so each commit tracks all MMAs before it.
    const uint32_t sbase = ptx::smem_u32(smem);
    // per-K-step A descriptor deltas, constant for the launch, kept in
    // registers (every index below is a compile-time constant)
    uint32_t kdr[28];
#pragma unroll
    for (int i = 0; i < 28; ++i) kdr[i] = ctl->kdelta[i];
    uint32_t kcr[9];  // parity-class K steps (SP): class | first << 7
#pragma unroll
    for (int i = 0; i < 9; ++i) kcr[i] = SP ? ctl->kcls[i] : 0u;
    const uint32_t lo_delta = (uint32_t)((q.P * q.plane_bytes) >> 4);  // hi -> lo planes
    const uint32_t tile_delta = (uint32_t)((q.R * q.RS * 16) >> 4);    // next M tile
    uint32_t g = 0, gb = 0, it = 0;
    // ring positions as counters (no integer division in the issue loop):
    // accumulator macc of phase mpar, stage ms of phase mph, weight slot msb
    int macc = 0, ms = 0, msb = 0;
    uint32_t mpar = 0, mph = 0, msbph = 0;
    // The tensor pipe queues only a few MMAs, so any stall of this warp
    // between bursts idles it.  Right after issuing a chunk the warp tests
    // (without blocking) the barriers the next chunk and the next unit will
    // wait on, while the queued MMAs run; a barrier seen complete then needs
    // no wait.
    bool pre_full = false, pre_acc = false;
    bool ok = true;
    if (q.b_resident) ok = wait_bar_warp(bars, B_FULL, 0, abort_flag, p.status, 0x20000000u);
    if constexpr (!SP) {
      // every other entry: one thread issues all units (CTA pairs: the even
      // CTA's, for both CTAs' tiles)
      if (ok && rank == 0) {
        int r = 1;
        if (ptx::elect_one())
          r = issue_units<PREC, U, POOL, !CL, PAIR>(q, units, sbase, tmem, bars, ctl->kdelta,
                                                    lo_delta, tile_delta, abort_flag, p.status)
                  ? 1 : 0;
        __syncwarp();
        ok = __shfl_sync(0xffffffffu, r, 0) != 0;
      }
    } else {
    // Parity-class pooled units (stride-2 transposed conv): the warp stays
    // converged and issues under elect.sync.
    for (long u = blockIdx.x; ok && u < units; u += gridDim.x, ++it) {
      const int cb = (int)fdiv((uint32_t)u, q.fd_cb);
      const int acc = macc;
      const uint32_t acc_par = mpar ^ 1;
      if (++macc == q.NACC) { macc = 0; mpar ^= 1; }
      if (!pre_acc && !wait_bar_warp(bars, ACC_EMPTY + acc, acc_par,
                                     abort_flag, p.status, 0x21000000u | it))
        break;
      ptx::tc_fence_after();
      if constexpr (SP) {
        if (q.SPLIT) {
          // half A (classes (0,0), (0,1)) over every chunk, then half B; the
          // generic wait above freed half A; a chunk's stage is released
          // after its half-B MMAs
          const int s0 = ms;
          const uint32_t ph0 = mph;
          int s = s0;
          uint32_t ph = ph0;
          for (int c = 0; ok && c < q.NCH; ++c) {
            if (!(c == 0 && pre_full) &&
                !wait_bar_warp(bars, A_FULL + s, ph, abort_flag, p.status, 0x22000000u | (g + c)))
              ok = false;
            ptx::tc_fence_after();
            const uint32_t a_lo = ((sbase + (uint32_t)(s * q.a_stage_bytes)) >> 4) & 0x3FFFu;
            const uint32_t bb = sbase + q.off_b + (uint32_t)(((long)cb * q.NCH + c) * q.b_chunk_bytes);
            const uint32_t b_lo = ((bb >> 4) & 0x3FFFu) | ((2048u >> 4) << 16);
            if (ok) {
              if (q.KS == 5) issue_subpix<PREC, 0, 2>(kdr, kcr, a_lo, b_lo, tmem, lo_delta, c == 0);
              else issue_subpix<PREC, 0, 3>(kdr, kcr, a_lo, b_lo, tmem, lo_delta, c == 0);
            }
            if (++s == q.S) { s = 0; ph ^= 1; }
          }
          if (!ok) break;
          if (ptx::elect_one()) ptx::tc_commit(&acc_full[0]);
          __syncwarp();
          if (!wait_bar_warp(bars, ACC_EMPTY + 1, acc_par, abort_flag, p.status, 0x21100000u | it)) break;
          ptx::tc_fence_after();
          s = s0;
          ph = ph0;
          for (int c = 0; c < q.NCH; ++c) {
            const uint32_t a_lo = ((sbase + (uint32_t)(s * q.a_stage_bytes)) >> 4) & 0x3FFFu;
            const uint32_t bb = sbase + q.off_b + (uint32_t)(((long)cb * q.NCH + c) * q.b_chunk_bytes);
            const uint32_t b_lo = ((bb >> 4) & 0x3FFFu) | ((2048u >> 4) << 16);
            if (q.KS == 5) issue_subpix<PREC, 2, 5>(kdr, kcr, a_lo, b_lo, tmem, lo_delta, c == 0);
            else issue_subpix<PREC, 3, 9>(kdr, kcr, a_lo, b_lo, tmem, lo_delta, c == 0);
            if (ptx::elect_one()) ptx::tc_commit(&a_empty[s]);
            __syncwarp();
            if (++s == q.S) { s = 0; ph ^= 1; }
          }
          ms = s;
          mph = ph;
          g += (uint32_t)q.NCH;
          pre_full = __all_sync(0xffffffffu, ptx::mbar_test_wait(&a_full[ms], mph));
          pre_acc = __all_sync(0xffffffffu, ptx::mbar_test_wait(&acc_empty[0], mpar ^ 1));
          if (ptx::elect_one()) ptx::tc_commit(&acc_full[1]);
          __syncwarp();
          continue;
        }
      }
      for (int c = 0; c < q.NCH; ++c, ++g) {
        const int s = ms;
        const uint32_t sph = mph;
        if (++ms == q.S) { ms = 0; mph ^= 1; }
        if (!pre_full && !wait_bar_warp(bars, A_FULL + s, sph, abort_flag, p.status, 0x22000000u | g)) {
          ok = false;
          break;
        }
        uint32_t bbase;
        int sb = 0;
        if (q.b_resident) {
          bbase = sbase + q.off_b + (uint32_t)(((long)cb * q.NCH + c) * q.b_chunk_bytes);
        } else {
          sb = msb;
          if (!wait_bar_warp(bars, B_FULL + sb, msbph, abort_flag, p.status, 0x23000000u | gb)) {
            ok = false;
            break;
          }
          bbase = sbase + q.off_b + (uint32_t)(sb * q.b_chunk_bytes);
        }
        ptx::tc_fence_after();
        // low descriptor words of this stage / weight chunk (start address
        // and leading byte offset); the high word is the same for all
        const uint32_t a_lo = ((sbase + (uint32_t)(s * q.a_stage_bytes)) >> 4) & 0x3FFFu;
        const uint32_t b_lo = ((bbase >> 4) & 0x3FFFu) | ((2048u >> 4) << 16);
        const uint32_t dacc = tmem + (uint32_t)(acc * U * 128);
        if (q.KS == 5) issue_subpix<PREC, 0, 5>(kdr, kcr, a_lo, b_lo, dacc, lo_delta, c == 0);
        else issue_subpix<PREC, 0, 9>(kdr, kcr, a_lo, b_lo, dacc, lo_delta, c == 0);
        // look ahead while the MMAs just issued run
        pre_full = __all_sync(0xffffffffu, ptx::mbar_test_wait(&a_full[ms], mph));
        if (c == q.NCH - 1)
          pre_acc = __all_sync(0xffffffffu, ptx::mbar_test_wait(&acc_empty[macc], mpar ^ 1));
        if (ptx::elect_one()) {
          ptx::tc_commit(&a_empty[s]);
          if (!q.b_resident) ptx::tc_commit(&b_empty[sb]);
        }
        __syncwarp();
        if (!q.b_resident) {
          ++gb;
          if (++msb == q.SB) { msb = 0; msbph ^= 1; }
        }
      }
      if (!ok) break;
      if (ptx::elect_one()) ptx::tc_commit(&acc_full[acc]);
      __syncwarp();
    }
    }  // parity-class units
    // wait until every MMA this warp issued has completed
    if (rank == 0) {
      if (ptx::elect_one()) {
        if constexpr (PAIR) ptx::tc_commit2(drain, 1);
        else ptx::tc_commit(drain);
      }
      __syncwarp();
      wait_bar_warp(bars, DRAIN, 0, abort_flag, p.status, 0x24000000u);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    if constexpr (PREC == 1) {
      // Bottom of the fp16 split's range: below 2^-14 the hi part of a value
      // is subnormal and below 2^-24 it vanishes, so data whose largest
      // magnitude is under 2^-12 would lose relative accuracy.  The largest
      // |w| (per-block maxima from the weight pack) is checked here, by one
      // warp of CTA 0 while it waits for its first accumulator; each CTA's
      // staged x at the end.  All-zero data is exact and not flagged.
      if (blockIdx.x == 0 && warp == kEpiWarps - 1 && p.wmax) {
        float wm = 0.0f;
#pragma unroll 8
        for (int i = lane; i < p.wmax_n; i += 32) wm = fmaxf(wm, __ldg(p.wmax + i));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
        if (lane == 0 && wm > 0.0f && wm < kF16SplitMin) atomicOr(p.status, ST_RANGE);
      }
    }
    // Warp w reads TMEM lane quadrant w % 4 (one output pixel per lane) and
    // channel half w / 4 (32 of the 64 channels; all 64 with 4 warps).
    const int quad = warp & 3, half = warp >> 2;
    const int m = quad * 32 + lane;  // TMEM lane = M row = output pixel
    const int m_row = m / q.RS, m_col = m - m_row * q.RS;  // staged row / column of m
    const float scale = PREC ? (1.0f / 2048.0f) : 1.0f;
    uint32_t it = 0;
    int eacc = 0;  // accumulator eacc of phase epar, as counters
    uint32_t epar = 0;
    for (long u = blockIdx.x; u < units; u += gridDim.x, ++it) {
      const UnitPos up = decode_unit(u, q);
      const int acc = eacc;
      const uint32_t acc_par = epar;
      if (++eacc == q.NACC) { eacc = 0; epar ^= 1; }
      if constexpr (POOL) {
        bool okw = wait_bar_warp(bars, ACC_FULL + acc, acc_par, abort_flag, p.status, 0x30000000u | it);
        okw = epi_all<kEpiThreads>(okw);
        if (!okw) break;
        ptx::tc_fence_after();
      }
      const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
      const int co_base = up.cb * 64;
      const int ch0 = half * 32;  // first channel (within the block) of this warp
      if constexpr (!POOL) {
        const int r = m_row, c = m_col;
        const int ow = up.ct * q.WT + c;
        const long plane = (long)p.Ho * p.Wo;
        const long cstride = (long)p.Do * plane;
        const int nco = p.CO - co_base - ch0;  // channels of this warp that exist
        bool okt = true;
#pragma unroll 1
        for (int t = 0; t < U; ++t) {  // the unit's M tiles, R output rows each
          if (!wait_bar_warp(bars, ACC_FULL + acc * U + t, acc_par, abort_flag, p.status,
                             0x30000000u | ((uint32_t)t << 20) | (it & 0xFFFFFu))) {
            okt = false;
            break;
          }
          ptx::tc_fence_after();
          const int oh = (up.rt * U + t) * q.R + r;
          const bool valid = r < q.R && c < q.WT && oh < p.Ho && ow < p.Wo;
          const uint32_t col0 = (uint32_t)((acc * U + t) * 128 + ch0);
          // Heavy chains (GELU, the general chain): the warp's 32 channels of
          // this tile leave tensor memory at once, are combined (hi + scale lo)
          // in registers and the accumulator is released before the chain and
          // the stores, so a later unit's MMAs overlap them (measured: conv3d
          // + GELU chain 0.653 -> 0.639 ms).  Light chains keep two loads of 16
          // channels and release after the stores (conv2d + ReLU + HardSwish
          // 0.122 ms, 0.133 ms with the early release).
          constexpr bool kEarly = CHAIN == CHAIN_LEAKY_ADD_CLAMP1_GELU ||
                                  CHAIN == CHAIN_LEAKY_ADD_CLAMP_GELU || CHAIN == CHAIN_GENERIC;
          float acc32[32];
          auto load_sums = [&](int c0, int n16) {
            uint32_t h0[16], l0[16], h1[16], l1[16];
            ptx::tmem_ld16(tl + col0 + c0, h0);
            ptx::tmem_ld16(tl + col0 + 64 + c0, l0);
            if (n16 == 2) {
              ptx::tmem_ld16(tl + col0 + c0 + 16, h1);
              ptx::tmem_ld16(tl + col0 + 80 + c0, l1);
            }
            ptx::tmem_wait_ld();
            const uint64_t sc2 = ptx::pk2(scale, scale);
#pragma unroll
            for (int j = 0; j < 16; j += 2)
              ptx::upk2(ptx::fma2(sc2, ptx::pk2(__uint_as_float(l0[j]), __uint_as_float(l0[j + 1])),
                                  ptx::pk2(__uint_as_float(h0[j]), __uint_as_float(h0[j + 1]))),
                        acc32[c0 + j], acc32[c0 + j + 1]);
            if (n16 == 2) {
#pragma unroll
              for (int j = 0; j < 16; j += 2)
                ptx::upk2(ptx::fma2(sc2, ptx::pk2(__uint_as_float(l1[j]), __uint_as_float(l1[j + 1])),
                                    ptx::pk2(__uint_as_float(h1[j]), __uint_as_float(h1[j + 1]))),
                          acc32[c0 + 16 + j], acc32[c0 + 16 + j + 1]);
            }
          };
          auto release = [&]() {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&acc_empty[acc * U + t]);
          };
          if constexpr (kEarly) {
            load_sums(0, 2);
            release();
          }
          float *yp = p.y + (((long)up.n * p.CO + co_base + ch0) * p.Do + up.od) * plane +
                      (long)oh * p.Wo + ow;
#pragma unroll
          for (int cc = 0; cc < 32; cc += 16) {
            if constexpr (!kEarly) load_sums(cc, 1);
            float *v = acc32 + cc;  // conv sums of channels cc .. cc + 15 (no bias yet)
            float bv[16], av[16];
            const float *sb = &ctl->bias[co_base + ch0 + cc];
            const float *sa = &ctl->addend[co_base + ch0 + cc];
  #pragma unroll
            for (int j = 0; j < 16; j += 4) {
              *reinterpret_cast<float4 *>(&bv[j]) = *reinterpret_cast<const float4 *>(sb + j);
              if constexpr (CHAIN == CHAIN_LEAKY_ADD_CLAMP_GELU || CHAIN == CHAIN_LEAKY_ADD_CLAMP1_GELU)
                *reinterpret_cast<float4 *>(&av[j]) = *reinterpret_cast<const float4 *>(sa + j);
              else
                av[j] = av[j + 1] = av[j + 2] = av[j + 3] = 0.0f;
            }
            float o[16];
            if constexpr (CHAIN == CHAIN_GENERIC) {
  #pragma unroll
              for (int j = 0; j < 16; ++j) o[j] = v[j] + bv[j];
              apply_chain_generic_n<16>(p.epi, co_base + ch0 + cc, nco - cc, o);
            } else if constexpr (CHAIN == CHAIN_RELU_HARDSWISH ||
                                 CHAIN == CHAIN_LEAKY_ADD_CLAMP1_GELU) {
  #pragma unroll
              for (int j = 0; j < 16; j += 2)  // channel pairs on the paired fp32 pipe
                apply_chain2x<CHAIN>(p.epi, v[j], v[j + 1], bv[j], bv[j + 1], av[j], av[j + 1],
                                     o[j], o[j + 1]);
            } else {
  #pragma unroll
              for (int j = 0; j < 16; ++j)
                o[j] = apply_chain<CHAIN>(p.epi, co_base + ch0 + cc + j, v[j] + bv[j], av[j]);
            }
            if constexpr (CL) {
              // channels-last output: this pixel's 16 channels are adjacent
              if (valid) {
                float *yc = p.y + ((((long)up.n * p.Do + up.od) * p.Ho + oh) * p.Wo + ow) * p.CO +
                            co_base + ch0 + cc;
                if (cc + 16 <= nco && (p.CO & 3) == 0) {  // 16-byte aligned vectors
  #pragma unroll
                  for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4 *>(yc + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
                } else {
  #pragma unroll
                  for (int j = 0; j < 16; ++j)
                    if (cc + j < nco) yc[j] = o[j];
                }
              }
            } else {
              float *yc = yp + (long)cc * cstride;
              if (valid && cc + 16 <= nco) {  // all 16 channels exist: no per-channel test
  #pragma unroll
                for (int j = 0; j < 16; ++j) {
                  *yc = o[j];
                  yc += cstride;
                }
              } else if (valid) {
  #pragma unroll
                for (int j = 0; j < 16; ++j) {
                  if (cc + j < nco) *yc = o[j];
                  yc += cstride;
                }
              }
            }
          }
          if constexpr (!kEarly) release();
        }
        if (!okt) break;
      } else if constexpr (GP) {
        // General max pool: lane m is conv column m of the tile; the row
        // maximum over the unit's U conv rows (the pooled row's window rows)
        // goes to shared memory, the accumulator is released, and the 256
        // epilogue threads take the windows across columns there.
        float *xb = reinterpret_cast<float *>(smem + q.off_xb);  // [64 channels][kXbPitch]
#pragma unroll 1
        for (int cc = 0; cc < 32; cc += 16) {
          float mx[16];
#pragma unroll 1
          for (int t = 0; t < U; ++t) {
            uint32_t h0[16], l0[16];
            const uint32_t col = (uint32_t)((acc * U + t) * 128 + ch0 + cc);
            ptx::tmem_ld16(tl + col, h0);
            ptx::tmem_ld16(tl + col + 64, l0);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float v = fmaf(scale, __uint_as_float(l0[j]), __uint_as_float(h0[j]));
              mx[j] = t ? fmaxf(mx[j], v) : v;
            }
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) xb[(ch0 + cc + j) * kXbPitch + m] = mx[j];
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&acc_empty[acc]);
        epi_sync<kEpiThreads>();
        // windows: thread (jq, ch) takes pooled columns jq, jq + 4, ... of
        // channel ch in increasing order; the bias is common to a window, so
        // it is added after the max (x -> x + b is monotone in fp32)
        const int et = warp * 32 + lane;  // 0 .. 255
        const int ch = et & 63, jq = et >> 6;
        const int Wp = (p.Wo - p.pk) / p.ps + 1;
        const float bias = ctl->bias[co_base + ch];
        float sum = 0.0f;
        for (int j = jq; j < q.PJ; j += 4) {
          if (up.ct * q.PJ + j >= Wp) break;
          const float *w = xb + ch * kXbPitch + j * p.ps;
          float mxw = w[0];
          for (int a = 1; a < p.pk; ++a) mxw = fmaxf(mxw, w[a]);
          sum += fminf(fmaxf(mxw + bias, p.ht_lo), p.ht_hi);
        }
        ctl->red[jq][ch] = sum;
        epi_sync<kEpiThreads>();
        if (et < 64) {
          const int T = q.n_rt * q.n_ct;
          const int t = up.rt * q.n_ct + up.ct;
          const int co = co_base + et;
          if (co < p.CO)
            partial[((long)up.n * T + t) * p.CO + co] =
                ((ctl->red[0][et] + ctl->red[1][et]) + ctl->red[2][et]) + ctl->red[3][et];
        }
        epi_sync<kEpiThreads>();
      } else if constexpr (SP) {
        // lane m = pooled pixel (rt R + m_row, ct WT + m_col); the 2x2 window
        // is the four class accumulators of that lane
        const int pi = up.rt * q.R + m_row, pj = up.ct * q.WT + m_col;
        const bool valid = m_row < q.R && m_col < q.WT && pi < p.Ho / 2 && pj < p.Wo / 2;
        if (q.SPLIT) {
          // half A (classes (0,0), (0,1), columns 0-255) is ready (waited
          // above); its max is kept while half B is computed
          float keep[2][16];
#pragma unroll
          for (int g2 = 0; g2 < 2; ++g2) {
            const int cc = g2 * 16;
            uint32_t h0[16], l0[16], h1[16], l1[16];
            ptx::tmem_ld16(tl + (uint32_t)(ch0 + cc), h0);
            ptx::tmem_ld16(tl + (uint32_t)(64 + ch0 + cc), l0);
            ptx::tmem_ld16(tl + (uint32_t)(128 + ch0 + cc), h1);
            ptx::tmem_ld16(tl + (uint32_t)(192 + ch0 + cc), l1);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j)
              keep[g2][j] = fmaxf(fmaf(scale, __uint_as_float(l0[j]), __uint_as_float(h0[j])),
                                  fmaf(scale, __uint_as_float(l1[j]), __uint_as_float(h1[j])));
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&acc_empty[0]);
          bool okw = wait_bar_warp(bars, ACC_FULL + 1, acc_par, abort_flag, p.status, 0x30100000u | it);
          okw = epi_all<kEpiThreads>(okw);
          if (!okw) break;
          ptx::tc_fence_after();
#pragma unroll
          for (int g2 = 0; g2 < 2; ++g2) {
            const int cc = g2 * 16;
            uint32_t h0[16], l0[16], h1[16], l1[16];
            ptx::tmem_ld16(tl + (uint32_t)(256 + ch0 + cc), h0);
            ptx::tmem_ld16(tl + (uint32_t)(320 + ch0 + cc), l0);
            ptx::tmem_ld16(tl + (uint32_t)(384 + ch0 + cc), h1);
            ptx::tmem_ld16(tl + (uint32_t)(448 + ch0 + cc), l1);
            ptx::tmem_wait_ld();
            float part[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              // bias is common to the four classes: added once after the max
              const float v = fmaxf(keep[g2][j],
                                    fmaxf(fmaf(scale, __uint_as_float(l0[j]), __uint_as_float(h0[j])),
                                          fmaf(scale, __uint_as_float(l1[j]), __uint_as_float(h1[j]))));
              const float bias = ctl->bias[co_base + ch0 + cc + j];
              part[j] = valid ? fminf(fmaxf(v + bias, p.ht_lo), p.ht_hi) : 0.0f;
            }
            lane_sum16(part, lane);
            if ((lane & 1) == 0) ctl->red[quad][ch0 + cc + ((lane >> 1) & 15)] = part[0];
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&acc_empty[1]);
          epi_sync<kEpiThreads>();
          if (warp == 0) {
            const int T = q.n_rt * q.n_ct;
            const int t = up.rt * q.n_ct + up.ct;
            float *dst = partial + ((long)up.n * T + t) * p.CO;
            for (int j = lane; j < 64; j += 32) {
              const int co = co_base + j;
              if (co < p.CO)
                dst[co] = ((ctl->red[0][j] + ctl->red[1][j]) + ctl->red[2][j]) + ctl->red[3][j];
            }
          }
          epi_sync<kEpiThreads>();
          continue;
        }
#pragma unroll 1
        for (int cc = 0; cc < 32; cc += 16) {
          float mx[16], bv[16];
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4 *>(&bv[j]) =
                *reinterpret_cast<const float4 *>(&ctl->bias[co_base + ch0 + cc + j]);
#pragma unroll 1
          for (int cls = 0; cls < 4; cls += 2) {  // two classes per tensor-memory wait
            uint32_t h0[16], l0[16], h1[16], l1[16];
            ptx::tmem_ld16(tl + (uint32_t)(cls * 128 + ch0 + cc), h0);
            ptx::tmem_ld16(tl + (uint32_t)(cls * 128 + 64 + ch0 + cc), l0);
            ptx::tmem_ld16(tl + (uint32_t)(cls * 128 + 128 + ch0 + cc), h1);
            ptx::tmem_ld16(tl + (uint32_t)(cls * 128 + 192 + ch0 + cc), l1);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float v0 = fmaf(scale, __uint_as_float(l0[j]), __uint_as_float(h0[j])) + bv[j];
              const float v1 = fmaf(scale, __uint_as_float(l1[j]), __uint_as_float(h1[j])) + bv[j];
              const float v = fmaxf(v0, v1);
              mx[j] = cls ? fmaxf(mx[j], v) : v;
            }
          }
          float part[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            part[j] = valid ? fminf(fmaxf(mx[j], p.ht_lo), p.ht_hi) : 0.0f;
          lane_sum16(part, lane);
          if ((lane & 1) == 0) ctl->red[quad][ch0 + cc + ((lane >> 1) & 15)] = part[0];
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&acc_empty[acc]);
        epi_sync<kEpiThreads>();
        if (warp == 0) {
          const int T = q.n_rt * q.n_ct;
          const int t = up.rt * q.n_ct + up.ct;
          float *dst = partial + ((long)up.n * T + t) * p.CO;
          for (int j = lane; j < 64; j += 32) {
            const int co = co_base + j;
            if (co < p.CO)
              dst[co] = ((ctl->red[0][j] + ctl->red[1][j]) + ctl->red[2][j]) + ctl->red[3][j];
          }
        }
        epi_sync<kEpiThreads>();
      } else {
        const int c = m;  // one output row per M tile
        const int ow = up.ct * q.WT + c;
        const bool valid = ((c & 1) == 0) && (c + 1 < q.WT) && (ow + 1 < p.Wo);
        const uint32_t col0 = (uint32_t)(acc * 256 + ch0);
        constexpr int kWarpCh = 256 / kEpiWarps;  // channels of this warp: 64 (4 warps)
#pragma unroll 1
        for (int cc = 0; cc < kWarpCh; cc += 16) {
          uint32_t h0[16], l0[16], h1[16], l1[16];
          ptx::tmem_ld16(tl + col0 + cc, h0);
          ptx::tmem_ld16(tl + col0 + 64 + cc, l0);
          ptx::tmem_ld16(tl + col0 + 128 + cc, h1);
          ptx::tmem_ld16(tl + col0 + 192 + cc, l1);
          ptx::tmem_wait_ld();
          float part[16], bv[16];
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4 *>(&bv[j]) =
                *reinterpret_cast<const float4 *>(&ctl->bias[co_base + ch0 + cc + j]);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float bias = bv[j];
            const float v0 = fmaf(scale, __uint_as_float(l0[j]), __uint_as_float(h0[j])) + bias;
            const float v1 = fmaf(scale, __uint_as_float(l1[j]), __uint_as_float(h1[j])) + bias;
            float mx = fmaxf(v0, v1);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fminf(fmaxf(mx, p.ht_lo), p.ht_hi);
            part[j] = valid ? mx : 0.0f;
          }
          // Sum over the warp's 32 pixels by halving exchanges: at each step a
          // lane keeps half of its channels and adds its partner's sums of
          // them.  Lane l ends with channel (l >> 1) & 15.
          lane_sum16(part, lane);
          if ((lane & 1) == 0) ctl->red[quad][ch0 + cc + ((lane >> 1) & 15)] = part[0];
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {  // (CTA pairs: the even CTA's barrier)
          if constexpr (PAIR) ptx::mbar_arrive_at(&acc_empty[acc], 0);
          else ptx::mbar_arrive(&acc_empty[acc]);
        }
        epi_sync<kEpiThreads>();
        if (warp == 0) {
          const int T = q.n_rt * q.n_ct;
          const int t = up.rt * q.n_ct + up.ct;
          float *dst = partial + ((long)up.n * T + t) * p.CO;
          for (int j = lane; j < 64; j += 32) {
            const int co = co_base + j;
            if (co < p.CO)
              dst[co] = ((ctl->red[0][j] + ctl->red[1][j]) + ctl->red[2][j]) + ctl->red[3][j];
          }
        }
        epi_sync<kEpiThreads>();
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  // CTA pairs: neither CTA leaves (nor frees its half of the tensor memory)
  // before the other is done with its shared memory and barriers
  if constexpr (PAIR) ptx::cluster_sync();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) {
    if constexpr (PAIR) ptx::tmem_dealloc2(tmem, (uint32_t)q.tmem_cols);
    else ptx::tmem_dealloc(tmem, (uint32_t)q.tmem_cols);
  }
  if constexpr (PREC == 1) {
    // Bottom of the fp16 split's range (see the weights' check above): this
    // CTA's staged x
    if (tid == kProdWarp0 * 32) {
      const float xm = __uint_as_float(ctl->amax_bits);
      if (xm > 0.0f && xm < kF16SplitMin) atomicOr(p.status, ST_RANGE);
    }
  }
}

// Failure-detection self-test: warp 0 waits, with a limit of `limit_ns`, on
// an mbarrier whose phase nothing completes; it gives up, records the wait
// (tag 0x71000001) and raises the block's abort flag.  Warp 1 waits on a
// second such barrier under the kernels' normal limit and gives up as soon
// as it sees the flag (record tag 0x71000002 | 0x08000000).  No fault, no
// hang: both waits are bounded and nothing else is in flight.
__global__ void selftest_wait_kernel(unsigned int *status, uint64_t limit_ns) {
  __shared__ uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars[0], 1);
    ptx::mbar_init(&bars[1], 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  volatile int *ab = &abort_flag;
  if (threadIdx.x < 32)
    wait_bar_warp(bars, 0, 0, ab, status, 0x71000001u, limit_ns);
  else
    wait_bar_warp(bars, 1, 0, ab, status, 0x71000002u);
  __syncthreads();
}

// cuTensorMapEncodeTiled, looked up once through the runtime (no link
// against the driver library).
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;

cudaError_t encode_fn() {
  if (g_encode_tiled) return cudaSuccess;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult qr;
  const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &qr);
  if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
  g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return cudaSuccess;
}

// Geometry of the tensor map of x for the tensor-copy staging (fp32):
// channels-first dims W, H, [D,] C, N with box BW x RIN x [1 x] chunk_ci;
// channels-last dims C, W, H, [D,] N with box chunk_ci x LW x RIN [x 1].
// The 3-D entry points always use the rank-5 form (a depth axis), whatever
// the kernel depth.  Strides in bytes for dims 1.. (dim 0 is contiguous).
struct XMapGeom {
  int rank;
  uint64_t dims[5], strides[4];
  uint32_t box[5];
};

XMapGeom x_map_geometry(const ConvProblem &p, const TcPlan &q) {
  XMapGeom g{};
  const bool d3 = p.entry == 1;
  const uint64_t C = p.C, D = p.D, H = p.H, W = p.W, N = p.N;
  if (!p.cl) {
    g.dims[0] = W; g.dims[1] = H;
    g.box[0] = q.BW; g.box[1] = q.RIN;
    if (d3) {
      g.dims[2] = D; g.dims[3] = C; g.dims[4] = N;
      g.box[2] = 1; g.box[3] = q.chunk_ci; g.box[4] = 1;
      g.rank = 5;
    } else {
      g.dims[2] = C; g.dims[3] = N;
      g.box[2] = q.chunk_ci; g.box[3] = 1;
      g.rank = 4;
    }
  } else {
    g.dims[0] = C; g.dims[1] = W; g.dims[2] = H;
    g.box[0] = q.chunk_ci; g.box[1] = q.LW; g.box[2] = q.RIN;
    if (d3) {
      g.dims[3] = D; g.dims[4] = N;
      g.box[3] = 1; g.box[4] = 1;
      g.rank = 5;
    } else {
      g.dims[3] = N;
      g.box[3] = 1;
      g.rank = 4;
    }
  }
  uint64_t st = 4;
  for (int i = 0; i < g.rank - 1; ++i) {
    st *= g.dims[i];
    g.strides[i] = st;
  }
  return g;
}

// The tensor map itself: zeros outside the tensor, no swizzle.
cudaError_t make_x_map(const ConvProblem &p, const TcPlan &q, CUtensorMap *m) {
  cudaError_t e = encode_fn();
  if (e != cudaSuccess) return e;
  const XMapGeom g = x_map_geometry(p, q);
  cuuint64_t dims[5], strides[4];
  cuuint32_t box[5], es[5] = {1, 1, 1, 1, 1};
  for (int i = 0; i < g.rank; ++i) {
    dims[i] = g.dims[i];
    box[i] = g.box[i];
    if (i < g.rank - 1) strides[i] = g.strides[i];
  }
  const CUresult r = g_encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)g.rank,
                                    const_cast<float *>(p.x), dims, strides, box, es,
                                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int g_num_sms = 0;

template <int PREC, int CHAIN, bool POOL, int U, bool S2 = false, bool SP = false, bool CL = false,
          bool GP = false, bool PAIR = false>
cudaError_t launch_kernel(const ConvProblem &p, const TcPlan &q, const uint8_t *bimg,
                          float *partial, const CUtensorMap &tm, cudaStream_t s) {
  auto kern = tc_conv_kernel<PREC, CHAIN, POOL, U, S2, SP, CL, GP, PAIR>;
  const int smem = q.smem_bytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (!g_num_sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 148;
  }
  long grid = q.units < g_num_sms ? q.units : g_num_sms;
  prof_begin(s);
  if constexpr (PAIR) {
    // clusters of two CTAs; units 2k and 2k + 1 go to the two CTAs of a pair
    grid &= ~1L;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p, q, bimg, partial, tm);
  } else {
    kern<<<(unsigned)grid, kThreads, smem, s>>>(p, q, bimg, partial, tm);
    e = cudaGetLastError();
  }
  prof_end(s, p.entry);
  return e;
}

template <int PREC, int U, bool S2, bool CL = false>
cudaError_t launch_chain(const ConvProblem &p, const TcPlan &q, const uint8_t *bimg,
                         float *partial, const CUtensorMap &tm, cudaStream_t s) {
  switch (p.chain) {
    case CHAIN_NONE: return launch_kernel<PREC, CHAIN_NONE, false, U, S2, false, CL>(p, q, bimg, partial, tm, s);
    case CHAIN_RELU_HARDSWISH:
      return launch_kernel<PREC, CHAIN_RELU_HARDSWISH, false, U, S2, false, CL>(p, q, bimg, partial, tm, s);
    case CHAIN_LEAKY_ADD_CLAMP_GELU:
      return launch_kernel<PREC, CHAIN_LEAKY_ADD_CLAMP_GELU, false, U, S2, false, CL>(p, q, bimg, partial, tm, s);
    case CHAIN_LEAKY_ADD_CLAMP1_GELU:
      return launch_kernel<PREC, CHAIN_LEAKY_ADD_CLAMP1_GELU, false, U, S2, false, CL>(p, q, bimg, partial, tm, s);
    default: return launch_kernel<PREC, CHAIN_GENERIC, false, U, S2, false, CL>(p, q, bimg, partial, tm, s);
  }
}

template <int PREC>
cudaError_t launch_prec(const ConvProblem &p, const TcPlan &q, const uint8_t *bimg,
                        float *partial, const CUtensorMap &tm, cudaStream_t s) {
  if (p.subpix) return launch_kernel<PREC, CHAIN_NONE, true, 1, false, true>(p, q, bimg, partial, tm, s);
  if (p.pool && q.GP) {  // general max pool: one tile per window row
    switch (q.U) {
      case 1: return launch_kernel<PREC, CHAIN_NONE, true, 1, false, false, false, true>(p, q, bimg, partial, tm, s);
      case 2: return launch_kernel<PREC, CHAIN_NONE, true, 2, false, false, false, true>(p, q, bimg, partial, tm, s);
      case 3: return launch_kernel<PREC, CHAIN_NONE, true, 3, false, false, false, true>(p, q, bimg, partial, tm, s);
      default: return launch_kernel<PREC, CHAIN_NONE, true, 4, false, false, false, true>(p, q, bimg, partial, tm, s);
    }
  }
  if (p.pool)
    return q.PAIR ? launch_kernel<PREC, CHAIN_NONE, true, 2, false, false, false, false, true>(
                        p, q, bimg, partial, tm, s)
                  : launch_kernel<PREC, CHAIN_NONE, true, 2>(p, q, bimg, partial, tm, s);
  // stride 2 (even / odd sub-plane staging) is its own instance, so the
  // stride-1 producer carries none of its index arithmetic
  if (q.S2)
    return q.U == 2 ? launch_chain<PREC, 2, true>(p, q, bimg, partial, tm, s)
                    : launch_chain<PREC, 1, true>(p, q, bimg, partial, tm, s);
  if (p.cl)  // channels-last input and output: its own instances
    return q.U == 2 ? launch_chain<PREC, 2, false, true>(p, q, bimg, partial, tm, s)
                    : launch_chain<PREC, 1, false, true>(p, q, bimg, partial, tm, s);
  return q.U == 2 ? launch_chain<PREC, 2, false>(p, q, bimg, partial, tm, s)
                  : launch_chain<PREC, 1, false>(p, q, bimg, partial, tm, s);
}

}  // namespace

bool tc_supported(const ConvProblem &p, int prec) { return make_plan(p, prec).ok != 0; }

int tc_uses_tma(const ConvProblem &p, int prec) {
  const TcPlan q = make_plan(p, prec);
  return q.ok && q.TMA;
}

cudaError_t selftest_wait_launch(unsigned int *status, uint64_t limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 64, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

size_t tc_weight_bytes(const ConvProblem &p) {
  if (!tc_kernel_ok(p)) return 0;
  size_t m = 0;
  for (int prec = 0; prec < 2; ++prec) {
    TcPlan q{};
    plan_chunks(p, prec, q);
    if (q.COB * 64 > kMaxCoTc) continue;
    const size_t b = (size_t)q.COB * q.NCH * q.b_chunk_bytes;
    if (b > m) m = b;
  }
  return m;
}

int tc_pool_tiles_per_image(const ConvProblem &p) {
  if (!p.pool) return 0;
  int m = 0;
  for (int prec = 0; prec < 2; ++prec) {
    TcPlan q = make_plan(p, prec);
    if (q.ok && q.n_rt * q.n_ct > m) m = q.n_rt * q.n_ct;
  }
  return m;
}

cudaError_t tc_launch(const ConvProblem &p, int prec, void *ws, const WsLayout &L,
                      cudaStream_t s, int *launches) {
  TcPlan q = make_plan(p, prec);
  if (!q.ok) return cudaErrorNotSupported;
  uint8_t *bimg = static_cast<uint8_t *>(ws) + L.tc_w;
  float *partial = reinterpret_cast<float *>(static_cast<char *>(ws) + L.partial);
  const long nelem = (long)q.COB * q.NCH * q.KS * 2 * 128 * q.E;
  int blocks = (int)((nelem + 255) / 256);
  if (blocks > kMaxPackBlocks) blocks = kMaxPackBlocks;
  ConvProblem pp = p;
  pp.wmax = reinterpret_cast<float *>(static_cast<char *>(ws) + L.wmax);
  pp.wmax_n = blocks;
  tc_pack_weights<<<blocks, 256, 0, s>>>(pp, q, bimg);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *launches = 1;
  CUtensorMap tm;
  memset(&tm, 0, sizeof(tm));
  if (q.TMA) {
    e = make_x_map(p, q, &tm);
    if (e != cudaSuccess) return e;
  }
  e = prec ? launch_prec<1>(pp, q, bimg, partial, tm, s) : launch_prec<0>(pp, q, bimg, partial, tm, s);
  if (e != cudaSuccess && q.PAIR) {
    // a cluster launch refused (no two free SMs of a pair, say): the same
    // units by single CTAs (same weight image, same partials)
    (void)cudaGetLastError();
    const TcPlan q1 = make_plan(p, prec, false);
    if (q1.ok)
      e = prec ? launch_prec<1>(pp, q1, bimg, partial, tm, s) : launch_prec<0>(pp, q1, bimg, partial, tm, s);
  }
  if (e != cudaSuccess) return e;
  *launches += 1;
  if (p.pool) {
    e = pool_finish_launch(p, partial, q.n_rt * q.n_ct, s);
    *launches += 1;
  }
  return e;
}

}  // namespace fc
