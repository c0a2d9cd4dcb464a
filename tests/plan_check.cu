// plan_check.cu -- host-only check of the tensor-core kernel's plans (test
// infrastructure; built and run by tests/test_plan_geometry.py, never part of
// the library).  For a set of shapes (stride 1 and 2, dilation 1 and 2, 2D
// and 3D, row-packed tiles and column strips, the pooled and the
// parity-class transposed convs) and both precisions it replays, on the
// host, (1) every producer store of a stage (the main / tail job split the
// kernel uses) and (2) every MMA operand address of every K step and M tile,
// and checks that each valid output row reads exactly the input pixel the
// convolution definition asks for (or a zero for padding), that nothing is
// written twice or read unwritten, and that the layout stays inside shared
// memory and the descriptor ranges.  Prints CHECK OK on success.
#include "../convolution_epilogue_gb300/csrc/fc_tc.cu"
#include <cstdio>
#include <vector>
namespace fc {
void prof_begin(cudaStream_t) {}
void prof_end(cudaStream_t, int) {}
cudaError_t pool_finish_launch(const ConvProblem &, const float *, int, cudaStream_t) { return cudaSuccess; }
}
using namespace fc;
static int fails = 0;
#define REQ(c, ...) do { if (!(c)) { if (fails < 40) { printf("FAIL: " __VA_ARGS__); printf("\n"); } ++fails; } } while (0)

struct Px { int id, ih, iw, plane; bool zero; };

void check_stage(const char *name, const ConvProblem &p, const TcPlan &q, int n, int od, int rt, int ct) {
  const long plane_px = q.plane_bytes / 16;
  const long tot_px = 2L * q.P * plane_px;
  std::vector<int> cnt(tot_px, 0);
  std::vector<Px> who(tot_px, Px{0, 0, 0, 0, true});
  StageSrc ss{};
  ss.xn = (long)n * p.C * p.D * p.H * p.W;
  ss.id0 = od * p.stride - p.pad_d;
  ss.ih0 = rt * q.ROWSTEP * p.stride - p.pad;
  ss.iw0 = ct * q.COLSTEP * p.stride - p.pad;
  ss.ci0 = 0;
  const int nrows = p.KD * q.RIN, jobs = q.P * nrows;
  const int s2sub = q.S2 ? q.SUB : 0;
  if (q.TMA) {
    // tensor-copy staging: replay the converters' items against the copy's
    // box layout (which x element each raw slot float holds)
    REQ(!q.S2 && !q.SP && q.LW == q.RS, "%s TMA plan geometry", name);
    const int iwt = ss.iw0 - (p.cl ? 0 : q.coff);
    REQ(p.cl || (iwt % 4 + 4) % 4 == 0, "%s tensor copy starts at column %d (not 16-byte aligned)",
        name, iwt);
    const int items = q.P * q.RIN * q.LW;
    // the tensor map: the box coordinates the loader passes (innermost
    // first, as in the kernel) and the map's strides must address the x
    // element the converter expects at every raw float
    const XMapGeom mg = x_map_geometry(p, q);
    REQ(mg.rank == (p.entry == 1 ? 5 : 4), "%s map rank", name);
    long boxn = 1;
    for (int i = 0; i < mg.rank; ++i) boxn *= mg.box[i];
    REQ(boxn * 4 == q.raw_tx, "%s box bytes %ld vs %d", name, boxn * 4, q.raw_tx);
    for (int kd = 0; kd < p.KD; ++kd) {
      const int id = ss.id0 + kd * p.dil;
      long c0[5];
      if (p.cl) { c0[0] = 0; c0[1] = iwt; c0[2] = ss.ih0; c0[3] = p.entry == 1 ? id : n; c0[4] = n; }
      else { c0[0] = iwt; c0[1] = ss.ih0; c0[2] = p.entry == 1 ? id : 0; c0[3] = p.entry == 1 ? 0 : n; c0[4] = n; }
      for (long f = 0; f < boxn; f += 7) {  // every 7th float of the box
        long rem = f, off = 0;
        bool inside = true;
        long co[5];
        for (int i = 0; i < mg.rank; ++i) {
          co[i] = c0[i] + rem % mg.box[i];
          rem /= mg.box[i];
          if (co[i] < 0 || co[i] >= (long)mg.dims[i]) inside = false;
          off += co[i] * (i ? (long)mg.strides[i - 1] / 4 : 1);
        }
        if (!inside) continue;
        // expected element offset of the same coordinates in x's own layout
        long want;
        if (p.cl) {
          const long c = co[0], w = co[1], h = co[2], d = p.entry == 1 ? co[3] : 0,
                     nn = p.entry == 1 ? co[4] : co[3];
          want = (((nn * p.D + d) * p.H + h) * p.W + w) * p.C + c;
        } else {
          const long w = co[0], h = co[1], d = p.entry == 1 ? co[2] : 0,
                     c = p.entry == 1 ? co[3] : co[2], nn = p.entry == 1 ? co[4] : co[3];
          want = (((nn * p.C + c) * p.D + d) * p.H + h) * p.W + w;
        }
        REQ(off == want, "%s map offset %ld, x offset %ld", name, off, want);
      }
    }
    for (int kd = 0; kd < p.KD; ++kd)
      for (int it = 0; it < items; ++it) {
        const int row = (int)fdiv((uint32_t)it, q.fd_lw), cc = it - row * q.LW;
        REQ(row == it / q.LW, "%s fast division by LW", name);
        const int pl = row >= q.RIN ? 1 : 0, r = row - pl * q.RIN;
        for (int e = 0; e < q.E; ++e) {
          long f;  // raw float read by the converter (as in the kernel)
          if (p.cl) f = ((long)r * q.LW + cc) * q.chunk_ci + pl * q.E + e;
          else f = ((long)pl * q.E * q.RIN + r) * q.BW + cc + q.coff + (long)e * q.RIN * q.BW;
          REQ(f >= 0 && f < q.raw_tx / 4, "%s raw read %ld outside the slot", name, f);
          int xc, xr, xw;  // x coordinates the copy put there
          if (p.cl) { xc = (int)(f % q.chunk_ci); xw = iwt + (int)((f / q.chunk_ci) % q.LW); xr = ss.ih0 + (int)(f / ((long)q.chunk_ci * q.LW)); }
          else { xw = iwt + (int)(f % q.BW); xr = ss.ih0 + (int)((f / q.BW) % q.RIN); xc = (int)(f / ((long)q.BW * q.RIN)); }
          REQ(xc == pl * q.E + e && xr == ss.ih0 + r && xw == ss.iw0 + cc,
              "%s converter item (%d,%d,%d,e%d) reads x (%d,%d,%d)", name, pl, r, cc, e, xc, xr, xw);
        }
        const long a = (long)pl * plane_px + kd * q.DSL + (long)r * q.RS + cc;
        REQ(a >= 0 && a < plane_px * q.P, "%s converter store outside hi planes", name);
        if (a < 0 || a >= plane_px * q.P) continue;
        const int id = ss.id0 + kd * p.dil, ih = ss.ih0 + r, iw = ss.iw0 + cc;
        const bool in = id >= 0 && id < p.D && ih >= 0 && ih < p.H && iw >= 0 && iw < p.W;
        for (int hl = 0; hl < 2; ++hl) {
          const long aa = a + hl * q.P * plane_px;
          cnt[aa]++;
          REQ(cnt[aa] == 1, "%s pixel %ld written twice (TMA)", name, aa);
          who[aa] = Px{id, ih, iw, pl, !in};
        }
      }
  } else {
  const int G = q.LW >> 5, parts = q.S2 ? (G + 3) >> 2 : (G ? 1 : 0), tail = q.LW - 32 * G, mjobs = jobs * parts;
  const int njobs = mjobs + (jobs * tail + 31) / 32;
  std::vector<std::pair<int, int>> stores;  // (row job, column)
  for (int J = 0; J < njobs; ++J)
    for (int lane = 0; lane < 32; ++lane) {
      if (J < mjobs) {
        MainJob mj = main_job(J, parts, G);
        REQ(mj.ngroups >= 1 && mj.ngroups <= 4, "%s main job of %d groups", name, mj.ngroups);
        for (int k = 0; k < mj.ngroups; ++k) stores.push_back({mj.row, mj.c0 + lane + 32 * k});
      } else {
        const int l = (J - mjobs) * 32 + lane, job = l / tail;
        if (job < jobs) stores.push_back({job, 32 * G + (l - job * tail)});
      }
    }
  REQ(q.S2 || G <= 4, "%s stride-1 row of %d pixels", name, q.LW);
  for (auto [job, cc] : stores) {
    RowJob jb = row_job(job, ss, q, p, nrows, q.E, q.S2);
    const int plane = job >= nrows ? 1 : 0, sr = job - plane * nrows;
    const int kdp = sr / q.RIN, r = sr % q.RIN;
    {
      const long a = jb.dst / 16 + col_px(cc, s2sub);
      REQ(a >= 0 && a < plane_px * q.P, "%s store outside hi planes (job %d cc %d)", name, job, cc);
      if (a < 0 || a >= plane_px * q.P) continue;
      for (int hl = 0; hl < 2; ++hl) {
        const long aa = a + hl * q.P * plane_px;
        cnt[aa]++;
        REQ(cnt[aa] == 1, "%s pixel %ld written twice", name, aa);
        const int id = ss.id0 + kdp * p.dil, ih = ss.ih0 + r, iw = ss.iw0 + cc;
        const bool in = jb.ok && iw >= 0 && iw < p.W;
        who[aa] = Px{id, ih, iw, plane, !in};
      }
    }
  }
  }
  // MMA operand reads for valid outputs
  for (int ks = 0; ks < q.KS; ++ks)
    for (int half = 0; half < 2; ++half) {
      int tap, plane;
      long off;
      if (q.SP) {
        tap = q.pairtaps ? q.perm[2 * ks + half] : q.perm[ks];
        plane = q.pairtaps ? 0 : half;
        off = q.skd[ks] & 0xFFFF;
        const long lbo = q.skd[ks] >> 16;
        REQ(lbo > 0 && lbo < (1 << 14), "%s SP LBO %ld", name, lbo);
        if (half) off += lbo;
      } else if (q.pairtaps) {
        tap = q.perm[2 * ks + half];
        plane = 0;
        const int t0 = q.perm[2 * ks];
        off = tap_shift(t0, q);
        if (half) {
          const int t1 = q.perm[2 * ks + 1];
          const long lbo = t1 < q.TAPS ? tap_shift(t1, q) - off : 1;
          REQ(lbo > 0 && lbo < (1 << 14), "%s LBO %ld", name, lbo);
          off += lbo;
        }
      } else {
        tap = q.perm[ks];
        plane = half;
        off = tap_shift(tap, q) + half * plane_px;
      }
      REQ(off >= 0 && off < (1 << 14), "%s K offset %ld", name, off);
      if (tap >= q.TAPS) continue;  // zero-weight slot: any finite data
      const int kd = tap / (q.KH * q.KW), kh = (tap / q.KW) % q.KH, kw = tap % q.KW;
      for (int t = 0; t < q.U; ++t)
        for (int m = 0; m < 128; ++m)
          for (int hl = 0; hl < 2; ++hl) {
            const long a = off + (long)t * q.R * q.RS + m + hl * q.P * plane_px;
            REQ(a >= 0 && a < tot_px, "%s MMA read outside the stage (ks %d m %d)", name, ks, m);
            if (a < 0 || a >= tot_px) continue;
            const int r = m / q.RS, c = m % q.RS;
            // the output pixel the epilogue assigns to this M row (its own
            // formulas, independent of the plan's unit steps)
            const int oh = q.GP ? rt * p.ps + t : (rt * q.U + t) * q.R + r;
            const int ow = q.GP ? ct * q.PJ * p.ps + c : ct * q.WT + c;
            const bool valid = q.SP ? (r < q.R && c < q.WT && oh < p.Ho / 2 && ow < p.Wo / 2)
                                    : (r < q.R && c < q.WT && oh < p.Ho && ow < p.Wo);
            if (!valid) continue;
            int id = od * p.stride + kd * p.dil - p.pad_d, ih = oh * p.stride + kh * p.dil - p.pad,
                      iw = ow * p.stride + kw * p.dil - p.pad;
            if (q.SP) {  // pooled pixel (oh, ow); class (a, b) tap reads (oh + da, ow + db)
              const int cls = q.kcls[ks] & 3, a = cls >> 1, b = cls & 1;
              REQ((a + 1 - kh) % 2 == 0 && (b + 1 - kw) % 2 == 0, "%s tap %d not in class %d", name, tap, cls);
              id = 0;
              ih = oh + (a + 1 - kh) / 2;
              iw = ow + (b + 1 - kw) / 2;
            }
            const bool in = id >= 0 && id < p.D && ih >= 0 && ih < p.H && iw >= 0 && iw < p.W;
            const Px &w = who[a];
            bool good;
            if (!cnt[a]) good = false;  // never written: must not be read
            else if (!in) good = w.zero;
            else good = !w.zero && w.id == id && w.ih == ih && w.iw == iw && w.plane == plane;
            if (!good) {
              REQ(false, "%s ks %d half %d t %d m %d: staged (%d,%d,%d,p%d,z%d written %d) want (%d,%d,%d,p%d,in%d)",
                  name, ks, half, t, m, w.id, w.ih, w.iw, w.plane, (int)w.zero, cnt[a], id, ih, iw, plane, (int)in);
              return;
            }
          }
    }
}

void check(const char *name, ConvProblem p) {
  for (int pv = 0; pv < 4; ++pv) {  // both precisions, both input stagings
    const int prec = pv & 1;
    p.staging = pv >> 1;
    TcPlan q = make_plan(p, prec);
    if (pv >= 2 && !q.TMA) continue;  // the tensor-copy plan fell back to loads: checked above
    if (!q.ok) { printf("%s prec%d: not supported\n", name, prec); continue; }
    printf("%s prec%d st%d: S2=%d U=%d P=%d NCH=%d KS=%d pair=%d R=%d RS=%d WT=%d RIN=%d LW=%d SR=%d DSL=%d NPIX=%d S=%d res=%d units=%ld smem=%d TMA=%d TR=%d CTApair=%d\n",
           name, prec, p.staging, q.S2, q.U, q.P, q.NCH, q.KS, q.pairtaps, q.R, q.RS, q.WT, q.RIN, q.LW, q.SR, q.DSL, q.NPIX, q.S, q.b_resident, q.units, q.smem_bytes, q.TMA, q.TR, q.PAIR);
    REQ(q.smem_bytes + 1024 <= 227 * 1024, "smem %d", q.smem_bytes);
    REQ(q.off_misc + (int)sizeof(SmemCtl) <= q.smem_bytes, "misc");
    REQ(q.off_misc % 16 == 0 && q.off_b % 16 == 0 && q.a_stage_bytes % 16 == 0 && q.plane_bytes % 16 == 0, "align");
    REQ(q.R * q.RS <= 128 || (q.R == 1 && q.WT == 128), "tile");
    REQ(((long)q.S * q.a_stage_bytes) == q.off_raw, "stages end at the raw slots");
    REQ((long)q.off_raw + (long)q.TR * q.raw_bytes == q.off_b, "raw slots end at B");
    REQ(q.off_raw % 128 == 0 && q.raw_bytes % 128 == 0, "raw slots 128-byte aligned");
    REQ(!q.TMA || (q.TR >= 2 && q.TR <= 4 && q.BW <= 256 && q.RIN <= 256 && q.chunk_ci <= 256),
        "TMA ring / box");
    REQ(!q.TMA || p.cl || (q.BW % 4 == 0 && (((-p.pad - q.coff) % 4) + 4) % 4 == 0), "TMA x alignment");
    REQ((((long)q.off_b + (q.b_resident ? (long)q.COB * q.NCH * q.b_chunk_bytes : (long)q.SB * q.b_chunk_bytes)) >> 4) < (1 << 14), "B desc range");
    if (q.PAIR) {
      // CTA pairs: 2x2 pool, units in pairs, this CTA's B half resident.
      // Each CTA's bulk copies put, per K step k, image rows 64 r + j of
      // slice sl at k 3072 + sl 1024 + 16 j and image rows 32 r + j at
      // k 3072 + 2048 + sl 512 + 16 j (CTA rank r); the M = 256 MMA takes
      // B column n of the N = 128 product from CTA n / 64 (its row n % 64
      // of the first block) and of the N = 64 product from CTA n / 32: both
      // must be image row n.
      REQ(p.pool && q.U == 2 && !q.GP && q.units % 2 == 0 && q.b_resident, "%s pair plan", name);
      REQ(q.b_kstep == 3072 && q.b_chunk_bytes == q.KS * 3072, "%s pair B size", name);
      for (int n = 0; n < 128; ++n) {
        const int r = n / 64, j = n % 64;
        REQ(64 * r + j == n, "%s pair N128 column %d", name, n);
        REQ(j * 16 + 16 <= 1024, "%s pair N128 slice", name);
      }
      for (int n = 0; n < 64; ++n) {
        const int r = n / 32, j = n % 32;
        REQ(32 * r + j == n, "%s pair N64 column %d", name, n);
        REQ(2048 + 512 + j * 16 + 16 <= 3072, "%s pair N64 slice", name);
      }
    }
    if (q.GP) {
      // General max pool: the row maxima buffer [64 channels][kXbPitch]
      // lies inside the plan's shared memory; every window reads columns
      // below 128 of its channel row; and the 32 channels one warp's window
      // threads read at a column (thread e of the epilogue takes channel
      // e % 64) fall in 32 distinct banks.
      REQ(q.XB == 64 * kXbPitch * 4 && kXbPitch >= 128, "%s row-maxima buffer size", name);
      REQ(q.off_xb >= q.off_misc + (int)sizeof(SmemCtl) && q.off_xb + q.XB <= q.smem_bytes,
          "%s row-maxima buffer inside shared memory", name);
      REQ(q.PJ >= 1 && (q.PJ - 1) * p.ps + p.pk <= 128, "%s windows inside the strip", name);
      for (int c0 = 0; c0 < 64; c0 += 32)
        for (int col = 0; col < 128; ++col) {
          uint32_t banks = 0;
          for (int l = 0; l < 32; ++l) banks |= 1u << (((c0 + l) * kXbPitch + col) % 32);
          REQ(banks == 0xffffffffu, "%s window loads of a warp share banks (col %d)", name, col);
        }
    }
    std::vector<int> seen(kMaxTaps + 2, 0);
    for (int k = 0; k < kMaxTaps + 2; ++k) if (q.perm[k] < q.TAPS) seen[q.perm[k]]++;
    for (int t = 0; t < q.TAPS; ++t) REQ(seen[t] == 1, "%s perm", name);
    const int n = p.N - 1;
    const int ods[2] = {0, p.Do - 1}, rts[3] = {0, q.n_rt / 2, q.n_rt - 1};
    for (int a : ods) for (int b : rts) for (int c = 0; c < q.n_ct; ++c) check_stage(name, p, q, n, a, b, c);
  }
}

ConvProblem conv2d(int N, int C, int H, int W, int CO, int pad, int stride = 1, int dil = 1) {
  ConvProblem p{}; p.N = N; p.C = C; p.D = 1; p.H = H; p.W = W; p.CO = CO; p.KD = 1; p.KH = p.KW = 3;
  p.pad = pad; p.stride = stride; p.dil = dil; p.Do = 1;
  p.Ho = (H + 2 * pad - 2 * dil - 1) / stride + 1; p.Wo = (W + 2 * pad - 2 * dil - 1) / stride + 1; return p;
}
ConvProblem conv3d(int N, int C, int D, int H, int W, int CO, int pad, int stride = 1, int dil = 1) {
  ConvProblem p = conv2d(N, C, H, W, CO, pad, stride, dil); p.D = D; p.KD = 3; p.pad_d = pad;
  p.entry = 1;
  p.Do = (D + 2 * pad - 2 * dil - 1) / stride + 1; return p;
}
// kernel size k (square / cubic)
ConvProblem convk(int N, int C, int D, int H, int W, int CO, int k, int pad, int stride = 1,
                  int dil = 1, bool d3 = false) {
  ConvProblem p{}; p.N = N; p.C = C; p.D = D; p.H = H; p.W = W; p.CO = CO;
  p.KD = d3 ? k : 1; p.KH = p.KW = k; p.pad = pad; p.pad_d = d3 ? pad : 0;
  p.stride = stride; p.dil = dil; p.entry = d3 ? 1 : 0;
  const int span = (k - 1) * dil + 1;
  p.Do = d3 ? (D + 2 * pad - span) / stride + 1 : 1;
  p.Ho = (H + 2 * pad - span) / stride + 1; p.Wo = (W + 2 * pad - span) / stride + 1; return p;
}
ConvProblem convT2(int N, int C, int H, int W, int CO, int op) {
  ConvProblem p = conv2d(N, C, H, W, CO, 0); p.pool = 1; p.wlayout = 1; p.subpix = 1;
  p.pk = p.ps = 2; p.tstride = 2; p.tpad = 1; p.entry = 2;
  p.Ho = 2 * H - 1 + op; p.Wo = 2 * W - 1 + op; return p;
}
ConvProblem convT(int N, int C, int H, int W, int CO, int pk = 2, int ps = 2) {
  ConvProblem p = conv2d(N, C, H, W, CO, 1); p.pool = 1; p.wlayout = 1; p.pk = pk; p.ps = ps;
  p.tstride = 1; p.tpad = 1; p.entry = 2; return p;
}
int main() {
  check("cfg1", conv2d(4, 8, 32, 32, 64, 0));
  check("cfg3", conv2d(128, 8, 128, 128, 64, 0));
  check("r2d-a", conv2d(2, 3, 9, 37, 10, 0));
  check("r2d-b", conv2d(1, 8, 33, 130, 64, 0));
  check("r2d-c", conv2d(3, 12, 17, 20, 70, 1));
  check("r2d-d", conv2d(1, 16, 5, 260, 64, 2));
  check("cfg4", conv3d(128, 8, 16, 64, 64, 64, 0));
  check("r3d-a", conv3d(1, 5, 5, 7, 9, 70, 0));
  check("r3d-b", conv3d(2, 8, 4, 12, 66, 64, 1));
  check("cfg2", convT(2, 64, 32, 32, 64));
  check("cfg5", convT(128, 64, 256, 256, 64));
  // the pooled workload at full size runs on CTA pairs (fp16 split); a
  // batch below 8192 units, an odd unit count and the tf32 split do not
  REQ(make_plan(convT(128, 64, 256, 256, 64), 1).PAIR == 1, "cfg5 fp16 on CTA pairs");
  REQ(make_plan(convT(128, 64, 256, 256, 64), 0).PAIR == 0, "cfg5 tf32 single CTAs");
  REQ(make_plan(convT(16, 64, 256, 256, 64), 1).PAIR == 0, "4096 units single CTAs");
  REQ(make_plan(convT(32, 64, 256, 200, 64), 1).PAIR == 1, "8192 units on pairs");
  REQ(make_plan(convT(32, 64, 256, 200, 64), 1, false).PAIR == 0, "pairs refused -> single CTAs");
  check("pair-ragged", convT(32, 64, 256, 200, 64));
  check("rT-d", convT(1, 9, 33, 31, 65));
  check("s2-cfg3", conv2d(128, 8, 128, 128, 64, 0, 2));
  check("s2-a", conv2d(2, 8, 33, 37, 70, 0, 2));
  check("s2-b", conv2d(1, 5, 20, 71, 70, 1, 2));
  check("s2-c", conv2d(2, 16, 9, 12, 70, 2, 2));
  check("s2-wide", conv2d(1, 8, 11, 300, 64, 1, 2));
  check("s2-c64", conv2d(2, 64, 40, 300, 64, 1, 2));
  check("s2-3d", conv3d(2, 8, 9, 12, 35, 64, 1, 2));
  check("s2-3d-b", conv3d(1, 16, 8, 20, 140, 64, 0, 2));
  check("d2-cfg3", conv2d(128, 8, 128, 128, 64, 2, 1, 2));
  check("d2-a", conv2d(2, 8, 33, 37, 70, 0, 1, 2));
  check("d2-b", conv2d(1, 5, 20, 71, 70, 3, 1, 2));
  check("d2-wide", conv2d(1, 8, 11, 300, 64, 4, 1, 2));
  check("d2-c64", conv2d(2, 64, 40, 300, 64, 2, 1, 2));
  check("d2s2-a", conv2d(2, 8, 33, 37, 70, 2, 2, 2));
  check("d2s2-wide", conv2d(1, 8, 15, 300, 64, 1, 2, 2));
  check("d2s2-c64", conv2d(2, 64, 40, 260, 64, 4, 2, 2));
  check("T2-a", convT2(2, 64, 16, 20, 64, 1));
  check("T2-b", convT2(1, 8, 9, 33, 64, 0));
  check("T2-c", convT2(2, 16, 12, 140, 70, 1));
  check("T2-d", convT2(1, 3, 5, 7, 64, 0));
  check("T2-big", convT2(128, 64, 128, 128, 64, 1));
  check("T2-w127", convT2(1, 8, 6, 127, 64, 1));
  check("T2-w300", convT2(1, 24, 4, 300, 130, 0));
  check("d2-3d", conv3d(2, 8, 9, 12, 35, 64, 2, 1, 2));
  check("d2-3d-b", conv3d(1, 16, 8, 20, 140, 64, 0, 1, 2));
  check("d2s2-3d", conv3d(2, 8, 11, 12, 35, 64, 2, 2, 2));
  check("d2s2-3d-c", conv3d(2, 8, 11, 12, 20, 64, 2, 2, 2));
  check("d2s2-3d-d", conv3d(2, 8, 11, 10, 12, 64, 1, 2, 2));
  check("d2-3d-c", conv3d(1, 16, 8, 20, 70, 64, 0, 1, 2));
  {  // channels-last (tensor-copy staging reads pixel-major slots)
    ConvProblem a = conv2d(2, 8, 33, 36, 64, 0); a.cl = 1; check("cl-a", a);
    ConvProblem b = conv2d(1, 12, 17, 20, 70, 1); b.cl = 1; check("cl-b", b);
    ConvProblem c = conv2d(1, 16, 9, 150, 64, 2, 1, 2); c.cl = 1; check("cl-c", c);
    ConvProblem d = conv3d(2, 8, 6, 10, 30, 64, 1); d.cl = 1; check("cl-3d", d);
    ConvProblem e = conv2d(2, 64, 10, 30, 64, 1); e.cl = 1; check("cl-c64", e);
  }
  // general max pool on the tensor cores: one tile per window row
  check("gp-3s2", convT(2, 16, 17, 21, 64, 3, 2));
  check("gp-4s4", convT(1, 8, 20, 40, 70, 4, 4));
  check("gp-2s1", convT(1, 8, 12, 40, 64, 2, 1));
  check("gp-1s1", convT(1, 8, 6, 7, 64, 1, 1));
  check("gp-3s3-wide", convT(1, 64, 9, 300, 64, 3, 3));
  check("gp-3s2-big", convT(16, 64, 256, 256, 64, 3, 2));
  check("gp-3s2-strips", convT(2, 8, 9, 260, 64, 3, 2));
  check("gp-3s3-strips", convT(1, 8, 9, 300, 64, 3, 3));
  check("gp-4s2-strips", convT(1, 8, 9, 520, 64, 4, 2));
  // kernel sizes 1, 5, 7 (2-D) and 1, 5 (3-D), strides / dilations 1-2
  check("k1", convk(2, 8, 1, 20, 36, 64, 1, 0));
  check("k1-c64", convk(1, 64, 1, 9, 40, 70, 1, 0));
  check("k5", convk(2, 8, 1, 21, 37, 64, 5, 2));
  check("k5-s2", convk(1, 16, 1, 19, 140, 64, 5, 1, 2));
  check("k5-d2", convk(1, 8, 1, 25, 60, 64, 5, 4, 1, 2));
  check("k7", convk(1, 8, 1, 23, 44, 64, 7, 3));
  check("k7-wide", convk(1, 12, 1, 12, 300, 70, 7, 0));
  check("k7-s2-d2", convk(1, 8, 1, 30, 70, 64, 7, 6, 2, 2));
  check("k1-3d", convk(1, 8, 6, 9, 20, 64, 1, 0, 1, 1, true));
  check("k5-3d", convk(1, 8, 9, 12, 20, 64, 5, 2, 1, 1, true));
  check("k5-3d-s2", convk(1, 8, 11, 13, 30, 64, 5, 1, 2, 1, true));
  // channels-first shapes that take the tensor copies (W a multiple of 4)
  check("tma-pad1-strips", conv2d(1, 8, 9, 260, 64, 1));
  check("tma-pad3-d2", conv2d(1, 8, 11, 132, 64, 3, 1, 2));
  check("tma-c12", conv2d(2, 12, 17, 20, 70, 1));
  check("tma-3d-d2", conv3d(1, 8, 8, 12, 36, 64, 2, 1, 2));
  printf(fails ? "CHECK FAILED (%d)\n" : "CHECK OK\n", fails);
  return fails != 0;
}
