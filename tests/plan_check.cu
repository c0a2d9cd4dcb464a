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
  ss.ih0 = rt * q.U * q.R * p.stride - p.pad;
  ss.iw0 = ct * q.WT * p.stride - p.pad;
  ss.ci0 = 0;
  const int nrows = p.KD * q.RIN, jobs = q.P * nrows;
  const int s2sub = q.S2 ? q.SUB : 0;
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
      const int kd = tap / 9, kh = (tap / 3) % 3, kw = tap % 3;
      for (int t = 0; t < q.U; ++t)
        for (int m = 0; m < 128; ++m)
          for (int hl = 0; hl < 2; ++hl) {
            const long a = off + (long)t * q.R * q.RS + m + hl * q.P * plane_px;
            REQ(a >= 0 && a < tot_px, "%s MMA read outside the stage (ks %d m %d)", name, ks, m);
            if (a < 0 || a >= tot_px) continue;
            const int r = m / q.RS, c = m % q.RS;
            const int oh = (rt * q.U + t) * q.R + r, ow = ct * q.WT + c;
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
  for (int prec = 0; prec < 2; ++prec) {
    TcPlan q = make_plan(p, prec);
    if (!q.ok) { printf("%s prec%d: not supported\n", name, prec); continue; }
    printf("%s prec%d: S2=%d U=%d P=%d NCH=%d KS=%d pair=%d R=%d RS=%d WT=%d RIN=%d LW=%d SR=%d DSL=%d NPIX=%d S=%d res=%d units=%ld smem=%d\n",
           name, prec, q.S2, q.U, q.P, q.NCH, q.KS, q.pairtaps, q.R, q.RS, q.WT, q.RIN, q.LW, q.SR, q.DSL, q.NPIX, q.S, q.b_resident, q.units, q.smem_bytes);
    REQ(q.smem_bytes + 1024 <= 227 * 1024, "smem %d", q.smem_bytes);
    REQ(q.off_misc + (int)sizeof(SmemCtl) <= q.smem_bytes, "misc");
    REQ(q.off_misc % 16 == 0 && q.off_b % 16 == 0 && q.a_stage_bytes % 16 == 0 && q.plane_bytes % 16 == 0, "align");
    REQ(q.R * q.RS <= 128 || (q.R == 1 && q.WT == 128), "tile");
    REQ(((long)q.S * q.a_stage_bytes) == q.off_b, "stages end at B");
    REQ((((long)q.off_b + (q.b_resident ? (long)q.COB * q.NCH * q.b_chunk_bytes : (long)q.SB * q.b_chunk_bytes)) >> 4) < (1 << 14), "B desc range");
    std::vector<int> seen(28, 0);
    for (int k = 0; k < 28; ++k) if (q.perm[k] < q.TAPS) seen[q.perm[k]]++;
    for (int t = 0; t < q.TAPS; ++t) REQ(seen[t] == 1, "%s perm", name);
    const int n = p.N - 1;
    const int ods[2] = {0, p.Do - 1}, rts[3] = {0, q.n_rt / 2, q.n_rt - 1}, cts[2] = {0, q.n_ct - 1};
    for (int a : ods) for (int b : rts) for (int c : cts) check_stage(name, p, q, n, a, b, c);
  }
}

ConvProblem conv2d(int N, int C, int H, int W, int CO, int pad, int stride = 1, int dil = 1) {
  ConvProblem p{}; p.N = N; p.C = C; p.D = 1; p.H = H; p.W = W; p.CO = CO; p.KD = 1; p.KH = p.KW = 3;
  p.pad = pad; p.stride = stride; p.dil = dil; p.Do = 1;
  p.Ho = (H + 2 * pad - 2 * dil - 1) / stride + 1; p.Wo = (W + 2 * pad - 2 * dil - 1) / stride + 1; return p;
}
ConvProblem conv3d(int N, int C, int D, int H, int W, int CO, int pad, int stride = 1, int dil = 1) {
  ConvProblem p = conv2d(N, C, H, W, CO, pad, stride, dil); p.D = D; p.KD = 3; p.pad_d = pad;
  p.Do = (D + 2 * pad - 2 * dil - 1) / stride + 1; return p;
}
ConvProblem convT2(int N, int C, int H, int W, int CO, int op) {
  ConvProblem p = conv2d(N, C, H, W, CO, 0); p.pool = 1; p.wlayout = 1; p.subpix = 1;
  p.Ho = 2 * H - 1 + op; p.Wo = 2 * W - 1 + op; return p;
}
ConvProblem convT(int N, int C, int H, int W, int CO) {
  ConvProblem p = conv2d(N, C, H, W, CO, 1); p.pool = 1; p.wlayout = 1; return p;
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
  printf(fails ? "CHECK FAILED (%d)\n" : "CHECK OK\n", fails);
  return fails != 0;
}
