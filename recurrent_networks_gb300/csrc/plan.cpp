// Kernel planner (see plan.h): for every kernel family, enumerate the
// instantiated tile parameters, keep the points that satisfy the divisibility,
// warp, register, shared-memory and cluster constraints, and pick the one with
// the smallest modelled step latency (ties go to fewer CTAs).
#include "plan.h"

#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "rnn.h"

namespace rnn {

static int gates_of(int fn) { return fn == 0 ? 4 : fn == 1 ? 3 : fn == 2 ? 1 : 4; }
static int states_of(int fn) { return fn == 0 ? 2 : fn == 1 ? 1 : fn == 2 ? 1 : 4; }

static const int kClusterSizes[] = {1, 2, 3, 4, 6, 8, 12, 16};
static const DeviceLimits kDefaultLimits;

static const DeviceLimits& limits_of(const PlanRequest& q) { return q.lim ? *q.lim : kDefaultLimits; }

// Waves of clusters the device runs the groups in: the co-resident cluster
// count when the device reports it, else CTAs over SMs. Returns 0 when the
// device cannot hold even one cluster of this shape (the point is infeasible).
static int cluster_waves(const PlanRequest& q, const DeviceLimits& lim, const FusedShape& fs, int groups) {
  int cap = lim.cluster_capacity ? lim.cluster_capacity(q.fn, q.bwd, fs) : -1;
  if (cap == 0) return 0;
  if (cap < 0) cap = lim.sms / fs.C;
  if (cap < 1) return 0;
  return (groups + cap - 1) / cap;
}
static const int kNT[] = {1, 2};
// instantiated k-tiles per warp of the forward cluster kernel: a warp holds
// all G gate tiles over a short K (allg) or one gate tile over a long K
static const int kKTAllG[] = {2, 3, 4};
static const int kKTOneG[] = {4, 6, 8, 12, 16};

// Warps of a forward kernel: the (U/16) * (G/GW) * KS that the product needs,
// or more when the cell update needs them (each thread carries at most
// FUSED_PPT (batch row, unit) pairs in registers).
static int fwd_warps(int U, int GQ, int KS, int nb) {
  const int mma = (U / 16) * GQ * KS;
  const int cell = (nb * U + FUSED_PPT * 32 - 1) / (FUSED_PPT * 32);
  return mma > cell ? mma : cell;
}

// Forward cluster kernel, candidate point (C, NT, KT, allg):
//   divisibility   D = C U, U = 16 m;  D / 16 = KS KT;
//   inequalities   1 <= warps <= 8, C <= 16, shared memory <= 227 KB,
//                  registers 4 GW KT (R) + 4 GW CH NT (accumulators) + 80 <= 255,
//                  with GW = G (allg) or 1, CH = 2 chains when GW = 1.
bool fused_fwd_feasible(const PlanRequest& q, int C, int NT, int KT, bool allg, const DeviceLimits& lim,
                        Plan* out) {
  const int G = gates_of(q.fn), S = states_of(q.fn), D = q.D;
  if (q.dtype != RNN_BF16) return false;
  if (C < 1 || C > lim.max_cluster || D % C) return false;
  const int U = D / C;
  if (U % 16) return false;
  if (D % 16 || (D / 16) % KT) return false;
  const int KS = (D / 16) / KT;
  if (KS > FUSED_MAX_KS) return false;
  const int GW = allg ? G : 1, GQ = G / GW, CH = GW == 1 ? 2 : 1;
  const int BC = 8 * NT;
  const int nb = q.B < BC ? q.B : BC;
  const int warps = fwd_warps(U, GQ, KS, nb);
  if (warps < 1 || warps > lim.max_warps) return false;
  const int regs = 4 * GW * KT + 4 * GW * CH * NT + 80;
  if (regs > lim.regs_per_thread) return false;
  const FusedSmem L = FusedSmem::make(G, S, D, U, BC, KS);
  if (L.total > lim.smem_per_cta) return false;
  const int groups = q.N * ((q.B + BC - 1) / BC);
  const int threads = warps * 32;
  // latency model of one step (cycles), calibrated on the phase trace: the
  // exchange round trip, the warp's MMA issue and dependent chain, the
  // shared-memory loads of the K-split partial sums (G KS per pair), the cell
  // update, and waves when the grid exceeds the SMs.
  double pairs = (double)nb * U / threads;
  if (pairs < 1) pairs = 1;
  double cyc = 900.0 + 10.0 * GW * KT * NT + 28.0 * KT / CH + 14.0 * G * KS * pairs + 250.0 * pairs +
               (C > 1 ? 600.0 : 0.0);
  FusedShape fs;
  fs.C = C; fs.U = U; fs.NT = NT; fs.KT = KT; fs.KS = KS; fs.allg = allg; fs.warps = warps; fs.smem = L.total;
  const int waves = cluster_waves(q, lim, fs, groups);
  if (waves < 1) return false;
  cyc *= waves;
  if (out) {
    *out = Plan{};
    out->path = RNN_PATH_FUSED;
    out->fs.C = C;
    out->fs.U = U;
    out->fs.NT = NT;
    out->fs.KT = KT;
    out->fs.KS = KS;
    out->fs.allg = allg;
    out->fs.warps = warps;
    out->fs.smem = L.total;
    out->groups = groups;
    out->regs_R = 4 * GW * KT;
    out->model_ns = cyc / 1.9;  // at ~1.9 GHz
  }
  return true;
}

// Optional restriction of the search (tests and tuning sweeps): the
// environment variables RNN_PLAN_C, RNN_PLAN_NT, RNN_PLAN_KT, RNN_PLAN_MT
// (backward) and RNN_PLAN_ALLG (forward: 1 for the all-gates warp mapping),
// when set, admit only candidates with that value.
static bool env_admits(const char* name, int v) {
  const char* s = getenv(name);
  return !s || !*s || atoi(s) == v;
}

static int fused_fwd_plan(const PlanRequest& q, Plan* best) {
  const DeviceLimits& lim = limits_of(q);
  int found = 0;
  for (int C : kClusterSizes)
    for (int ag = 0; ag < 2; ++ag)
      for (int NT : kNT) {
        if (!ag && NT != 1) continue;  // one-gate kernels are built for one n-tile
        const int* kts = ag ? kKTAllG : kKTOneG;
        const int nkt = ag ? 3 : 5;
        for (int x = 0; x < nkt; ++x) {
          const int KT = kts[x];
          Plan p;
          if (!env_admits("RNN_PLAN_C", C) || !env_admits("RNN_PLAN_NT", NT) ||
              !env_admits("RNN_PLAN_KT", KT) || !env_admits("RNN_PLAN_ALLG", ag))
            continue;
          if (!fused_fwd_feasible(q, C, NT, KT, ag != 0, lim, &p)) continue;
          ++found;
          const int ctas = p.groups * p.fs.C, bctas = best->groups * best->fs.C;
          if (found == 1 || p.model_ns < best->model_ns - 1e-9 ||
              (p.model_ns < best->model_ns + 1e-9 && ctas < bctas))
            *best = p;
        }
      }
  best->candidates = found;
  return found ? RNN_OK : RNN_EUNSUPPORTED;
}

// Backward cluster kernel, candidate point (C, NT, MT):
//   divisibility   D = C * U, U = 16 m;  D / 16 = warps * MT (row blocks of dh);
//   inequalities   G U / 16 <= 8 (own gradient block k-tiles), 1 <= warps <= 8,
//                  C <= 16, shared memory (FusedBwdSmem) <= 227 KB,
//                  registers 32 MT (resident R) + 4 MT NT + 64 <= 255.
static const int kMT[] = {1, 2};

bool fused_bwd_feasible(const PlanRequest& q, int C, int NT, int MT, const DeviceLimits& lim, Plan* out) {
  const int G = gates_of(q.fn), S = states_of(q.fn), D = q.D;
  const int K = (q.fn == 1 ? 4 : G) + S;
  if (q.dtype != RNN_BF16) return false;
  if (C < 1 || C > lim.max_cluster || D % C) return false;
  const int U = D / C;
  if (U % 16 || D % 16) return false;
  const int KTA = G * U / 16;
  if (KTA < 1 || KTA > FUSED_BWD_MAX_KTA) return false;
  if ((D / 16) % MT) return false;
  const int warps = (D / 16) / MT;
  if (warps < 1 || warps > lim.max_warps) return false;
  const int BC = 8 * NT;
  if ((q.B < BC ? q.B : BC) * U > FUSED_PPT * warps * 32) return false;  // carried pairs in registers
  const int regs = 32 * MT + 4 * MT * NT + 64;
  if (regs > lim.regs_per_thread) return false;
  const FusedBwdSmem L = FusedBwdSmem::make(G, S, K, U, BC, C);
  if (L.total > lim.smem_per_cta) return false;
  const int groups = q.N * ((q.B + BC - 1) / BC);
  const int threads = warps * 32;
  const int nb = q.B < BC ? q.B : BC;
  double pairs = (double)nb * U / threads;
  if (pairs < 1) pairs = 1;
  const double mma = (double)MT * KTA * NT;
  double cyc = 900.0 + 18.0 * mma + (160.0 + 4.0 * C) * pairs + 25.0 * MT * NT + (C > 1 ? 150.0 : 0.0);
  FusedShape fs;
  fs.C = C; fs.U = U; fs.NT = NT; fs.MT = MT; fs.KT = KTA; fs.warps = warps; fs.smem = L.total;
  const int waves = cluster_waves(q, lim, fs, groups);
  if (waves < 1) return false;
  cyc *= waves;
  if (out) {
    *out = Plan{};
    out->path = RNN_PATH_FUSED;
    out->fs.C = C;
    out->fs.U = U;
    out->fs.NT = NT;
    out->fs.MT = MT;
    out->fs.KT = KTA;
    out->fs.warps = warps;
    out->fs.smem = L.total;
    out->groups = groups;
    out->regs_R = 4 * MT * KTA;
    out->model_ns = cyc / 1.9;
  }
  return true;
}

static int fused_bwd_plan(const PlanRequest& q, Plan* best) {
  const DeviceLimits& lim = limits_of(q);
  int found = 0;
  for (int C : kClusterSizes)
    for (int NT : kNT)
      for (int MT : kMT) {
        Plan p;
        if (!env_admits("RNN_PLAN_C", C) || !env_admits("RNN_PLAN_NT", NT) || !env_admits("RNN_PLAN_MT", MT))
          continue;
        if (!fused_bwd_feasible(q, C, NT, MT, lim, &p)) continue;
        ++found;
        const int ctas = p.groups * p.fs.C, bctas = best->groups * best->fs.C;
        if (found == 1 || p.model_ns < best->model_ns - 1e-9 ||
            (p.model_ns < best->model_ns + 1e-9 && ctas < bctas))
          *best = p;
      }
  best->candidates = found;
  return found ? RNN_OK : RNN_EUNSUPPORTED;
}

static int fused_plan(const PlanRequest& q, Plan* best) {
  return q.bwd ? fused_bwd_plan(q, best) : fused_fwd_plan(q, best);
}

// Grid kernels (cooperative launch, h / dr exchanged through L2), candidate
// point (C, NT, KT):
//   divisibility   D = C U, U = 16 m; forward D/16 = KS KT, backward
//                  G D / 16 = KS KT; warps = (U / 16) KS;
//   inequalities   1 <= warps <= 8, groups * C <= SMs (every CTA resident),
//                  registers (forward 4 G KT + 4 G NT + 48, backward
//                  4 KT + 4 NT + 64) <= 255, shared memory <= 227 KB;
//   KT takes the instantiated values (forward 4, 8; backward 8, 16, 24, 32).
static const int kGridC[] = {8, 16, 32, 64, 128};
static const int kGridFwdKT[] = {8, 16, 32};
static const int kGridBwdKT[] = {8, 16, 24, 32};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool grid_feasible(const PlanRequest& q, int C, int NT, int KT, const DeviceLimits& lim, Plan* out) {
  const int G = gates_of(q.fn), S = states_of(q.fn), D = q.D;
  const int K = (q.fn == 1 ? 4 : G) + S;
  if (q.dtype != RNN_BF16 || D % C) return false;
  const int U = D / C;
  if (U % 16 || D % 16) return false;
  const int klen = q.bwd ? G * D : D;
  if ((klen / 16) % KT) return false;
  const int KS = (klen / 16) / KT;
  const int BC = 8 * NT;
  // forward: one gate tile per warp (G tiles per 16-unit group)
  const int warps = q.bwd ? (U / 16) * KS : fwd_warps(U, G, KS, q.B < BC ? q.B : BC);
  if (warps < 1 || warps > lim.max_warps) return false;
  const int groups = q.N * ((q.B + BC - 1) / BC);
  if (groups * C > lim.sms) return false;
  const int regs = q.bwd ? 4 * KT + 4 * NT + 64 : 4 * KT + 8 * NT + 80;
  if (regs > lim.regs_per_thread) return false;
  const size_t smem = q.bwd ? GridBwdSmem::make(G, S, K, D, U, BC, KS).total
                            : FusedSmem::make(G, S, D, U, BC, KS).total;
  if (smem > lim.smem_per_cta) return false;
  const int nb = q.B < BC ? q.B : BC;
  double pairs = (double)nb * U / (warps * 32);
  if (pairs < 1) pairs = 1;
  // step: counter round trip through L2, the gathered vector from L2
  // (~64 B/clk/SM), the warp's MMA chain, the K-split reduction and the cell
  const double gather = (double)nb * klen * 2 / 64.0;
  double cyc = 2200.0 + gather + 18.0 * KT * NT + 6.0 * KS * (q.bwd ? 1 : G) * pairs + 150.0 * pairs;
  if (out) {
    *out = Plan{};
    out->path = RNN_PATH_GRID;
    out->fs.C = C;
    out->fs.U = U;
    out->fs.NT = NT;
    out->fs.KT = KT;
    out->fs.KS = KS;
    out->fs.warps = warps;
    out->fs.smem = smem;
    out->groups = groups;
    out->regs_R = 4 * KT;
    // the exchange buffers, then the step counters and die tickets
    out->scratch_bytes = align256((size_t)2 * groups * BC * klen * 2) +
                         align256(GRID_CTR_BYTES + (size_t)groups * 4);
    out->model_ns = cyc / 1.9;
  }
  return true;
}

static int grid_plan(const PlanRequest& q, Plan* best) {
  const DeviceLimits& lim = limits_of(q);
  int found = 0;
  const int* kts = q.bwd ? kGridBwdKT : kGridFwdKT;
  const int nkt = q.bwd ? 4 : 3;
  for (int C : kGridC)
    for (int NT : kNT)
      for (int x = 0; x < nkt; ++x) {
        const int KT = kts[x];
        Plan p;
        if (!env_admits("RNN_PLAN_C", C) || !env_admits("RNN_PLAN_NT", NT) || !env_admits("RNN_PLAN_KT", KT))
          continue;
        if (!grid_feasible(q, C, NT, KT, lim, &p)) continue;
        ++found;
        if (found == 1 || p.model_ns < best->model_ns - 1e-9) *best = p;
      }
  best->candidates = found;
  return found ? RNN_OK : RNN_EUNSUPPORTED;
}

// Alternating path: one kernel per step streams R from L2 / HBM; feasible for
// bf16 whenever the unit tiles (16 units; 64 for Elman) divide D. The model is
// the step's R bytes at an L2 rate of ~10 TB/s plus ~2 us of launch spacing.
static int alt_plan(const PlanRequest& q, Plan* p) {
  *p = Plan{};
  if (q.dtype != RNN_BF16 || !alt_supported(q.fn, q.D)) return RNN_EUNSUPPORTED;
  p->path = RNN_PATH_ALTERNATING;
  p->fs.NT = q.B <= 16 ? 1 : 2;
  p->groups = q.N * ((q.B + 16 * p->fs.NT - 1) / (16 * p->fs.NT));
  p->scratch_bytes = alt_scratch_bytes(q.fn, q.B, q.N, q.D, q.bwd);
  p->model_ns = 2000.0 + (double)gates_of(q.fn) * q.N * q.D * q.D * 2 / 1.0e4;
  p->candidates = 1;
  return RNN_OK;
}

static void simt_plan(const PlanRequest& q, Plan* p) {
  *p = Plan{};
  p->path = RNN_PATH_SIMT;
  p->fs.NT = 1;
  p->groups = q.N * ((q.B + 7) / 8);
}

int plan_select(const PlanRequest& q, Plan* out) {
  Plan p;
  switch (q.path) {
    case RNN_PATH_SIMT:
      simt_plan(q, &p);
      *out = p;
      return RNN_OK;
    case RNN_PATH_AUTO:
      // the cluster kernels when a feasible point exists (bf16), then the grid
      // kernels (R too large for one cluster), then the alternating path (R
      // streamed every step), else the plain path
      if (fused_plan(q, &p) == RNN_OK || grid_plan(q, &p) == RNN_OK || alt_plan(q, &p) == RNN_OK) {
        *out = p;
        return RNN_OK;
      }
      simt_plan(q, &p);
      *out = p;
      return RNN_OK;
    case RNN_PATH_GRID:
      if (grid_plan(q, &p) == RNN_OK) {
        *out = p;
        return RNN_OK;
      }
      snprintf(p.why, sizeof(p.why),
               "no grid plan for fn=%d dtype=%d D=%d B=%d N=%d%s (bf16 only; U = D/C multiple of 16, <= 8 "
               "warps, all CTAs resident)",
               q.fn, q.dtype, q.D, q.B, q.N, q.bwd ? " (backward)" : "");
      *out = p;
      return RNN_EUNSUPPORTED;
    case RNN_PATH_ALTERNATING:
      if (alt_plan(q, &p) == RNN_OK) {
        *out = p;
        return RNN_OK;
      }
      snprintf(p.why, sizeof(p.why),
               "no alternating plan for fn=%d dtype=%d D=%d (bf16 only; D a multiple of the 16-unit tile, "
               "64 for elman)",
               q.fn, q.dtype, q.D);
      *out = p;
      return RNN_EUNSUPPORTED;
    case RNN_PATH_FUSED:
      if (fused_plan(q, &p) == RNN_OK) {
        *out = p;
        return RNN_OK;
      }
      snprintf(p.why, sizeof(p.why),
               "no cluster plan for fn=%d dtype=%d D=%d B=%d%s (bf16 only; D = C*U with U %% 16 == 0, "
               "D/16 = KS*KT, <= 8 warps, smem <= 227 KB)",
               q.fn, q.dtype, q.D, q.B, q.bwd ? " (backward)" : "");
      *out = p;
      return RNN_EUNSUPPORTED;
    default:
      snprintf(p.why, sizeof(p.why), "path %d not available for fn=%d D=%d", q.path, q.fn, q.D);
      *out = p;
      return RNN_EUNSUPPORTED;
  }
}

void plan_describe(const Plan& p, int rc, char* buf, size_t len) {
  if (rc != RNN_OK) {
    snprintf(buf, len, "unsupported: %s", p.why);
    return;
  }
  const char* names[] = {"auto", "fused", "alternating", "simt", "grid"};
  snprintf(buf, len,
           "path=%s C=%d U=%d NT=%d KT=%d KS=%d MT=%d allg=%d warps=%d groups=%d regs_R=%d smem=%zu "
           "scratch=%zu model_ns=%.1f candidates=%d",
           names[(p.path >= 0 && p.path <= 4) ? p.path : 0], p.fs.C, p.fs.U, p.fs.NT, p.fs.KT, p.fs.KS, p.fs.MT,
           (int)p.fs.allg, p.fs.warps, p.groups, p.regs_R, p.fs.smem, p.scratch_bytes, p.model_ns, p.candidates);
}

}  // namespace rnn
