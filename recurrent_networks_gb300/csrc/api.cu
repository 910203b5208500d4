// C ABI of the head-wise recurrent scan library: validation, workspace layout,
// path selection and launches. Declarations and argument documentation are in
// include/rnn.h.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "dies.h"
#include "kernels.cuh"
#include "plan.h"
#include "umma.cuh"
#include "rnn.h"

namespace rnn {

static std::atomic<unsigned long long> g_launches{0};
void note_launch(int count) { g_launches.fetch_add((unsigned long long)count); }

namespace {
struct AttrEntry {
  const void* func;
  int dev;
  size_t smem;
  bool nonportable;
};
std::mutex g_attr_mu;
std::vector<AttrEntry> g_attrs;

AttrEntry* attr_entry(const void* func, int dev) {
  for (auto& e : g_attrs)
    if (e.func == func && e.dev == dev) return &e;
  g_attrs.push_back(AttrEntry{func, dev, 0, false});
  return &g_attrs.back();
}
}  // namespace

cudaError_t set_smem_attr(const void* func, size_t smem) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  AttrEntry* a = attr_entry(func, dev);
  if (smem <= a->smem) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) a->smem = smem;
  return e;
}

cudaError_t set_nonportable_cluster(const void* func) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  AttrEntry* a = attr_entry(func, dev);
  if (a->nonportable) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) a->nonportable = true;
  return e;
}

// ---- device limits of the planner ------------------------------------------
namespace {
constexpr int kMaxDev = 64;
std::mutex g_lim_mu;
bool g_lim_known[kMaxDev] = {};
DeviceLimits g_lim[kMaxDev];
bool g_lim_override = false;
DeviceLimits g_lim_forced;
// co-resident clusters per (device, cell, direction, shape)
std::map<std::tuple<int, int, int, int, int, int, int, int, int, size_t>, int> g_cap;

int capacity_cb(int fn, bool bwd, const FusedShape& fs) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  const auto key = std::make_tuple(dev, fn, (int)bwd, fs.C, fs.NT, fs.KT, fs.MT, (int)fs.allg, fs.warps, fs.smem);
  {
    std::lock_guard<std::mutex> lock(g_lim_mu);
    auto it = g_cap.find(key);
    if (it != g_cap.end()) return it->second;
  }
  const int cap = fused_capacity(fn, bwd, fs);
  if (cap >= 0) {
    std::lock_guard<std::mutex> lock(g_lim_mu);
    g_cap[key] = cap;
  }
  return cap;
}
}  // namespace

int cluster_capacity_of(const void* func, const FusedShape& sh) {
  if (set_smem_attr(func, sh.smem) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  if (sh.C > 8 && set_nonportable_cluster(func) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;  // the device refuses clusters above the portable size
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sh.C);
  cfg.blockDim = dim3(sh.warps * 32);
  cfg.dynamicSmemBytes = sh.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = sh.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, func, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  return clusters;
}

// The limits the planner uses: forced ones (rnn_plan_set_limits), else those
// of the current device (SM count, opt-in shared memory per block, cluster
// co-residency asked per candidate), else the GB300 defaults when no device
// can be asked (a size query on a host without a GPU).
DeviceLimits device_limits() {
  std::lock_guard<std::mutex> lock(g_lim_mu);
  if (g_lim_override) return g_lim_forced;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    (void)cudaGetLastError();
    return DeviceLimits{};
  }
  if (!g_lim_known[dev]) {
    DeviceLimits l;
    int sms = 0, smem = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || sms < 1) {
      (void)cudaGetLastError();
      return DeviceLimits{};
    }
    l.sms = sms;
    l.smem_per_cta = (size_t)smem;
    l.cluster_capacity = capacity_cb;
    g_lim[dev] = l;
    g_lim_known[dev] = true;
  }
  return g_lim[dev];
}

int device_sms() { return device_limits().sms; }

// Optional events recorded around the scan kernel (rnn_profile_events).
static cudaEvent_t g_prof[2][2] = {{nullptr, nullptr}, {nullptr, nullptr}};
static void prof_mark(int which, int edge, cudaStream_t st) {
  if (g_prof[which][edge]) cudaEventRecord(g_prof[which][edge], st);
}

static inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Sizes {
  int G, S, K;
  size_t esize, wx, r, bias, st, st0, tape, dr;
};

bool dims_ok(const rnn_dims_t* d) {
  return d && d->B >= 1 && d->T >= 0 && d->N >= 1 && d->D >= 1 && d->function >= 0 &&
         d->function <= 4 && (d->dtype == RNN_F32 || d->dtype == RNN_BF16) && d->path >= 0 &&
         d->path <= 4 && (size_t)d->B * d->N * d->D < ((size_t)1 << 40);
}

static Sizes sizes_of(const rnn_dims_t* d) {
  Sizes z;
  z.G = fn_gates(d->function);
  z.S = fn_states(d->function);
  z.K = fn_tape(d->function);
  z.esize = d->dtype == RNN_BF16 ? 2 : 4;
  const size_t B = d->B, T = d->T, N = d->N, D = d->D;
  z.wx = B * T * z.G * N * D;
  z.r = (size_t)z.G * N * D * D;
  z.bias = (size_t)z.G * N * D;
  z.st = (size_t)z.S * B * T * N * D;
  z.st0 = (size_t)z.S * B * N * D;
  z.tape = T * B * N * z.K * D * sizeof(float);
  z.dr = z.wx * z.esize;
  return z;
}

static bool aligned(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Workspace layout: [status 256 B][path scratch][dr buffer (bwd)][db partials of the
// persistent backward kernels (bwd)][split-K partials of the weight gradients
// (bwd)][tape (bwd recompute)]
struct WsLayout {
  size_t status, path, dr, dbp, wg, tape, total;
};

static WsLayout ws_layout(const rnn_dims_t* d, int kind, const Plan& plan) {
  WsLayout w;
  Sizes z = sizes_of(d);
  w.status = 0;
  w.path = 256;
  size_t off = w.path + align256(plan.scratch_bytes);
  w.dr = off;
  if (kind != RNN_WS_FWD) off += align256(z.dr);
  w.dbp = off;  // [ceil(B / 8) batch blocks][G][N][D] fp32: enough for any block height
  if (kind != RNN_WS_FWD) off += align256((size_t)((d->B + 7) / 8) * z.bias * sizeof(float));
  w.wg = off;
  if (kind != RNN_WS_FWD) {
    size_t wg = wgrad_scratch_bytes(d->B, d->T, d->N, d->D, z.G, d->dtype);
    // dR beside the grid backward: one fp32 partial per chunk
    const size_t beside = d->dtype == RNN_BF16 && d->D % 64 == 0 && d->D >= 256
                              ? (size_t)DR_BESIDE_CHUNKS * z.r * sizeof(float) : 0;
    off += align256(wg > beside ? wg : beside);
  }
  w.tape = off;
  if (kind == RNN_WS_BWD_RECOMPUTE) off += align256(z.tape);
  w.total = off;
  return w;
}

static int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return RNN_OK;
  fprintf(stderr, "librnn_gb300: CUDA error: %s\n", cudaGetErrorString(e));
  return RNN_ECUDA;
}

// Plans are cached per (dims, direction, device, limits in force, planner
// restriction variables): the enumeration and its co-residency queries run
// once per shape, not on every call.
namespace {
std::mutex g_plan_mu;
std::map<std::string, std::pair<int, Plan>> g_plans;
}  // namespace

static int choose(const rnn_dims_t* d, bool bwd, Plan* plan) {
  const DeviceLimits lim = device_limits();
  int dev = -1;  // stated limits (no device query) or no device: -1
  if (lim.cluster_capacity && cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    dev = -1;
  }
  char key[320];
  int n = snprintf(key, sizeof(key), "%d %d %d %d %d %d %d %d | %d %d %d %zu %d |", d->B, d->T, d->N, d->D,
                   d->function, d->dtype, d->path, (int)bwd, dev, lim.sms, lim.max_cluster, lim.smem_per_cta,
                   lim.cluster_capacity != nullptr);
  for (const char* v : {"RNN_PLAN_C", "RNN_PLAN_NT", "RNN_PLAN_KT", "RNN_PLAN_MT", "RNN_PLAN_ALLG"}) {
    const char* e = getenv(v);
    if (n > 0 && n < (int)sizeof(key)) n += snprintf(key + n, sizeof(key) - n, " %s", e ? e : "-");
  }
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    auto it = g_plans.find(key);
    if (it != g_plans.end()) {
      *plan = it->second.second;
      return it->second.first;
    }
  }
  PlanRequest q{d->B, d->T, d->N, d->D, d->function, d->dtype, d->path, bwd, &lim};
  const int rc = plan_select(q, plan);
  std::lock_guard<std::mutex> lock(g_plan_mu);
  g_plans[key] = std::make_pair(rc, *plan);
  return rc;
}

// Grid path scratch inside the workspace (after the 256-byte status word):
// the exchange buffers [2][groups][BC][L] bf16 (L = D forward, G D backward)
// followed by one step counter per group.
static void grid_scratch(const rnn_dims_t* d, const Plan& plan, char* ws, bool bwd, FusedArgs* f) {
  const size_t L = bwd ? (size_t)fn_gates(d->function) * d->D : (size_t)d->D;
  const size_t hx = (size_t)2 * plan.groups * 8 * plan.fs.NT * L * 2;
  f->hx = ws + 256;
  // the counter region starts on a 1 KB boundary: its blocks are the units
  // whose L2 home die is measured
  const uintptr_t c = ((uintptr_t)(ws + 256 + align256(hx)) + 1023) & ~(uintptr_t)1023;
  f->counters = (unsigned int*)c;
}

// Bytes of the counter region zeroed before each grid launch: the counters
// (one per group, or one per 1 KB block under die placement) and the tickets.
static size_t grid_counter_bytes(const Plan& plan) {
  const size_t words = plan.groups > GRID_CTR_BLOCKS * 256 ? (size_t)plan.groups : (size_t)GRID_CTR_BLOCKS * 256;
  return words * sizeof(unsigned) + 256;
}

// Die placement of the grid kernels' batch groups: each group's C CTAs on one
// die of the GPU and its step counter in a block homed on that die, so that
// the exchange's L2 round trips stay on the die (about 1750 cycles each
// instead of about 3000 when a leg crosses). Off (groups by block index) when
// die_plan declines.
static void grid_die_setup(const Plan& plan, cudaStream_t st, FusedArgs* f) {
  DiePlan p;
  if (!die_plan(plan.groups, plan.fs.C, f->counters, st, &p)) return;
  for (int g = 0; g < plan.groups; ++g) f->ctr_word[g] = p.ctr_word[g];
  f->die_of_sm = p.table;
  f->tickets = f->counters + GRID_CTR_BLOCKS * 256;
  for (int d = 0; d < 2; ++d) {
    f->die_grp0[d] = p.grp0[d];
    f->die_ngrp[d] = p.ngrp[d];
  }
  f->launch_ctas = p.sms;
}

// dR beside the grid backward (dr_beside.cuh): the launch's spare CTAs take
// the tiles of chunks of steps the scan has finished, so that after the scan
// only the sum of the chunks' partials is left. Chunks of 64-step tiles in
// the scan's order, shrinking toward t = 0 (6 : 4 : 3 : 2 : 1), so that the
// chunk still open when the scan ends is short. Off when RNN_DR_BESIDE=0,
// for fp32, D not a multiple of 64 or under 256, fewer than 16 tiles of
// steps, fewer than 8 spare SMs, or a workspace without room.
static bool dr_beside_setup(const rnn_dims_t* d, const Plan& plan, const Sizes& z, const void* states,
                            const void* states0, void* drbuf, void* dR, char* slots, size_t slot_bytes,
                            FusedArgs* f, UmmaMaps* dm) {
  const char* env = getenv("RNN_DR_BESIDE");
  if ((env && env[0] == '0') || !dR || d->dtype != RNN_BF16 || d->D % 64 || d->D < 256) return false;
  const int nt = (d->T + UM_BK - 1) / UM_BK;
  // the worker runs on four warps (TMEM lanes and a 128-thread barrier)
  if (nt < 16 || plan.fs.warps < 4 || plan.groups * plan.fs.C + 8 > device_sms()) return false;
  if ((size_t)DR_BESIDE_CHUNKS * z.r * sizeof(float) > slot_bytes) return false;
  static const int weight[DR_BESIDE_CHUNKS] = {6, 4, 3, 2, 1};
  int left = nt, hi = nt;
  for (int c = 0; c < DR_BESIDE_CHUNKS; ++c) {
    int n = c + 1 < DR_BESIDE_CHUNKS ? (nt * weight[c] + 8) / 16 : left;
    if (n < 1) n = 1;
    if (n > left - (DR_BESIDE_CHUNKS - 1 - c)) n = left - (DR_BESIDE_CHUNKS - 1 - c);
    f->drw.tt_n[c] = n;
    f->drw.tt_lo[c] = hi - n;
    hi -= n;
    left -= n;
  }
  WgradArgs wa{d->B, d->T, d->N, d->D, z.G, states, states0, drbuf, dR, nullptr};
  if (umma_encode_maps(wa, 256, true, dm) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  f->drw.nc = DR_BESIDE_CHUNKS;
  f->drw.s0_tiles = states0 ? (d->B + UM_BK - 1) / UM_BK : 0;
  f->drw.slots = (float*)slots;
  f->drw.next = f->counters + GRID_CTR_BLOCKS * 256 + 32;  // in the tickets' line, zeroed with the counters
  return true;
}

// Alternating path scratch inside the workspace: the bf16 ping-pong buffer,
// then the fp32 carried values.
static void alt_scratch(const rnn_dims_t* d, char* ws, bool bwd, AltArgs* a) {
  const size_t per = (size_t)d->B * d->N * d->D;
  const size_t x = bwd ? 2 * per * fn_gates(d->function) * 2 : 2 * per * 2;
  a->xbuf = ws + 256;
  a->cst = (float*)(ws + 256 + align256(x));
}

// Upper bound of every device-side wait.
static unsigned long long g_wait_limit_ns = 2000000000ull;
unsigned long long wait_limit_ns() { return g_wait_limit_ns; }

// Phase trace of the persistent kernels (rnn_trace).
static unsigned long long* g_trace_buf = nullptr;
static int g_trace_t0 = 0, g_trace_steps = 0;
// Fault injection of the forward persistent kernels (rnn_debug_inject_wait).
static int g_inject_step = -1;
static unsigned long long g_inject_limit_ns = 0;

static void with_trace(FusedArgs* f) {
  f->trace = g_trace_buf;
  f->trace_t0 = g_trace_t0;
  f->trace_steps = g_trace_steps;
  f->inject_step = g_inject_step;
  f->inject_limit_ns = g_inject_limit_ns;
}

// Runs the forward kernels (states/last/tape each optional); ws is the
// workspace base (status word at offset 0).
static int run_forward(const rnn_dims_t* d, const Plan& plan, const void* Wx, const void* R,
                       const void* b, const void* s0, void* states, void* last, float* tape,
                       char* ws, cudaStream_t st) {
  SimtArgs a{};
  a.B = d->B; a.T = d->T; a.N = d->N; a.D = d->D;
  a.Wx = Wx; a.R = R; a.bias = b; a.s0 = s0;
  a.states = states; a.last = last; a.tape = tape;
  a.trace = g_trace_buf; a.trace_t0 = g_trace_t0; a.trace_steps = g_trace_steps;
  int rc = RNN_EUNSUPPORTED;
  prof_mark(0, 0, st);
  switch (plan.path) {
    case RNN_PATH_SIMT:
      rc = cuda_status(simt_run(d->function, d->dtype, a, false, st));
      break;
    case RNN_PATH_FUSED: {
      FusedArgs f{};
      f.B = d->B; f.T = d->T; f.N = d->N; f.D = d->D;
      f.C = plan.fs.C; f.U = plan.fs.U; f.KS = plan.fs.KS;
      f.Wx = Wx; f.R = R; f.bias = b; f.s0 = s0;
      f.states = states; f.last = last; f.tape = tape;
      f.status = (unsigned int*)ws;
      f.wait_limit_ns = g_wait_limit_ns;
      with_trace(&f);
      rc = cuda_status(fused_fwd_run(d->function, plan.fs, f, st));
      break;
    }
    case RNN_PATH_GRID: {
      FusedArgs f{};
      f.B = d->B; f.T = d->T; f.N = d->N; f.D = d->D;
      f.C = plan.fs.C; f.U = plan.fs.U; f.KS = plan.fs.KS;
      f.Wx = Wx; f.R = R; f.bias = b; f.s0 = s0;
      f.states = states; f.last = last; f.tape = tape;
      f.status = (unsigned int*)ws;
      f.wait_limit_ns = g_wait_limit_ns;
      with_trace(&f);
      grid_scratch(d, plan, ws, false, &f);
      grid_die_setup(plan, st, &f);
      rc = cuda_status(cudaMemsetAsync(f.counters, 0, grid_counter_bytes(plan), st));
      if (rc == RNN_OK) rc = cuda_status(grid_fwd_run(d->function, plan.fs, f, st));
      break;
    }
    case RNN_PATH_ALTERNATING: {
      AltArgs g{};
      g.B = d->B; g.T = d->T; g.N = d->N; g.D = d->D;
      g.Wx = Wx; g.R = R; g.bias = b; g.s0 = s0;
      g.states = states; g.last = last; g.tape = tape;
      alt_scratch(d, ws, false, &g);
      rc = cuda_status(alt_fwd_run(d->function, g, st));
      break;
    }
  }
  prof_mark(0, 1, st);
  return rc;
}

}  // namespace rnn

using namespace rnn;

extern "C" {

int rnn_num_gates(int function) { return function >= 0 && function <= 4 ? fn_gates(function) : -1; }
int rnn_num_states(int function) { return function >= 0 && function <= 4 ? fn_states(function) : -1; }

size_t rnn_tape_size(const rnn_dims_t* d) {
  if (!dims_ok(d)) return 0;
  return sizes_of(d).tape;
}

size_t rnn_workspace_size(const rnn_dims_t* d, int kind) {
  if (!dims_ok(d) || kind < 0 || kind > 2) return 0;
  Plan plan;
  if (choose(d, kind != RNN_WS_FWD, &plan) != RNN_OK) {
    // size for the plain path so that callers can still allocate
    plan = Plan{};
    plan.path = RNN_PATH_SIMT;
  }
  if (kind == RNN_WS_BWD_RECOMPUTE) {
    Plan fplan;
    if (choose(d, false, &fplan) == RNN_OK && fplan.scratch_bytes > plan.scratch_bytes)
      plan.scratch_bytes = fplan.scratch_bytes;
  }
  return ws_layout(d, kind, plan).total;
}

int rnn_fwd(const rnn_dims_t* d, const void* Wx, const void* R, const void* b,
            const void* states0, void* states, void* last, void* tape, void* workspace,
            size_t ws_bytes, void* stream) {
  if (!dims_ok(d)) return RNN_EINVAL;
  if (!R || !b || !workspace || (d->T > 0 && (!Wx || !states))) return RNN_EINVAL;
  const void* ptrs[] = {Wx, R, b, states0, states, last, tape, workspace};
  for (const void* p : ptrs)
    if (p && !aligned(p)) return RNN_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  Sizes z = sizes_of(d);
  Plan plan;
  int rc = choose(d, false, &plan);
  if (rc != RNN_OK) return rc;
  WsLayout w = ws_layout(d, RNN_WS_FWD, plan);
  if (ws_bytes < w.total) return RNN_ENOSPC;
  char* ws = (char*)workspace;
  rc = cuda_status(cudaMemsetAsync(ws + w.status, 0, 256, st));
  if (rc) return rc;
  if (d->T == 0) {
    if (!last) return RNN_OK;
    if (states0) return cuda_status(cudaMemcpyAsync(last, states0, z.st0 * z.esize, cudaMemcpyDeviceToDevice, st));
    return cuda_status(cudaMemsetAsync(last, 0, z.st0 * z.esize, st));
  }
  return run_forward(d, plan, Wx, R, b, states0, states, last, (float*)tape, ws, st);
}

int rnn_bwd(const rnn_dims_t* d, const void* Wx, const void* R, const void* b,
            const void* states0, const void* states, const void* tape, const void* dstates,
            const void* dlast, void* dWx, void* dR, void* db, void* dstates0, void* workspace,
            size_t ws_bytes, void* stream) {
  if (!dims_ok(d)) return RNN_EINVAL;
  if (!R || !b || !workspace || (d->T > 0 && (!Wx || !states))) return RNN_EINVAL;
  const void* ptrs[] = {Wx, R, b, states0, states, tape, dstates, dlast, dWx, dR, db, dstates0, workspace};
  for (const void* p : ptrs)
    if (p && !aligned(p)) return RNN_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  Sizes z = sizes_of(d);
  Plan plan;
  int rc = choose(d, true, &plan);
  if (rc != RNN_OK) return rc;
  const int kind = tape ? RNN_WS_BWD : RNN_WS_BWD_RECOMPUTE;
  size_t need = rnn_workspace_size(d, kind);
  if (ws_bytes < need) return RNN_ENOSPC;
  WsLayout w = ws_layout(d, kind, plan);
  char* ws = (char*)workspace;
  rc = cuda_status(cudaMemsetAsync(ws + w.status, 0, 256, st));
  if (rc) return rc;
  if (d->T == 0) {
    if (dstates0) {
      rc = dlast ? cuda_status(cudaMemcpyAsync(dstates0, dlast, z.st0 * z.esize, cudaMemcpyDeviceToDevice, st))
                 : cuda_status(cudaMemsetAsync(dstates0, 0, z.st0 * z.esize, st));
      if (rc) return rc;
    }
    if (dR && (rc = cuda_status(cudaMemsetAsync(dR, 0, z.r * z.esize, st)))) return rc;
    if (db && (rc = cuda_status(cudaMemsetAsync(db, 0, z.bias * z.esize, st)))) return rc;
    return RNN_OK;
  }
  const float* tp = (const float*)tape;
  if (!tp) {
    Plan fplan;
    rc = choose(d, false, &fplan);
    if (rc != RNN_OK) return rc;
    float* t2 = (float*)(ws + w.tape);
    rc = run_forward(d, fplan, Wx, R, b, states0, nullptr, nullptr, t2, ws, st);
    if (rc) return rc;
    tp = t2;
  }
  SimtArgs a{};
  a.B = d->B; a.T = d->T; a.N = d->N; a.D = d->D;
  a.R = R; a.s0 = states0; a.tape = (float*)tp;
  a.trace = g_trace_buf; a.trace_t0 = g_trace_t0; a.trace_steps = g_trace_steps;
  // the recurrent-branch gradient equals dWx except for the GRU candidate gate:
  // reuse dWx as the weight-gradient operand when it is there
  void* drbuf = (d->function != RNN_GRU && dWx) ? dWx : (void*)(ws + w.dr);
  a.dstates = dstates; a.dlast = dlast; a.dWx = dWx; a.dr = drbuf; a.ds0 = dstates0;
  rc = RNN_EUNSUPPORTED;
  int dbp_blocks = 0;  // > 0: the scan kernel left db partials at ws + w.dbp
  int dr_parts = 0;    // > 0: the scan kernel left dR as that many fp32 partials at ws + w.wg
  prof_mark(1, 0, st);
  switch (plan.path) {
    case RNN_PATH_SIMT:
      if ((dR || db) && simt_fuses_wgrad(d->function, d->B, d->T, d->D)) {
        a.fuse_wgrad = 1;  // dR and db from the backward kernel itself
        a.dR = dR;
        a.db = db;
      }
      rc = cuda_status(simt_run(d->function, d->dtype, a, true, st));
      break;
    case RNN_PATH_FUSED: {
      FusedArgs f{};
      f.B = d->B; f.T = d->T; f.N = d->N; f.D = d->D;
      f.C = plan.fs.C; f.U = plan.fs.U; f.KS = plan.fs.KS;
      f.R = R; f.s0 = states0; f.tape = (float*)tp;
      f.dstates = dstates; f.dlast = dlast; f.dWx = dWx; f.dr = drbuf; f.ds0 = dstates0;
      f.status = (unsigned int*)ws;
      f.wait_limit_ns = g_wait_limit_ns;
      if (db && d->dtype == RNN_BF16) {  // db summed inside the kernel, per batch block
        f.dbp = (float*)(ws + w.dbp);
        dbp_blocks = (d->B + 8 * plan.fs.NT - 1) / (8 * plan.fs.NT);
      }
      with_trace(&f);
      rc = cuda_status(fused_bwd_run(d->function, plan.fs, f, st));
      break;
    }
    case RNN_PATH_GRID: {
      FusedArgs f{};
      f.B = d->B; f.T = d->T; f.N = d->N; f.D = d->D;
      f.C = plan.fs.C; f.U = plan.fs.U; f.KS = plan.fs.KS;
      f.R = R; f.s0 = states0; f.tape = (float*)tp;
      f.dstates = dstates; f.dlast = dlast; f.dWx = dWx; f.dr = drbuf; f.ds0 = dstates0;
      f.status = (unsigned int*)ws;
      f.wait_limit_ns = g_wait_limit_ns;
      if (db && d->dtype == RNN_BF16) {  // db summed inside the kernel, per batch block
        f.dbp = (float*)(ws + w.dbp);
        dbp_blocks = (d->B + 8 * plan.fs.NT - 1) / (8 * plan.fs.NT);
      }
      with_trace(&f);
      grid_scratch(d, plan, ws, true, &f);
      grid_die_setup(plan, st, &f);
      UmmaMaps dm;
      bool beside = dr_beside_setup(d, plan, z, states, states0, drbuf, dR, ws + w.wg, w.tape - w.wg, &f, &dm);
      rc = cuda_status(cudaMemsetAsync(f.counters, 0, grid_counter_bytes(plan), st));
      if (rc == RNN_OK) {
        cudaError_t e = grid_bwd_run(d->function, plan.fs, f, st, beside ? &dm : nullptr);
        if (e == cudaErrorNotSupported && beside) {  // no spare CTAs after all: dR after the scan
          (void)cudaGetLastError();
          f.drw.nc = 0;
          beside = false;
          e = grid_bwd_run(d->function, plan.fs, f, st);
        }
        rc = cuda_status(e);
      }
      if (beside) dr_parts = f.drw.nc;
      break;
    }
    case RNN_PATH_ALTERNATING: {
      AltArgs g{};
      g.B = d->B; g.T = d->T; g.N = d->N; g.D = d->D;
      g.R = R; g.s0 = states0; g.tape = (float*)tp;
      g.dstates = dstates; g.dlast = dlast; g.dWx = dWx; g.dr = drbuf; g.ds0 = dstates0;
      alt_scratch(d, ws, true, &g);
      rc = cuda_status(alt_bwd_run(d->function, g, st));
      break;
    }
  }
  prof_mark(1, 1, st);
  if (rc) return rc;
  if ((dR || db) && !a.fuse_wgrad) {
    WgradArgs g{d->B, d->T, d->N, d->D, z.G, states, states0, drbuf, dR, db};
    g.scratch = (float*)(ws + w.wg);
    g.scratch_bytes = w.tape - w.wg;
    g.status = (unsigned int*)ws;
    g.wait_limit_ns = g_wait_limit_ns;
    if (dbp_blocks > 0) {
      g.dbp = (const float*)(ws + w.dbp);
      g.dbp_blocks = dbp_blocks;
    }
    rc = cuda_status(dr_parts > 0 ? wgrad_sum_partials(g, dr_parts, st) : wgrad_run(d->dtype, g, st));
  }
  return rc;
}

int rnn_check_status(void* workspace, void* stream) {
  if (!workspace) return RNN_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned int h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  if (h != STATUS_OK) {
    e = cudaMemsetAsync(workspace, 0, sizeof(h), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e);
    return RNN_ETIMEOUT;
  }
  return RNN_OK;
}

int rnn_die_layout(int* sms_die0, int* sms_die1) {
  int dev = 0, cnt[2] = {0, 0}, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RNN_ECUDA;
  if (!die_counts(dev, cnt, &sms)) return RNN_EUNSUPPORTED;
  if (sms_die0) *sms_die0 = cnt[0];
  if (sms_die1) *sms_die1 = cnt[1];
  return RNN_OK;
}

int rnn_die_plan_for(int groups, int C, const unsigned long long* sm_lat, int nsm,
                     const unsigned long long* blk_lat, int nblocks, int* sms_die0, int* sms_die1,
                     int* groups_die0, int* ctr_words) {
  if (groups < 1 || groups > GRID_CTR_BLOCKS || groups > FUSED_MAX_GROUP_CTR || C < 1 || !sm_lat || nsm < 2 ||
      nsm > 4096 || !blk_lat || nblocks < 1 || nblocks > GRID_CTR_BLOCKS)
    return RNN_EINVAL;
  std::vector<signed char> die(nsm);
  int cnt[2] = {0, 0};
  if (!classify_sms(sm_lat, nsm, die.data(), cnt)) return RNN_EUNSUPPORTED;
  if (sms_die0) *sms_die0 = cnt[0];
  if (sms_die1) *sms_die1 = cnt[1];
  const int g0 = die_split_groups(groups, C, cnt);
  signed char home[GRID_CTR_BLOCKS];
  int words[GRID_CTR_BLOCKS];
  if (g0 < 0 || !classify_blocks(blk_lat, nblocks, home) || !die_assign_counters(groups, g0, home, nblocks, words))
    return RNN_EUNSUPPORTED;
  if (groups_die0) *groups_die0 = g0;
  if (ctr_words)
    for (int g = 0; g < groups; ++g) ctr_words[g] = words[g];
  return RNN_OK;
}

int rnn_plan_set_limits(int sms, int smem_per_cta, int max_cluster) {
  std::lock_guard<std::mutex> lock(g_lim_mu);
  if (sms <= 0) {
    g_lim_override = false;
    return RNN_OK;
  }
  if (sms > 4096 || smem_per_cta < 1024 || smem_per_cta > (1 << 20) || max_cluster < 1 || max_cluster > 16)
    return RNN_EINVAL;
  DeviceLimits l;
  l.sms = sms;
  l.smem_per_cta = (size_t)smem_per_cta;
  l.max_cluster = max_cluster;
  l.cluster_capacity = nullptr;  // a stated device: co-residency from the SM count alone
  g_lim_forced = l;
  g_lim_override = true;
  return RNN_OK;
}

int rnn_plan_describe(const rnn_dims_t* d, int for_backward, char* buf, size_t len) {
  if (!dims_ok(d) || !buf || len == 0) return RNN_EINVAL;
  Plan plan;
  int rc = choose(d, for_backward != 0, &plan);
  plan_describe(plan, rc, buf, len);
  return rc;
}

unsigned long long rnn_kernel_launches(void) { return g_launches.load(); }

int rnn_profile_events(int which, void* before, void* after) {
  if (which < 0 || which > 1) return RNN_EINVAL;
  g_prof[which][0] = (cudaEvent_t)before;
  g_prof[which][1] = (cudaEvent_t)after;
  return RNN_OK;
}

int rnn_trace(void* buf, int t0, int steps) {
  if (buf && (t0 < 0 || steps < 1)) return RNN_EINVAL;
  g_trace_buf = (unsigned long long*)buf;
  g_trace_t0 = buf ? t0 : 0;
  g_trace_steps = buf ? steps : 0;
  return RNN_OK;
}

int rnn_debug_inject_wait(int step, unsigned long long limit_ns) {
  if (step >= 0 && (limit_ns == 0 || limit_ns > 10000000000ull)) return RNN_EINVAL;
  g_inject_step = step < 0 ? -1 : step;
  g_inject_limit_ns = step < 0 ? 0 : limit_ns;
  return RNN_OK;
}

const char* rnn_strerror(int status) {
  switch (status) {
    case RNN_OK: return "ok";
    case RNN_EINVAL: return "invalid argument (dimensions, null pointer or alignment)";
    case RNN_EUNSUPPORTED: return "no feasible kernel plan for the requested path";
    case RNN_ENOSPC: return "workspace too small";
    case RNN_ETIMEOUT: return "a device-side wait timed out";
    case RNN_ECUDA: return "CUDA runtime error";
  }
  return "unknown status";
}

}  // extern "C"
