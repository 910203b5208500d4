// rnn_bwd_noalloc: the backward through time for callers that cannot
// allocate device memory (see include/rnn.h).
//
// The backward normally needs caller-provided workspace: a status word and,
// for GRU (or when dWx is not requested), a buffer for the recurrent-branch
// gradients that the weight-gradient pass reads, plus optional split-K
// partial sums. Here that scratch is a file-scope __device__ array of fixed
// size instead. Every GPU that loads the library holds the array until the
// process exits. Every call shares it, so calls whose work overlaps on the GPU
// (two streams, or two threads) race on it; calls on one stream run one after
// another and are safe.
#include <mutex>

#include "kernels.cuh"
#include "plan.h"
#include "rnn.h"

namespace rnn {

bool dims_ok(const rnn_dims_t* d);  // api.cu: the argument bounds every entry point shares

// [0, 256): device status word of the bounded waits; [256, ...): recurrent-
// branch gradients [B][T][G][N][D] in the storage type when needed, then
// whatever is left serves as the weight gradient's split-K scratch.
static __device__ __align__(256) unsigned char g_bwd_scratch[RNN_BWD_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t kStatusBytes = 256;

std::mutex g_mu;
constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device, looked up once per
// device (the host-side symbol is only a stand-in, never a device address).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RNN_ECUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess || !p) return RNN_ECUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return RNN_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace
}  // namespace rnn

using namespace rnn;

extern "C" int rnn_bwd_noalloc(const rnn_dims_t* d, const void* Wx, const void* R, const void* b,
                               const void* states0, const void* states, const void* tape,
                               const void* dstates, const void* dlast, void* dWx, void* dR, void* db,
                               void* dstates0, void* stream) {
  if (!dims_ok(d)) return RNN_EINVAL;
  if (!R || !b || (d->T > 0 && (!Wx || !states || !tape))) return RNN_EINVAL;
  const void* ptrs[] = {Wx, R, b, states0, states, tape, dstates, dlast, dWx, dR, db, dstates0};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return RNN_EINVAL;
  // the cluster and plain kernels need no scratch beyond dr; the grid and
  // alternating paths need exchange buffers that this entry point does not hold
  if (d->path == RNN_PATH_GRID || d->path == RNN_PATH_ALTERNATING) return RNN_EUNSUPPORTED;
  const int G = fn_gates(d->function), S = fn_states(d->function);
  const size_t e = d->dtype == RNN_BF16 ? 2 : 4;
  const size_t wx_elems = (size_t)d->B * d->T * G * d->N * d->D;
  const bool need_dr = d->function == RNN_GRU || !dWx;
  const size_t dr_bytes = need_dr ? align256(wx_elems * e) : 0;
  const size_t need = kStatusBytes + dr_bytes;
  if (need > (size_t)RNN_BWD_NOALLOC_SCRATCH_BYTES) return RNN_ENOSPC;  // problem too large for the static scratch

  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != RNN_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned char* base = (unsigned char*)scratch;
  if (cudaMemsetAsync(base, 0, kStatusBytes, st) != cudaSuccess) return RNN_ECUDA;  // status starts clear

  const size_t st0 = (size_t)S * d->B * d->N * d->D;
  if (d->T == 0) {
    cudaError_t ce = cudaSuccess;
    if (dstates0)
      ce = dlast ? cudaMemcpyAsync(dstates0, dlast, st0 * e, cudaMemcpyDeviceToDevice, st)
                 : cudaMemsetAsync(dstates0, 0, st0 * e, st);
    if (ce == cudaSuccess && dR) ce = cudaMemsetAsync(dR, 0, (size_t)G * d->N * d->D * d->D * e, st);
    if (ce == cudaSuccess && db) ce = cudaMemsetAsync(db, 0, (size_t)G * d->N * d->D * e, st);
    return ce == cudaSuccess ? RNN_OK : RNN_ECUDA;
  }

  Plan plan;
  PlanRequest q{d->B, d->T, d->N, d->D, d->function, d->dtype, d->path, true};
  rc = plan_select(q, &plan);
  if (rc != RNN_OK) return rc;
  if (plan.path == RNN_PATH_GRID || plan.path == RNN_PATH_ALTERNATING) {
    // AUTO chose a path whose exchange buffers live in a workspace: the plain
    // kernel computes the same backward with no scratch beyond dr
    PlanRequest qs = q;
    qs.path = RNN_PATH_SIMT;
    rc = plan_select(qs, &plan);
    if (rc != RNN_OK) return rc;
  }
  void* drbuf = need_dr ? (void*)(base + kStatusBytes) : dWx;
  cudaError_t ce = cudaErrorInvalidValue;
  if (plan.path == RNN_PATH_SIMT) {
    SimtArgs a{};
    a.B = d->B; a.T = d->T; a.N = d->N; a.D = d->D;
    a.R = R; a.s0 = states0; a.tape = (float*)tape;
    a.dstates = dstates; a.dlast = dlast; a.dWx = dWx; a.dr = drbuf; a.ds0 = dstates0;
    ce = simt_run(d->function, d->dtype, a, true, st);
  } else if (plan.path == RNN_PATH_FUSED) {
    FusedArgs f{};
    f.B = d->B; f.T = d->T; f.N = d->N; f.D = d->D;
    f.C = plan.fs.C; f.U = plan.fs.U; f.KS = plan.fs.KS;
    f.R = R; f.s0 = states0; f.tape = (float*)tape;
    f.dstates = dstates; f.dlast = dlast; f.dWx = dWx; f.dr = drbuf; f.ds0 = dstates0;
    f.status = (unsigned int*)base;
    f.wait_limit_ns = wait_limit_ns();
    ce = fused_bwd_run(d->function, plan.fs, f, st);
  } else {
    return RNN_EUNSUPPORTED;
  }
  if (ce != cudaSuccess) return RNN_ECUDA;
  if (dR || db) {
    WgradArgs g{d->B, d->T, d->N, d->D, G, states, states0, drbuf, dR, db};
    // the rest of the array holds the split-K partial sums when they fit;
    // otherwise the weight-gradient pass runs without splitting K
    const size_t used = kStatusBytes + dr_bytes;
    g.scratch = (float*)(base + used);
    g.scratch_bytes = (size_t)RNN_BWD_NOALLOC_SCRATCH_BYTES - used;
    g.status = (unsigned int*)base;
    g.wait_limit_ns = wait_limit_ns();
    if (wgrad_run(d->dtype, g, st) != cudaSuccess) return RNN_ECUDA;
  }
  return RNN_OK;
}

extern "C" int rnn_bwd_noalloc_status(void* stream) {
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != RNN_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned int h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, scratch, sizeof(h), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return RNN_ECUDA;
  if (h != STATUS_OK) {
    e = cudaMemsetAsync(scratch, 0, sizeof(h), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e == cudaSuccess ? RNN_ETIMEOUT : RNN_ECUDA;
  }
  return RNN_OK;
}
