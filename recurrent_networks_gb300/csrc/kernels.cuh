// Internal declarations shared by the kernel translation units and the C ABI.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "cells.cuh"

namespace rnn {

// Counts kernel launches for rnn_kernel_launches(); every launcher calls it.
void note_launch(int count = 1);

// The upper bound (ns) every device-side wait of the library's kernels uses.
unsigned long long wait_limit_ns();

// cudaFuncSetAttribute, called once per (device, kernel) for the largest
// dynamic shared memory requested so far (and once for the non-portable
// cluster size): the runtime call costs microseconds of host time that a
// small problem's launch would otherwise pay on every call.
cudaError_t set_smem_attr(const void* func, size_t smem);
cudaError_t set_nonportable_cluster(const void* func);

// Arguments of the plain per-head kernels (and of the weight-gradient pass).
struct SimtArgs {
  int B, T, N, D, BB;
  int r_smem = 0;  // 1: the head's R (fp32) is staged in shared memory (transposed for the backward)
  const void* Wx;
  const void* R;
  const void* bias;
  const void* s0;
  void* states;
  void* last;
  float* tape;  // fwd: out (may be null); bwd: in
  const void* dstates;
  const void* dlast;
  void* dWx;
  void* dr;  // bwd: recurrent-branch gradients [B,T,G,N,D] (storage type)
  void* ds0;
  // bwd: dR and db computed by the backward kernel itself (simt_fuses_wgrad)
  int fuse_wgrad = 0;
  void* dR = nullptr;
  void* db = nullptr;
  // optional phase trace (rnn_trace): CTA 0, thread 0 writes clock64() at the
  // phase points of steps [trace_t0, trace_t0 + trace_steps) (processing order)
  unsigned long long* trace = nullptr;
  int trace_t0 = 0, trace_steps = 0;
};

int simt_supported(int fn, int B, int D, bool bwd);
// Whether the plain backward computes dR and db itself: one CTA holds every
// batch row of a head, the problem is small (G D^2 B T <= 2^21) and the
// steps' recurrent-branch gradients and h_{t-1} fit in shared memory.
bool simt_fuses_wgrad(int fn, int B, int T, int D);
cudaError_t simt_run(int fn, int dtype, const SimtArgs& a, bool bwd, cudaStream_t st);

// dR[g,n,i,j] = sum_{b,t} hprev[b,t,n,i] dr[b,t,g,n,j];  db[g,n,j] = sum_{b,t} dr[b,t,g,n,j]
// with hprev[b,t] = states[0,b,t-1] (t > 0) or states0[0,b,0] (t = 0, zeros if null).
struct WgradArgs {
  int B, T, N, D, G;
  const void* states;
  const void* s0;
  const void* dr;
  void* dR;  // may be null
  void* db;  // may be null
  float* scratch = nullptr;  // optional: split-K partial sums (wgrad_scratch_bytes)
  size_t scratch_bytes = 0;
  // optional: db already summed by the backward scan kernel per batch block,
  // fp32 [dbp_blocks][G][N][D]; db is then their sum in block order
  const float* dbp = nullptr;
  int dbp_blocks = 0;
  unsigned int* status = nullptr;  // device status word for the bounded waits (may be null)
  unsigned long long wait_limit_ns = 2000000000ull;
};
// Bytes of split-K scratch the tensor-core weight-gradient pass can use.
size_t wgrad_scratch_bytes(int B, int T, int N, int D, int G, int dtype);
cudaError_t wgrad_run(int dtype, const WgradArgs& a, cudaStream_t st);
// dR as the sum of `parts` fp32 partials [parts][G][N][D][D] at a.scratch
// (added in part order), then db: for dR computed beside the backward scan.
cudaError_t wgrad_sum_partials(const WgradArgs& a, int parts, cudaStream_t st);

constexpr int FUSED_MAX_GROUP_CTR = 16;  // groups whose counter word FusedArgs::ctr_word places

// One-time measurements of the GPU's two dies (dies.cu): the SM count on
// each die (false when the device shows no two-die structure or cannot be
// measured now), the device table of the die of each SM id, and the home
// die of each 1 KB block of `region` (measured on stream `st` once per
// address; false while `st` is capturing or when the homes are unclear).
bool die_counts(int dev, int count[2], int* sms);
const signed char* die_table_device();
bool block_homes(int dev, unsigned* region, int nblocks, cudaStream_t st, signed char* home);
// Die placement of `groups` groups of C CTAs whose step counters live in the
// 16 1 KB blocks of `ctr_region` (1 KB aligned): groups [0, ngrp[0]) on die
// 0, the rest on die 1, the split closest to even that fits each die; each
// group's counter at the start of a block homed on its die (word ctr_word[g]
// of the region); launched as one CTA per SM (sms). False (block-index
// placement) when RNN_DIE_PLACEMENT=0, the dies or the homes cannot be
// measured, or the groups do not fit.
struct DiePlan {
  const signed char* table = nullptr;
  int grp0[2] = {0, 0}, ngrp[2] = {0, 0};
  int ctr_word[16] = {};
  int sms = 0;
};
bool die_plan(int groups, int C, unsigned* ctr_region, cudaStream_t st, DiePlan* out);

// Arguments of the persistent cluster kernels (bf16 storage).
struct FusedArgs {
  int B, T, N, D, C, U, KS;
  const void* Wx;
  const void* R;
  const void* bias;
  const void* s0;
  void* states;  // may be null (tape-only forward)
  void* last;    // may be null
  float* tape;   // may be null
  const void* dstates;
  const void* dlast;
  void* dWx;
  void* dr;
  void* ds0;
  // optional (backward): fp32 [B / BC blocks][G][N][D], each CTA's column
  // sums of dr over its batch block and all steps (db partials)
  float* dbp = nullptr;
  unsigned int* status;  // device status word (bounded waits)
  unsigned long long wait_limit_ns;
  // grid mode (cooperative persistent kernel): h exchange buffers
  // [2][groups][BC][D] and one step counter per group, zeroed before launch;
  // group g's counter is word ctr_word[g] of `counters` (g < 16), word g above
  void* hx = nullptr;
  unsigned int* counters = nullptr;
  int ctr_word[16] = {0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15};
  // die placement (grid mode, optional): with die_of_sm set (the SM-id ->
  // die table) the launch holds one CTA per SM; groups [die_grp0[d],
  // die_grp0[d] + die_ngrp[d]) run on die d, a CTA taking its (group, rank)
  // from ticket d (zeroed before launch), and the spare CTAs leave
  const signed char* die_of_sm = nullptr;
  unsigned int* tickets = nullptr;
  int die_grp0[2] = {0, 0}, die_ngrp[2] = {0, 0};
  int launch_ctas = 0;  // die placement: CTAs launched (the SM count)
  int groups = 0;       // grid mode: the launch's batch groups (CTAs past groups x C are spare)
  // dR beside the backward scan (grid mode, optional, dr_beside.cuh): chunk
  // c covers the 64-step tiles [tt_lo[c], tt_lo[c] + tt_n[c]) in the scan's
  // order (from t = T-1 down; the last chunk holds t = 0 and the
  // initial-state k-tiles), its fp32 partial of dR at slots + c G N D D
  struct {
    int nc = 0;  // chunks; 0 = off
    int tt_lo[8] = {}, tt_n[8] = {};
    int s0_tiles = 0;
    float* slots = nullptr;
    unsigned int* next = nullptr;  // the unit counter, zeroed before launch
  } drw;
  // optional phase trace (rnn_trace): CTA 0, thread 0 writes clock64() at 8
  // phase points of steps [trace_t0, trace_t0 + trace_steps) (processing order)
  unsigned long long* trace = nullptr;
  int trace_t0 = 0, trace_steps = 0;
  // fault injection (rnn_debug_inject_wait): at this step (processing order)
  // CTA 0 also waits on a barrier that nothing signals, for inject_limit_ns;
  // -1 = off
  int inject_step = -1;
  unsigned long long inject_limit_ns = 0;
};

// Arguments of the alternating path (one launch per step, replayed as a graph).
struct AltArgs {
  int B, T, N, D;
  const void* Wx;
  const void* R;
  const void* bias;
  const void* s0;
  void* states;  // may be null
  void* last;    // may be null
  float* tape;   // fwd: may be null; bwd: in
  const void* dstates;
  const void* dlast;
  void* dWx;
  void* dr;
  void* ds0;
  void* xbuf;  // fwd: h ping-pong [2][B][N][D]; bwd: dr ping-pong [2][B][G][N][D] (bf16)
  float* cst;  // fwd: carried states; bwd: carried state gradients [S][B][N][D] (fp32)
};
cudaError_t alt_fwd_run(int fn, const AltArgs& a, cudaStream_t st);
cudaError_t alt_bwd_run(int fn, const AltArgs& a, cudaStream_t st);

struct FusedShape;
// Clusters of kernel `func` (the cluster kernel of shape `sh`) the current
// device holds at once: sets the kernel's shared-memory and cluster-size
// attributes and asks cudaOccupancyMaxActiveClusters. -1 when the device
// cannot be asked (no device, or the query failed).
int cluster_capacity_of(const void* func, const FusedShape& sh);
// The same for the cluster kernels of one cell (the planner's callback).
int fused_capacity(int fn, bool bwd, const FusedShape& sh);
// SM count of the current device; the GB300's 152 when no device can be asked.
int device_sms();
cudaError_t fused_fwd_run(int fn, const FusedShape& sh, const FusedArgs& a, cudaStream_t st);
cudaError_t grid_fwd_run(int fn, const FusedShape& sh, const FusedArgs& a, cudaStream_t st);
struct UmmaMaps;
// dmaps: the dR operand maps when a.drw.nc > 0 (see dr_beside.cuh)
cudaError_t grid_bwd_run(int fn, const FusedShape& sh, const FusedArgs& a, cudaStream_t st,
                         const UmmaMaps* dmaps = nullptr);

// Encodes a tiled TMA descriptor for a dense row-major bf16 tensor whose
// dims[0] is innermost; box[] gives the tile. No swizzle, zero fill.
cudaError_t encode_tensor_map_bf16(void* map, const void* base, int rank,
                                   const unsigned long long* dims, const unsigned int* box);
cudaError_t encode_tensor_map(void* map, const void* base, int elem_bytes, int rank,
                              const unsigned long long* dims, const unsigned int* box);
// the same with the shared-memory side swizzled in spans of swizzle_bytes
// (0, 32, 64 or 128)
cudaError_t encode_tensor_map_swizzled(void* map, const void* base, int elem_bytes, int rank,
                                       const unsigned long long* dims, const unsigned int* box, int swizzle_bytes);
// bf16, 128-byte swizzle (box[0] * 2 <= 128): the layout the tcgen05 operands read
cudaError_t encode_tensor_map_sw128(void* map, const void* base, int rank, const unsigned long long* dims,
                                    const unsigned int* box);
// The same with explicit byte strides of dimensions 1 .. rank-1 (any order:
// a dimension may step by less than the one before it), so that one box can
// gather several 64-element slabs of a row into consecutive 8 KB blocks.
cudaError_t encode_tensor_map_sw128_strided(void* map, const void* base, int rank, const unsigned long long* dims,
                                            const unsigned long long* strides, const unsigned int* box);
// dR on the 5th-generation tensor cores (bf16, D % 8 == 0); the caller adds db.
bool wgrad_umma_supported(const WgradArgs& a);
int wgrad_umma_splits(int B, int T, int N, int D, int G);
// splits: asked for on entry; on return the count launched (K-tiles are dealt
// out evenly, which can leave fewer splits), the number of partials to reduce.
cudaError_t wgrad_umma_run(const WgradArgs& a, int& splits, cudaStream_t st);
cudaError_t fused_bwd_run(int fn, const FusedShape& sh, const FusedArgs& a, cudaStream_t st);

}  // namespace rnn
