// Plain per-head kernels of the head-wise recurrent scan (any size, fp32 or
// bf16 storage, fp32 arithmetic). One CTA runs one head n over a group of BB
// batch rows for the whole sequence; each thread owns a fixed set of units j
// and keeps their carried states in shared memory. R is read through L2 every
// step. This is the fp32 path and the universal fallback; the fused cluster
// kernels are the fast path for bf16.
//
// Forward per step (FlashRNN announcement, usage example; developnotes 5.3):
//   rec_g[j] = sum_i h[i] R[g,n,i,j] + b[g,n,j]; cell update.
// Backward per step: cell derivative, then dh_{t-1}[i] = sum_{g,j} dr_g[j] R[g,n,i,j].
#include "kernels.cuh"

namespace rnn {

constexpr int SIMT_BBM = 8;  // max batch rows per CTA
constexpr int SIMT_PD = 4;   // steps ahead the per-step inputs of a thread's first pair are loaded

// Every step runs in phases separated by CTA barriers, each spread over all
// threads:
//   forward   A: rec[g][bb][j] = b[g, j] + sum_i h[bb][i] R[g, n, i, j]   (one (g, bb, j) per thread)
//             B: cell update of (bb, j)                                   (one pair per thread)
//   backward  A: cell derivative of (bb, j) -> dr[g][bb][j]
//             B: part[g][bb][i] = sum_j dr[g][bb][j] R[g, n, i, j]       (one (g, bb, i) per thread)
//             C: dS[0][bb][i] += sum_g part[g][bb][i]   (folded into the next step's phase A)
// R (fp32) sits in shared memory when it fits (transposed for the backward,
// so that consecutive threads read consecutive addresses); otherwise it is
// read through L1 / L2. Each dot product keeps four independent partial sums;
// head sizes 32 and 64 get kernels with D fixed at compile time, whose dot
// products unroll completely. σ and tanh come from ex2 / rcp (relative error
// about 3e-7) in fp32 as in bf16 storage.
// When one CTA holds every batch row of its head and the problem is small, the
// backward also computes dR and db for its head at the end (the recurrent-branch
// gradients and h_{t-1} of every step are kept in shared memory for it), so a
// small backward is one launch.

// Coordinates (g, bb, j) of a flat index e = (g * BB + bb) * D + j walked with
// a fixed stride: the stride is split into the same digits once, and each step
// adds digit by digit with carries, so no division runs inside the time loop.
struct Walk3 {
  int g, bb, j;          // the current coordinates
  int dg, dbb, dj;       // the stride's digits
  int BB, D;
  __device__ __forceinline__ Walk3(int e0, int stride, int BB_, int D_) : BB(BB_), D(D_) {
    g = e0 / (BB * D);
    bb = (e0 - g * BB * D) / D;
    j = e0 - (g * BB + bb) * D;
    dg = stride / (BB * D);
    dbb = (stride - dg * BB * D) / D;
    dj = stride - (dg * BB + dbb) * D;
  }
  __device__ __forceinline__ void next() {
    j += dj;
    if (j >= D) {
      j -= D;
      ++bb;
    }
    bb += dbb;
    if (bb >= BB) {
      bb -= BB;
      ++g;
    }
    g += dg;
  }
};

// Loads count elements src(e) into dst[e] (e < count) with up to eight loads
// in flight per thread before their stores.
template <typename F>
__device__ __forceinline__ void stage_batched(int count, F&& load_store) {
  for (int e0 = threadIdx.x; e0 < count; e0 += 8 * blockDim.x) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int e = e0 + k * blockDim.x;
      v[k] = e < count ? load_store(e, 0.0f, false) : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int e = e0 + k * blockDim.x;
      if (e < count) load_store(e, v[k], true);
    }
  }
}

template <int FN, typename T, int DS>
__global__ void __launch_bounds__(256) simt_fwd_kernel(SimtArgs a) {
  constexpr int G = FnInfo<FN>::G, S = FnInfo<FN>::S, P = FnInfo<FN>::P, K = P + S;
  constexpr bool FAST = true;
  const int n = blockIdx.x, b0 = blockIdx.y * a.BB, D = DS ? DS : a.D, N = a.N, B = a.B, TT = a.T;
  const int BS = a.BB, BB = min(a.BB, B - b0);
  const T* Wx = (const T*)a.Wx;
  const T* R = (const T*)a.R;
  const T* bias = (const T*)a.bias;
  const T* s0 = (const T*)a.s0;
  T* states = (T*)a.states;
  T* last = (T*)a.last;
  extern __shared__ float smem[];
  float* cur = smem;                       // [S][BS][D]  carried states
  float* hop = cur + S * BS * D;           // [2][BS][D]  h as the contraction operand
  float* rec = hop + 2 * BS * D;           // [G][BS][D]  recurrent branch of the step
  float* bsm = rec + G * BS * D;           // [G][D]      bias of the head
  float* Rs = bsm + G * D;                 // [G][D][D]   R[g, n] in fp32 when it fits (r_smem)
  if (a.r_smem)
    stage_batched(G * D * D, [&](int e, float v, bool st) {
      const int g = e / (D * D), r = e - g * D * D;
      if (st) Rs[e] = v;
      return st ? v : ldf(R + (size_t)(g * N + n) * D * D + r);
    });
  stage_batched(G * D, [&](int e, float v, bool st) {
    const int g = e / D, j = e - g * D;
    if (st) bsm[e] = v;
    return st ? v : ldf(bias + (size_t)(g * N + n) * D + j);
  });
  for (int e = threadIdx.x; e < BB * D; e += blockDim.x) {
    const int bb = e / D, j = e - bb * D;
    for (int s = 0; s < S; ++s) {
      const float v = s0 ? ldf(s0 + ((size_t)(s * B + b0 + bb) * N + n) * D + j) : 0.0f;
      cur[(s * BS + bb) * D + j] = v;
      if (s == 0) hop[bb * D + j] = v;
    }
  }
  __syncthreads();

  // Wx of the thread's first pair is loaded SIMT_PD steps ahead, so that a load
  // from HBM (about a microsecond) lands before its step's cell update
  float xq[SIMT_PD][G];
  const int e0 = threadIdx.x;
  const bool has0 = e0 < BB * D;
  const int bbq = e0 / D, jq = e0 - bbq * D;
  const T* wxq = Wx + ((size_t)(b0 + bbq) * TT * G) * N * D + (size_t)n * D + jq;  // step 0, gate 0
#pragma unroll
  for (int k = 0; k < SIMT_PD; ++k)
#pragma unroll
    for (int g = 0; g < G; ++g) xq[k][g] = (has0 && k < TT) ? ldf(wxq + ((size_t)k * G + g) * N * D) : 0.0f;

  const Walk3 walk0(threadIdx.x, blockDim.x, BB, D);  // this thread's first index, divided once
  // With D fixed at compile time and one dot product per thread, the thread's
  // column R[g, n, :, j] stays in registers for the whole sequence.
  constexpr int DR = DS > 0 ? DS : 1;
  const bool r_regs = DS > 0 && G * BB * D <= (int)blockDim.x;
  float rreg[DR];
  if (r_regs && threadIdx.x < G * BB * D) {
#pragma unroll
    for (int i = 0; i < DR; ++i) rreg[i] = ldf(R + ((size_t)(walk0.g * N + n) * D + i) * D + walk0.j);
  }
  // the output addresses of the thread's first pair, advanced by a fixed stride per step
  T* st_ptr = states ? states + ((size_t)(b0 + walk0.bb) * TT) * N * D + (size_t)n * D + walk0.j : nullptr;
  const size_t st_sstride = (size_t)B * TT * N * D;
  float* tp_ptr = a.tape ? a.tape + ((size_t)(b0 + walk0.bb) * N + n) * K * D + walk0.j : nullptr;
  const size_t tp_tstride = (size_t)B * N * K * D;
  const bool tracer = a.trace && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0;
#define RNN_TRACE(k)                                                               \
  if (tracer && t >= a.trace_t0 && t < a.trace_t0 + a.trace_steps)                 \
    a.trace[(size_t)(t - a.trace_t0) * 16 + (k)] = (unsigned long long)clock64();
  for (int t = 0; t < TT; ++t) {
    RNN_TRACE(0)
    const float* hin = hop + (t & 1) * BS * D;
    float* hout = hop + ((t + 1) & 1) * BS * D;
    // phase A: the G * BB * D dot products of the step
    Walk3 wa = walk0;
    for (int e = threadIdx.x; e < G * BB * D; e += blockDim.x, wa.next()) {
      const int g = wa.g, bb = wa.bb, j = wa.j;
      const float* hv = hin + bb * D;
      float p0 = 0.0f, p1 = 0.0f, p2 = 0.0f, p3 = 0.0f;
      int i = 0;
      if (r_regs) {
#pragma unroll
        for (int i4 = 0; i4 < DR; i4 += 4) {
          const float4 h4 = *(const float4*)(hv + i4);
          p0 = fmaf(h4.x, rreg[i4], p0);
          p1 = fmaf(h4.y, rreg[i4 + 1], p1);
          p2 = fmaf(h4.z, rreg[i4 + 2], p2);
          p3 = fmaf(h4.w, rreg[i4 + 3], p3);
        }
      } else if (a.r_smem) {
        const float* rc = Rs + (size_t)g * D * D + j;
#pragma unroll
        for (; i + 4 <= D; i += 4) {
          p0 = fmaf(hv[i], rc[(size_t)i * D], p0);
          p1 = fmaf(hv[i + 1], rc[(size_t)(i + 1) * D], p1);
          p2 = fmaf(hv[i + 2], rc[(size_t)(i + 2) * D], p2);
          p3 = fmaf(hv[i + 3], rc[(size_t)(i + 3) * D], p3);
        }
        for (; i < D; ++i) p0 = fmaf(hv[i], rc[(size_t)i * D], p0);
      } else {
        const T* rc = R + (size_t)(g * N + n) * D * D + j;
        for (; i + 4 <= D; i += 4) {
          p0 = fmaf(hv[i], ldf(rc + (size_t)i * D), p0);
          p1 = fmaf(hv[i + 1], ldf(rc + (size_t)(i + 1) * D), p1);
          p2 = fmaf(hv[i + 2], ldf(rc + (size_t)(i + 2) * D), p2);
          p3 = fmaf(hv[i + 3], ldf(rc + (size_t)(i + 3) * D), p3);
        }
        for (; i < D; ++i) p0 = fmaf(hv[i], ldf(rc + (size_t)i * D), p0);
      }
      rec[(g * BS + bb) * D + j] = bsm[g * D + j] + ((p0 + p1) + (p2 + p3));
    }
    RNN_TRACE(1)
    __syncthreads();
    RNN_TRACE(2)
    // phase B: the cell update of every (batch row, unit) pair
    Walk3 wb = walk0;
    for (int e = threadIdx.x; e < BB * D; e += blockDim.x, wb.next()) {
      const int bb = wb.bb, j = wb.j, b = b0 + bb;
      float x[G], r[G], sp[S], sn[S], pre[P];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        x[g] = e == e0 ? xq[0][g] : ldf(Wx + (((size_t)b * TT + t) * G + g) * N * D + (size_t)n * D + j);
        r[g] = rec[(g * BS + bb) * D + j];
      }
      if (e == e0) {  // shift the ring and load step t + SIMT_PD
#pragma unroll
        for (int k = 0; k + 1 < SIMT_PD; ++k)
#pragma unroll
          for (int g = 0; g < G; ++g) xq[k][g] = xq[k + 1][g];
        const int tn = t + SIMT_PD;
#pragma unroll
        for (int g = 0; g < G; ++g) xq[SIMT_PD - 1][g] = tn < TT ? ldf(wxq + ((size_t)tn * G + g) * N * D) : 0.0f;
      }
#pragma unroll
      for (int s = 0; s < S; ++s) sp[s] = cur[(s * BS + bb) * D + j];
      if (e == e0) RNN_TRACE(5)
      cell_fwd<FN, FAST>(x, r, sp, sn, pre);
      if (e == e0) RNN_TRACE(6)
      hout[bb * D + j] = roundas((const T*)nullptr, sn[0]);
#pragma unroll
      for (int s = 0; s < S; ++s) cur[(s * BS + bb) * D + j] = sn[s];
      T* stp = e == e0 ? st_ptr : (states ? states + (((size_t)b * TT + t) * N * D + (size_t)n * D + j) : nullptr);
      float* tp = e == e0 ? tp_ptr : (a.tape ? a.tape + (((size_t)t * B + b) * N + n) * K * D + j : nullptr);
      if (stp) {
#pragma unroll
        for (int s = 0; s < S; ++s) stf(stp + (size_t)s * st_sstride, sn[s]);
      }
      if (tp) {
#pragma unroll
        for (int k = 0; k < P; ++k) tp[k * D] = pre[k];
#pragma unroll
        for (int s = 0; s < S; ++s) tp[(P + s) * D] = sn[s];
      }
    }
    if (st_ptr) st_ptr += (size_t)N * D;
    if (tp_ptr) tp_ptr += tp_tstride;
    RNN_TRACE(3)
    __syncthreads();
    RNN_TRACE(4)
  }
#undef RNN_TRACE
  if (last)
    for (int e = threadIdx.x; e < BB * D; e += blockDim.x) {
      const int bb = e / D, j = e - bb * D;
      for (int s = 0; s < S; ++s)
        stf(last + ((size_t)(s * B + b0 + bb) * N + n) * D + j, cur[(s * BS + bb) * D + j]);
    }
}

template <int FN, typename T, int DS>
__global__ void __launch_bounds__(256) simt_bwd_kernel(SimtArgs a) {
  constexpr int G = FnInfo<FN>::G, S = FnInfo<FN>::S, P = FnInfo<FN>::P, K = P + S;
  constexpr bool FAST = true;
  const int n = blockIdx.x, b0 = blockIdx.y * a.BB, D = DS ? DS : a.D, N = a.N, B = a.B, TT = a.T;
  const int BS = a.BB, BB = min(a.BB, B - b0);
  const T* R = (const T*)a.R;
  const T* s0 = (const T*)a.s0;
  const T* dstates = (const T*)a.dstates;
  const T* dlast = (const T*)a.dlast;
  T* dWx = (T*)a.dWx;
  T* dr_out = (T*)a.dr;
  T* ds0 = (T*)a.ds0;
  extern __shared__ float smem[];
  float* dS = smem;                        // [S][BS][D]  carried deltas
  float* drs = dS + S * BS * D;            // [G][BS][D]  recurrent-branch grads of the step (operand)
  float* part = drs + G * BS * D;          // [G][BS][D]  per-gate partial dh_{t-1}
  float* RTs = part + G * BS * D;          // [G][D j][D i] R[g, n]^T in fp32 when it fits (r_smem)
  // fused weight gradients: dr [T][BS][G][D] and h_{t-1} [T][BS][D] of every step
  float* wdr = RTs + (a.r_smem ? G * D * D : 0);
  float* whp = wdr + (a.fuse_wgrad ? (size_t)TT * BS * G * D : 0);
  if (a.r_smem)
    stage_batched(G * D * D, [&](int e, float v, bool st) {
      const int g = e / (D * D), r = e - g * D * D, i = r / D, j = r - i * D;
      if (st) RTs[((size_t)g * D + j) * D + i] = v;
      return st ? v : ldf(R + (size_t)(g * N + n) * D * D + r);
    });
  for (int e = threadIdx.x; e < BB * D; e += blockDim.x) {
    const int bb = e / D, j = e - bb * D;
    for (int s = 0; s < S; ++s) {
      float v = 0.0f;
      if (TT == 0 && dlast) v = ldf(dlast + ((size_t)(s * B + b0 + bb) * N + n) * D + j);
      dS[(s * BS + bb) * D + j] = v;
    }
    for (int g = 0; g < G; ++g) part[(g * BS + bb) * D + j] = 0.0f;
  }
  __syncthreads();

  // the step's tape record, previous states and upstream gradients of the
  // thread's first pair are loaded one step ahead
  const int e0 = threadIdx.x;
  float npre[P], nsn[S], nsp[S], nup[S];
  auto fetch = [&](int tt, int bb, int j, float* pre, float* sn, float* sp, float* up, bool with_up = true) {
    const int b = b0 + bb;
    const float* tp = a.tape + (((size_t)tt * B + b) * N + n) * K * D + j;
#pragma unroll
    for (int k = 0; k < P; ++k) pre[k] = tp[k * D];
#pragma unroll
    for (int s = 0; s < S; ++s) sn[s] = tp[(P + s) * D];
    if (tt > 0) {
      const float* tq = a.tape + (((size_t)(tt - 1) * B + b) * N + n) * K * D + j;
#pragma unroll
      for (int s = 0; s < S; ++s) sp[s] = tq[(P + s) * D];
    } else {
#pragma unroll
      for (int s = 0; s < S; ++s) sp[s] = s0 ? ldf(s0 + ((size_t)(s * B + b) * N + n) * D + j) : 0.0f;
    }
    if (with_up) {
#pragma unroll
      for (int s = 0; s < S; ++s) {
        float d = 0.0f;
        if (dstates) d += ldf(dstates + (((size_t)s * B + b) * TT + tt) * N * D + (size_t)n * D + j);
        if (dlast && tt == TT - 1) d += ldf(dlast + ((size_t)(s * B + b) * N + n) * D + j);
        up[s] = d;
      }
    }
  };
  const int bb0 = e0 / D, j00 = e0 - bb0 * D;
  if (e0 < BB * D && TT > 0) fetch(TT - 1, bb0, j00, npre, nsn, nsp, nup, false);
  // the upstream gradients dstates[:, b, t] of the first pair come from HBM:
  // loaded SIMT_PD steps ahead (processing order t = T-1 .. 0)
  float uq[SIMT_PD][S];
  const bool has0 = e0 < BB * D;
  auto upstream = [&](int tt, int s) {
    return (dstates && has0 && tt >= 0) ? ldf(dstates + (((size_t)s * B + b0 + bb0) * TT + tt) * N * D + (size_t)n * D + j00)
                                        : 0.0f;
  };
#pragma unroll
  for (int k = 0; k < SIMT_PD; ++k)
#pragma unroll
    for (int s2 = 0; s2 < S; ++s2) uq[k][s2] = upstream(TT - 1 - k, s2);

  const Walk3 walk0(threadIdx.x, blockDim.x, BB, D);  // this thread's first index, divided once
  // With D fixed at compile time and one dot product per thread, the thread's
  // row R[g, n, i, :] stays in registers for the whole sequence.
  constexpr int DR = DS > 0 ? DS : 1;
  const bool r_regs = DS > 0 && G * BB * D <= (int)blockDim.x;
  float rreg[DR];
  if (r_regs && threadIdx.x < G * BB * D) {
#pragma unroll
    for (int j = 0; j < DR; ++j) rreg[j] = ldf(R + ((size_t)(walk0.g * N + n) * D + walk0.j) * D + j);
  }
  const bool tracer = a.trace && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0;
#define RNN_TRACE(k)                                                                   \
  if (tracer && TT - 1 - t >= a.trace_t0 && TT - 1 - t < a.trace_t0 + a.trace_steps)    \
    a.trace[(size_t)(TT - 1 - t - a.trace_t0) * 16 + (k)] = (unsigned long long)clock64();
  for (int t = TT - 1; t >= 0; --t) {
    RNN_TRACE(0)
    // phase A: cell derivative of every pair; dh_t gathers the G partials of
    // the later step first
    Walk3 wc = walk0;
    for (int e = threadIdx.x; e < BB * D; e += blockDim.x, wc.next()) {
      const int bb = wc.bb, j = wc.j, b = b0 + bb;
      float hsum = 0.0f;
#pragma unroll
      for (int g = 0; g < G; ++g) hsum += part[(g * BS + bb) * D + j];
      float pre[P], sp[S], sn[S], up[S], dsn[S], dx[G], dr[G], dsp[S];
      if (e == e0) {
#pragma unroll
        for (int k = 0; k < P; ++k) pre[k] = npre[k];
#pragma unroll
        for (int s = 0; s < S; ++s) {
          sn[s] = nsn[s];
          sp[s] = nsp[s];
          up[s] = uq[0][s] + ((dlast && t == TT - 1) ? ldf(dlast + ((size_t)(s * B + b) * N + n) * D + j) : 0.0f);
        }
#pragma unroll
        for (int k = 0; k + 1 < SIMT_PD; ++k)
#pragma unroll
          for (int s = 0; s < S; ++s) uq[k][s] = uq[k + 1][s];
#pragma unroll
        for (int s = 0; s < S; ++s) uq[SIMT_PD - 1][s] = upstream(t - SIMT_PD, s);
        if (t > 0) fetch(t - 1, bb0, j00, npre, nsn, nsp, nup, false);
      } else {
        fetch(t, bb, j, pre, sn, sp, up);
      }
#pragma unroll
      for (int s = 0; s < S; ++s) {
        float d = dS[(s * BS + bb) * D + j] + up[s];
        if (s == 0) d += hsum;
        dsn[s] = d;
      }
      cell_bwd<FN, FAST>(pre, sp, sn, dsn, dx, dr, dsp);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const size_t o = (((size_t)b * TT + t) * G + g) * N * D + (size_t)n * D + j;
        if (dWx) stf(dWx + o, dx[g]);
        stf(dr_out + o, dr[g]);
        const float drv = roundas((const T*)nullptr, dr[g]);
        drs[(g * BS + bb) * D + j] = drv;
        if (a.fuse_wgrad) wdr[(((size_t)t * BS + bb) * G + g) * D + j] = drv;
      }
      if (a.fuse_wgrad) whp[((size_t)t * BS + bb) * D + j] = roundas((const T*)nullptr, sp[0]);
#pragma unroll
      for (int s = 0; s < S; ++s) dS[(s * BS + bb) * D + j] = dsp[s];
    }
    RNN_TRACE(1)
    __syncthreads();
    RNN_TRACE(2)
    // phase B: part[g][bb][i] = sum_j dr[g][bb][j] R[g, n, i, j]
    Walk3 wd = walk0;
    for (int e = threadIdx.x; e < G * BB * D; e += blockDim.x, wd.next()) {
      const int g = wd.g, bb = wd.bb, i = wd.j;
      const float* dv = drs + (g * BS + bb) * D;
      float p0 = 0.0f, p1 = 0.0f, p2 = 0.0f, p3 = 0.0f;
      int j = 0;
      if (r_regs) {
#pragma unroll
        for (int j4 = 0; j4 < DR; j4 += 4) {
          const float4 d4 = *(const float4*)(dv + j4);
          p0 = fmaf(d4.x, rreg[j4], p0);
          p1 = fmaf(d4.y, rreg[j4 + 1], p1);
          p2 = fmaf(d4.z, rreg[j4 + 2], p2);
          p3 = fmaf(d4.w, rreg[j4 + 3], p3);
        }
      } else if (a.r_smem) {
        const float* rc = RTs + (size_t)g * D * D + i;
  #pragma unroll
        for (; j + 4 <= D; j += 4) {
          p0 = fmaf(dv[j], rc[(size_t)j * D], p0);
          p1 = fmaf(dv[j + 1], rc[(size_t)(j + 1) * D], p1);
          p2 = fmaf(dv[j + 2], rc[(size_t)(j + 2) * D], p2);
          p3 = fmaf(dv[j + 3], rc[(size_t)(j + 3) * D], p3);
        }
        for (; j < D; ++j) p0 = fmaf(dv[j], rc[(size_t)j * D], p0);
      } else {
        const T* row = R + ((size_t)(g * N + n) * D + i) * D;
        for (; j + 4 <= D; j += 4) {
          p0 = fmaf(dv[j], ldf(row + j), p0);
          p1 = fmaf(dv[j + 1], ldf(row + j + 1), p1);
          p2 = fmaf(dv[j + 2], ldf(row + j + 2), p2);
          p3 = fmaf(dv[j + 3], ldf(row + j + 3), p3);
        }
        for (; j < D; ++j) p0 = fmaf(dv[j], ldf(row + j), p0);
      }
      part[(g * BS + bb) * D + i] = (p0 + p1) + (p2 + p3);
    }
    RNN_TRACE(3)
    __syncthreads();
    RNN_TRACE(4)
  }
#undef RNN_TRACE
  if (ds0)
    for (int e = threadIdx.x; e < BB * D; e += blockDim.x) {
      const int bb = e / D, j = e - bb * D;
      float hsum = 0.0f;
#pragma unroll
      for (int g = 0; g < G; ++g) hsum += part[(g * BS + bb) * D + j];
      for (int s = 0; s < S; ++s)
        stf(ds0 + ((size_t)(s * B + b0 + bb) * N + n) * D + j, dS[(s * BS + bb) * D + j] + (s == 0 ? hsum : 0.0f));
    }
  if (a.fuse_wgrad) {
    // dR[g, n, i, j] = sum_{b, t} h_{t-1}[b, i] dr_t[b, g, j], db[g, n, j] = sum_{b, t} dr_t[b, g, j]:
    // this CTA holds every row of head n, so it owns these sums. Each thread
    // takes 4 x 4 (i, j) tiles of one gate: per (step, row) two 16-byte
    // shared loads feed 16 products; the tiles with i0 = 0 also sum db.
    // The order of the sums is fixed (deterministic).
    __syncthreads();
    T* dRo = (T*)a.dR;
    T* dbo = (T*)a.db;
    const int D4 = D / 4;
    for (int e = threadIdx.x; e < G * D4 * D4; e += blockDim.x) {
      const int g = e / (D4 * D4), r = e - g * D4 * D4, i0 = 4 * (r / D4), j0 = 4 * (r - (r / D4) * D4);
      float acc[4][4], dbs[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        dbs[x] = 0.0f;
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = 0.0f;
      }
      for (int t = 0; t < TT; ++t)
        for (int bb = 0; bb < BB; ++bb) {
          const float4 h4 = *(const float4*)(whp + ((size_t)t * BS + bb) * D + i0);
          const float4 d4 = *(const float4*)(wdr + (((size_t)t * BS + bb) * G + g) * D + j0);
          const float hv[4] = {h4.x, h4.y, h4.z, h4.w}, dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            dbs[x] += dv[x];
#pragma unroll
            for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(hv[x], dv[y], acc[x][y]);
          }
        }
      if (dRo)
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y)
            stf(dRo + ((size_t)(g * N + n) * D + i0 + x) * D + j0 + y, acc[x][y]);
      if (dbo && i0 == 0)
#pragma unroll
        for (int y = 0; y < 4; ++y) stf(dbo + (size_t)(g * N + n) * D + j0 + y, dbs[y]);
    }
  }
}

// ---- host launchers ----------------------------------------------------------

static int simt_bb(int fn, int B, int D, bool bwd, size_t* smem_out) {
  const int S = fn_states(fn), G = fn_gates(fn);
  // shared floats per batch row: fwd (S + 2 + G) D ; bwd (S + 2 G) D
  size_t per = (bwd ? (size_t)(S + 2 * G) * D : (size_t)(S + 2 + G) * D) * sizeof(float);
  int bb = B < SIMT_BBM ? B : SIMT_BBM;
  while (bb > 0 && per * bb > 200 * 1024) --bb;
  *smem_out = per * (bb > 0 ? bb : 1);
  return bb;
}

// Shared memory of a plain kernel launch: the state buffers of simt_bb, the
// bias (forward), R when it fits, the fused weight-gradient staging (backward).
struct SimtSmem {
  int BB = 0;
  bool r_smem = false, fuse = false;
  size_t bytes = 0;
};
static SimtSmem simt_smem(int fn, int B, int T, int D, bool bwd, bool want_fuse) {
  SimtSmem m;
  size_t smem;
  m.BB = simt_bb(fn, B, D, bwd, &smem);
  if (m.BB <= 0) return m;
  const int G = fn_gates(fn);
  if (!bwd) smem += (size_t)G * D * sizeof(float);
  const size_t rbytes = (size_t)G * D * D * sizeof(float);
  m.r_smem = smem + rbytes <= 200 * 1024;
  if (m.r_smem) smem += rbytes;
  if (bwd && want_fuse && m.BB >= B && D % 4 == 0 && (double)G * D * D * B * T <= (double)(1 << 21)) {
    const size_t wb = (size_t)T * m.BB * (G + 1) * D * sizeof(float);
    if (smem + wb <= 200 * 1024) {
      m.fuse = true;
      smem += wb;
    }
  }
  m.bytes = smem;
  return m;
}

bool simt_fuses_wgrad(int fn, int B, int T, int D) { return T > 0 && simt_smem(fn, B, T, D, true, true).fuse; }

template <int FN, typename T>
static cudaError_t launch_simt(const SimtArgs& a0, bool bwd, cudaStream_t st) {
  SimtArgs a = a0;
  const SimtSmem m = simt_smem(FN, a.B, a.T, a.D, bwd, a.fuse_wgrad != 0);
  if (m.BB <= 0) return cudaErrorInvalidValue;
  if (a.fuse_wgrad && !m.fuse) return cudaErrorInvalidValue;  // the caller asked simt_fuses_wgrad first
  a.BB = m.BB;
  a.r_smem = m.r_smem ? 1 : 0;
  dim3 grid(a.N, (a.B + m.BB - 1) / m.BB);
  // head sizes 32 and 64 run kernels with D fixed at compile time
  void (*k)(SimtArgs) = nullptr;
  if (a.D == 32) k = bwd ? simt_bwd_kernel<FN, T, 32> : simt_fwd_kernel<FN, T, 32>;
  else if (a.D == 64) k = bwd ? simt_bwd_kernel<FN, T, 64> : simt_fwd_kernel<FN, T, 64>;
  else k = bwd ? simt_bwd_kernel<FN, T, 0> : simt_fwd_kernel<FN, T, 0>;
  cudaError_t e = set_smem_attr((const void*)k, m.bytes);
  if (e != cudaSuccess) return e;
  // one (gate, row, unit) dot product per thread in the wide phase
  const int work = FnInfo<FN>::G * m.BB * a.D;
  int threads = work >= 256 ? 256 : ((work + 31) / 32) * 32;
  k<<<grid, threads, m.bytes, st>>>(a);
  note_launch();
  return cudaGetLastError();
}

int simt_supported(int fn, int B, int D, bool bwd) {
  size_t smem;
  return simt_bb(fn, B, D, bwd, &smem) > 0;
}

cudaError_t simt_run(int fn, int dtype, const SimtArgs& a, bool bwd, cudaStream_t st) {
#define RNN_SIMT_CASE(F)                                                     \
  case F:                                                                    \
    return dtype == 1 ? launch_simt<F, __nv_bfloat16>(a, bwd, st)            \
                      : launch_simt<F, float>(a, bwd, st);
  switch (fn) {
    RNN_SIMT_CASE(LSTM)
    RNN_SIMT_CASE(GRU)
    RNN_SIMT_CASE(ELMAN)
    RNN_SIMT_CASE(SLSTM)
    RNN_SIMT_CASE(SLSTM_LS)
  }
#undef RNN_SIMT_CASE
  return cudaErrorInvalidValue;
}

}  // namespace rnn
