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

// Every step runs in phases separated by CTA barriers, each spread over all
// threads:
//   forward   A: rec[g][bb][j] = b[g, j] + sum_i h[bb][i] R[g, n, i, j]   (one (g, bb, j) per thread)
//             B: cell update of (bb, j)                                   (one pair per thread)
//   backward  A: cell derivative of (bb, j) -> dr[g][bb][j]
//             B: part[g][bb][i] = sum_j dr[g][bb][j] R[g, n, i, j]       (one (g, bb, i) per thread)
//             C: dS[0][bb][i] += sum_g part[g][bb][i]   (folded into the next step's phase A)
// R (fp32) sits in shared memory when it fits (transposed for the backward,
// so that consecutive threads read consecutive addresses); otherwise it is
// read through L1 / L2. Each dot product keeps four independent partial sums.

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

template <int FN, typename T>
__global__ void __launch_bounds__(256) simt_fwd_kernel(SimtArgs a) {
  constexpr int G = FnInfo<FN>::G, S = FnInfo<FN>::S, P = FnInfo<FN>::P, K = P + S;
  constexpr bool FAST = sizeof(T) == 2;
  const int n = blockIdx.x, b0 = blockIdx.y * a.BB, D = a.D, N = a.N, B = a.B, TT = a.T;
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
  float* Rs = rec + G * BS * D;            // [G][D][D]   R[g, n] in fp32 when it fits (r_smem)
  if (a.r_smem)
    for (int e = threadIdx.x; e < G * D * D; e += blockDim.x) {
      const int g = e / (D * D), r = e - g * D * D;
      Rs[e] = ldf(R + (size_t)(g * N + n) * D * D + r);
    }
  for (int e = threadIdx.x; e < BB * D; e += blockDim.x) {
    const int bb = e / D, j = e - bb * D;
    for (int s = 0; s < S; ++s) {
      const float v = s0 ? ldf(s0 + ((size_t)(s * B + b0 + bb) * N + n) * D + j) : 0.0f;
      cur[(s * BS + bb) * D + j] = v;
      if (s == 0) hop[bb * D + j] = v;
    }
  }
  __syncthreads();

  // Wx of the thread's first pair is loaded one step ahead (its latency hides
  // behind the next step's dot products)
  float xnext[G];
  const int e0 = threadIdx.x;
  if (e0 < BB * D && TT > 0) {
    const int bb = e0 / D, j = e0 - bb * D;
#pragma unroll
    for (int g = 0; g < G; ++g) xnext[g] = ldf(Wx + (((size_t)(b0 + bb) * TT + 0) * G + g) * N * D + (size_t)n * D + j);
  }

  const Walk3 walk0(threadIdx.x, blockDim.x, BB, D);  // this thread's first index, divided once
  for (int t = 0; t < TT; ++t) {
    const float* hin = hop + (t & 1) * BS * D;
    float* hout = hop + ((t + 1) & 1) * BS * D;
    // phase A: the G * BB * D dot products of the step
    Walk3 wa = walk0;
    for (int e = threadIdx.x; e < G * BB * D; e += blockDim.x, wa.next()) {
      const int g = wa.g, bb = wa.bb, j = wa.j;
      const float* hv = hin + bb * D;
      float p0 = 0.0f, p1 = 0.0f, p2 = 0.0f, p3 = 0.0f;
      int i = 0;
      if (a.r_smem) {
        const float* rc = Rs + (size_t)g * D * D + j;
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
      rec[(g * BS + bb) * D + j] = ldf(bias + (size_t)(g * N + n) * D + j) + ((p0 + p1) + (p2 + p3));
    }
    __syncthreads();
    // phase B: the cell update of every (batch row, unit) pair
    Walk3 wb = walk0;
    for (int e = threadIdx.x; e < BB * D; e += blockDim.x, wb.next()) {
      const int bb = wb.bb, j = wb.j, b = b0 + bb;
      float x[G], r[G], sp[S], sn[S], pre[P];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        x[g] = e == e0 ? xnext[g] : ldf(Wx + (((size_t)b * TT + t) * G + g) * N * D + (size_t)n * D + j);
        r[g] = rec[(g * BS + bb) * D + j];
      }
      if (e == e0 && t + 1 < TT) {
#pragma unroll
        for (int g = 0; g < G; ++g) xnext[g] = ldf(Wx + (((size_t)b * TT + t + 1) * G + g) * N * D + (size_t)n * D + j);
      }
#pragma unroll
      for (int s = 0; s < S; ++s) sp[s] = cur[(s * BS + bb) * D + j];
      cell_fwd<FN, FAST>(x, r, sp, sn, pre);
#pragma unroll
      for (int s = 0; s < S; ++s) {
        cur[(s * BS + bb) * D + j] = sn[s];
        if (states) stf(states + (((size_t)s * B + b) * TT + t) * N * D + (size_t)n * D + j, sn[s]);
      }
      hout[bb * D + j] = roundas((const T*)nullptr, sn[0]);
      if (a.tape) {
        float* tp = a.tape + (((size_t)t * B + b) * N + n) * K * D + j;
#pragma unroll
        for (int k = 0; k < P; ++k) tp[k * D] = pre[k];
#pragma unroll
        for (int s = 0; s < S; ++s) tp[(P + s) * D] = sn[s];
      }
    }
    __syncthreads();
  }
  if (last)
    for (int e = threadIdx.x; e < BB * D; e += blockDim.x) {
      const int bb = e / D, j = e - bb * D;
      for (int s = 0; s < S; ++s)
        stf(last + ((size_t)(s * B + b0 + bb) * N + n) * D + j, cur[(s * BS + bb) * D + j]);
    }
}

template <int FN, typename T>
__global__ void __launch_bounds__(256) simt_bwd_kernel(SimtArgs a) {
  constexpr int G = FnInfo<FN>::G, S = FnInfo<FN>::S, P = FnInfo<FN>::P, K = P + S;
  constexpr bool FAST = sizeof(T) == 2;
  const int n = blockIdx.x, b0 = blockIdx.y * a.BB, D = a.D, N = a.N, B = a.B, TT = a.T;
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
  if (a.r_smem)
    for (int e = threadIdx.x; e < G * D * D; e += blockDim.x) {
      const int g = e / (D * D), r = e - g * D * D, i = r / D, j = r - i * D;
      RTs[((size_t)g * D + j) * D + i] = ldf(R + (size_t)(g * N + n) * D * D + r);
    }
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
  auto fetch = [&](int tt, int bb, int j, float* pre, float* sn, float* sp, float* up) {
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
#pragma unroll
    for (int s = 0; s < S; ++s) {
      float d = 0.0f;
      if (dstates) d += ldf(dstates + (((size_t)s * B + b) * TT + tt) * N * D + (size_t)n * D + j);
      if (dlast && tt == TT - 1) d += ldf(dlast + ((size_t)(s * B + b) * N + n) * D + j);
      up[s] = d;
    }
  };
  const int bb0 = e0 / D, j00 = e0 - bb0 * D;
  if (e0 < BB * D && TT > 0) fetch(TT - 1, bb0, j00, npre, nsn, nsp, nup);

  const Walk3 walk0(threadIdx.x, blockDim.x, BB, D);  // this thread's first index, divided once
  for (int t = TT - 1; t >= 0; --t) {
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
        for (int s = 0; s < S; ++s) { sn[s] = nsn[s]; sp[s] = nsp[s]; up[s] = nup[s]; }
        if (t > 0) fetch(t - 1, bb0, j00, npre, nsn, nsp, nup);
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
        drs[(g * BS + bb) * D + j] = roundas((const T*)nullptr, dr[g]);
      }
#pragma unroll
      for (int s = 0; s < S; ++s) dS[(s * BS + bb) * D + j] = dsp[s];
    }
    __syncthreads();
    // phase B: part[g][bb][i] = sum_j dr[g][bb][j] R[g, n, i, j]
    Walk3 wd = walk0;
    for (int e = threadIdx.x; e < G * BB * D; e += blockDim.x, wd.next()) {
      const int g = wd.g, bb = wd.bb, i = wd.j;
      const float* dv = drs + (g * BS + bb) * D;
      float p0 = 0.0f, p1 = 0.0f, p2 = 0.0f, p3 = 0.0f;
      int j = 0;
      if (a.r_smem) {
        const float* rc = RTs + (size_t)g * D * D + i;
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
    __syncthreads();
  }
  if (ds0)
    for (int e = threadIdx.x; e < BB * D; e += blockDim.x) {
      const int bb = e / D, j = e - bb * D;
      float hsum = 0.0f;
#pragma unroll
      for (int g = 0; g < G; ++g) hsum += part[(g * BS + bb) * D + j];
      for (int s = 0; s < S; ++s)
        stf(ds0 + ((size_t)(s * B + b0 + bb) * N + n) * D + j, dS[(s * BS + bb) * D + j] + (s == 0 ? hsum : 0.0f));
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

template <int FN, typename T>
static cudaError_t launch_simt(const SimtArgs& a0, bool bwd, cudaStream_t st) {
  SimtArgs a = a0;
  size_t smem;
  int BB = simt_bb(FN, a.B, a.D, bwd, &smem);
  if (BB <= 0) return cudaErrorInvalidValue;
  a.BB = BB;
  // the head's R in shared memory (fp32) when it fits beside the state buffers
  const size_t rbytes = (size_t)FnInfo<FN>::G * a.D * a.D * sizeof(float);
  a.r_smem = smem + rbytes <= 200 * 1024 ? 1 : 0;
  if (a.r_smem) smem += rbytes;
  dim3 grid(a.N, (a.B + BB - 1) / BB);
  void (*k)(SimtArgs) = bwd ? simt_bwd_kernel<FN, T> : simt_fwd_kernel<FN, T>;
  cudaError_t e = set_smem_attr((const void*)k, (size_t)smem);
  if (e != cudaSuccess) return e;
  // one (gate, row, unit) dot product per thread in the wide phase
  const int work = FnInfo<FN>::G * BB * a.D;
  int threads = work >= 256 ? 256 : ((work + 31) / 32) * 32;
  k<<<grid, threads, smem, st>>>(a);
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
