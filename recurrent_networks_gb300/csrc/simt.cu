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
  float* cur = smem;                       // [S][BS][D]  carried states (thread-owned units)
  float* hop = smem + S * BS * D;          // [2][BS][D]  h as the contraction operand

  for (int j = threadIdx.x; j < D; j += blockDim.x)
    for (int bb = 0; bb < BB; ++bb)
      for (int s = 0; s < S; ++s) {
        float v = s0 ? ldf(s0 + ((size_t)(s * B + b0 + bb) * N + n) * D + j) : 0.0f;
        cur[(s * BS + bb) * D + j] = v;
        if (s == 0) hop[bb * D + j] = v;
      }
  __syncthreads();

  for (int t = 0; t < TT; ++t) {
    const float* hin = hop + (t & 1) * BS * D;
    float* hout = hop + ((t + 1) & 1) * BS * D;
    for (int j = threadIdx.x; j < D; j += blockDim.x) {
      float acc[G][SIMT_BBM];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float bv = ldf(bias + (size_t)(g * N + n) * D + j);
#pragma unroll
        for (int bb = 0; bb < SIMT_BBM; ++bb) acc[g][bb] = bv;
      }
      for (int i = 0; i < D; ++i) {
        float rv[G];
#pragma unroll
        for (int g = 0; g < G; ++g) rv[g] = ldf(R + ((size_t)(g * N + n) * D + i) * D + j);
#pragma unroll
        for (int bb = 0; bb < SIMT_BBM; ++bb) {
          if (bb < BB) {
            float hv = hin[bb * D + i];
#pragma unroll
            for (int g = 0; g < G; ++g) acc[g][bb] = fmaf(hv, rv[g], acc[g][bb]);
          }
        }
      }
#pragma unroll
      for (int bb = 0; bb < SIMT_BBM; ++bb) {
        if (bb < BB) {
          const int b = b0 + bb;
          float x[G], r[G], sp[S], sn[S], pre[P];
#pragma unroll
          for (int g = 0; g < G; ++g) {
            x[g] = ldf(Wx + (((size_t)b * TT + t) * G + g) * N * D + (size_t)n * D + j);
            r[g] = acc[g][bb];
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
      }
    }
    __syncthreads();
  }
  if (last)
    for (int j = threadIdx.x; j < D; j += blockDim.x)
      for (int bb = 0; bb < BB; ++bb)
        for (int s = 0; s < S; ++s)
          stf(last + ((size_t)(s * B + b0 + bb) * N + n) * D + j, cur[(s * BS + bb) * D + j]);
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
  float* dS = smem;                       // [S][BS][D] carried deltas (thread-owned units)
  float* drs = smem + S * BS * D;         // [2][G][BS][D] recurrent-branch grads of the step

  for (int j = threadIdx.x; j < D; j += blockDim.x)
    for (int bb = 0; bb < BB; ++bb)
      for (int s = 0; s < S; ++s) {
        float v = 0.0f;
        if (TT == 0 && dlast) v = ldf(dlast + ((size_t)(s * B + b0 + bb) * N + n) * D + j);
        dS[(s * BS + bb) * D + j] = v;
      }

  for (int t = TT - 1; t >= 0; --t) {
    float* drw = drs + (t & 1) * G * BS * D;
    for (int j = threadIdx.x; j < D; j += blockDim.x) {
#pragma unroll
      for (int bb = 0; bb < SIMT_BBM; ++bb) {
        if (bb < BB) {
          const int b = b0 + bb;
          float pre[P], sp[S], sn[S], dsn[S], dx[G], dr[G], dsp[S];
          const float* tp = a.tape + (((size_t)t * B + b) * N + n) * K * D + j;
#pragma unroll
          for (int k = 0; k < P; ++k) pre[k] = tp[k * D];
#pragma unroll
          for (int s = 0; s < S; ++s) sn[s] = tp[(P + s) * D];
          if (t > 0) {
            const float* tq = a.tape + (((size_t)(t - 1) * B + b) * N + n) * K * D + j;
#pragma unroll
            for (int s = 0; s < S; ++s) sp[s] = tq[(P + s) * D];
          } else {
#pragma unroll
            for (int s = 0; s < S; ++s)
              sp[s] = s0 ? ldf(s0 + ((size_t)(s * B + b) * N + n) * D + j) : 0.0f;
          }
#pragma unroll
          for (int s = 0; s < S; ++s) {
            float d = dS[(s * BS + bb) * D + j];
            if (dstates) d += ldf(dstates + (((size_t)s * B + b) * TT + t) * N * D + (size_t)n * D + j);
            if (dlast && t == TT - 1) d += ldf(dlast + ((size_t)(s * B + b) * N + n) * D + j);
            dsn[s] = d;
          }
          cell_bwd<FN, FAST>(pre, sp, sn, dsn, dx, dr, dsp);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            size_t o = (((size_t)b * TT + t) * G + g) * N * D + (size_t)n * D + j;
            if (dWx) stf(dWx + o, dx[g]);
            stf(dr_out + o, dr[g]);
            drw[(g * BS + bb) * D + j] = roundas((const T*)nullptr, dr[g]);
          }
#pragma unroll
          for (int s = 0; s < S; ++s) dS[(s * BS + bb) * D + j] = dsp[s];
        }
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < D; i += blockDim.x) {
      float acc[SIMT_BBM];
#pragma unroll
      for (int bb = 0; bb < SIMT_BBM; ++bb) acc[bb] = 0.0f;
      for (int g = 0; g < G; ++g) {
        const T* row = R + ((size_t)(g * N + n) * D + i) * D;
        for (int j = 0; j < D; ++j) {
          float rv = ldf(row + j);
#pragma unroll
          for (int bb = 0; bb < SIMT_BBM; ++bb)
            if (bb < BB) acc[bb] = fmaf(drw[(g * BS + bb) * D + j], rv, acc[bb]);
        }
      }
#pragma unroll
      for (int bb = 0; bb < SIMT_BBM; ++bb)
        if (bb < BB) dS[bb * D + i] += acc[bb];
    }
  }
  if (ds0) {
    __syncthreads();
    for (int j = threadIdx.x; j < D; j += blockDim.x)
      for (int bb = 0; bb < BB; ++bb)
        for (int s = 0; s < S; ++s)
          stf(ds0 + ((size_t)(s * B + b0 + bb) * N + n) * D + j, dS[(s * BS + bb) * D + j]);
  }
}

// ---- host launchers ----------------------------------------------------------

static int simt_bb(int fn, int B, int D, bool bwd, size_t* smem_out) {
  const int S = fn_states(fn), G = fn_gates(fn);
  // shared floats per batch row: fwd S*D + 2*D ; bwd S*D + 2*G*D
  size_t per = (bwd ? (size_t)(S + 2 * G) * D : (size_t)(S + 2) * D) * sizeof(float);
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
  dim3 grid(a.N, (a.B + BB - 1) / BB);
  void (*k)(SimtArgs) = bwd ? simt_bwd_kernel<FN, T> : simt_fwd_kernel<FN, T>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int threads = a.D >= 256 ? 256 : ((a.D + 31) / 32) * 32;
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
