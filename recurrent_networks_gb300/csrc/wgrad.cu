// Weight gradients of the recurrent branch, after the reverse scan:
//   dR[g,n,i,j] = sum_{b,t} h_{t-1}[b,n,i] * dr[b,t,g,n,j]     (one dense GEMM per (g,n),
//                                                              M = N = D, K = B*T)
//   db[g,n,j]   = sum_{b,t} dr[b,t,g,n,j]
// dr is the gradient of the recurrent branch rec_g = h.R_g + b_g of each step
// (equal to dWx except for the GRU candidate gate, where it carries the reset
// gate factor). h_{t-1} is read from the forward's states (t > 0) or from the
// initial states (t = 0). This file holds the plain fp32-FMA tiled version,
// used for fp32 storage; the tensor-core version for bf16 lives in
// wgrad_mma.cu.
#include "kernels.cuh"

namespace rnn {

constexpr int WG_TILE = 64, WG_KC = 32;

template <typename T>
__device__ __forceinline__ float hprev_at(const WgradArgs& a, int k, int n, int i) {
  const int b = k / a.T, t = k - b * a.T;
  if (t > 0) return ldf((const T*)a.states + (((size_t)b * a.T + (t - 1)) * a.N + n) * a.D + i);
  return a.s0 ? ldf((const T*)a.s0 + ((size_t)b * a.N + n) * a.D + i) : 0.0f;
}

template <typename T>
__global__ void __launch_bounds__(256) wgrad_simt_kernel(WgradArgs a) {
  __shared__ float As[WG_KC][WG_TILE];
  __shared__ float Bs[WG_KC][WG_TILE];
  const int j0 = blockIdx.x * WG_TILE, i0 = blockIdx.y * WG_TILE;
  const int gn = blockIdx.z, g = gn / a.N, n = gn - g * a.N;
  const int K = a.B * a.T, D = a.D;
  const int ti = threadIdx.x / 16, tj = threadIdx.x % 16;
  const T* dr = (const T*)a.dr;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += WG_KC) {
    for (int e = threadIdx.x; e < WG_KC * WG_TILE; e += 256) {
      int kk = e / WG_TILE, c = e % WG_TILE, k = k0 + kk;
      float av = 0.0f, bv = 0.0f;
      if (k < K) {
        if (i0 + c < D) av = hprev_at<T>(a, k, n, i0 + c);
        if (j0 + c < D) bv = ldf(dr + ((size_t)k * a.G + g) * a.N * D + (size_t)n * D + j0 + c);
      }
      As[kk][c] = av;
      Bs[kk][c] = bv;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < WG_KC; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        av[q] = As[kk][ti * 4 + q];
        bv[q] = Bs[kk][tj * 4 + q];
      }
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[p][q] = fmaf(av[p], bv[q], acc[p][q]);
    }
    __syncthreads();
  }
  T* dR = (T*)a.dR;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    int i = i0 + ti * 4 + p;
    if (i >= D) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int j = j0 + tj * 4 + q;
      if (j < D) stf(dR + (((size_t)g * a.N + n) * D + i) * D + j, acc[p][q]);
    }
  }
}

// db: block = 32 units x 8 k-slices, reduced through shared memory.
template <typename T>
__global__ void __launch_bounds__(256) bgrad_kernel(WgradArgs a) {
  __shared__ float part[8][33];
  const int lane = threadIdx.x % 32, ks = threadIdx.x / 32;
  const int j = blockIdx.x * 32 + lane;
  const int gn = blockIdx.y, g = gn / a.N, n = gn - g * a.N;
  const int K = a.B * a.T, D = a.D;
  const T* dr = (const T*)a.dr;
  float s = 0.0f;
  if (j < D)
    for (int k = ks; k < K; k += 8) s += ldf(dr + ((size_t)k * a.G + g) * a.N * D + (size_t)n * D + j);
  part[ks][lane] = s;
  __syncthreads();
  if (ks == 0 && j < D) {
    float tot = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) tot += part[q][lane];
    stf((T*)a.db + ((size_t)g * a.N + n) * D + j, tot);
  }
}

template <typename T>
static cudaError_t wgrad_launch(const WgradArgs& a, cudaStream_t st) {
  const int GN = a.G * a.N;
  if (a.dR) {
    dim3 grid((a.D + WG_TILE - 1) / WG_TILE, (a.D + WG_TILE - 1) / WG_TILE, GN);
    wgrad_simt_kernel<T><<<grid, 256, 0, st>>>(a);
    note_launch();
  }
  if (a.db) {
    dim3 grid((a.D + 31) / 32, GN);
    bgrad_kernel<T><<<grid, 256, 0, st>>>(a);
    note_launch();
  }
  return cudaGetLastError();
}

cudaError_t wgrad_run(int dtype, const WgradArgs& a, cudaStream_t st) {
  return dtype == 1 ? wgrad_launch<__nv_bfloat16>(a, st) : wgrad_launch<float>(a, st);
}

}  // namespace rnn
