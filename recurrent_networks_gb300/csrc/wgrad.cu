// Weight gradients of the recurrent branch, after the reverse scan:
//   dR[g,n,i,j] = sum_{b,t} h_{t-1}[b,n,i] * dr[b,t,g,n,j]     (one dense GEMM per (g,n),
//                                                              M = N = D, K = B*T)
//   db[g,n,j]   = sum_{b,t} dr[b,t,g,n,j]
// dr is the gradient of the recurrent branch rec_g = h.R_g + b_g of each step
// (equal to dWx except for the GRU candidate gate, where it carries the reset
// gate factor). h_{t-1} is read from the forward's states (t > 0) or from the
// initial states (t = 0). The plain fp32-FMA tiled version serves fp32
// storage; bf16 storage goes through the tensor-core version further down.
#include "colsum.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

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

// db: block = 32 units x 32 k-slices (strided rows, several loads in flight
// per thread), reduced through shared memory in a fixed order.
constexpr int BG_KS = 32;
template <typename T>
__global__ void __launch_bounds__(32 * BG_KS) bgrad_kernel(WgradArgs a) {
  __shared__ float part[BG_KS][33];
  const int lane = threadIdx.x % 32, ks = threadIdx.x / 32;
  const int j = blockIdx.x * 32 + lane;
  const int gn = blockIdx.y, g = gn / a.N, n = gn - g * a.N;
  const int K = a.B * a.T, D = a.D;
  const T* dr = (const T*)a.dr;
  float s0 = 0.0f, s1 = 0.0f;
  if (j < D) {
    const size_t stride = (size_t)a.G * a.N * D;
    const T* p = dr + (size_t)g * a.N * D + (size_t)n * D + j;
    int k = ks;
    for (; k + BG_KS < K; k += 2 * BG_KS) {
      s0 += ldf(p + (size_t)k * stride);
      s1 += ldf(p + (size_t)(k + BG_KS) * stride);
    }
    if (k < K) s0 += ldf(p + (size_t)k * stride);
  }
  part[ks][lane] = s0 + s1;
  __syncthreads();
  if (ks == 0 && j < D) {
    float tot = 0.0f;
#pragma unroll 8
    for (int q = 0; q < BG_KS; ++q) tot += part[q][lane];
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
    bgrad_kernel<T><<<grid, 32 * BG_KS, 0, st>>>(a);
    note_launch();
  }
  return cudaGetLastError();
}

// ---- tensor-core version (bf16 operands, fp32 accumulation) -------------------
// dR[g,n] (D x D) = Hprev^T (D x K) * dr (K x D), K = B*T, one 128 x 128 output
// tile per CTA (8 warps, 64 x 32 each, mma.sync m16n8k16). Both operands are
// K-major in memory (rows of D contiguous units), so a 32-row k-slab of each is
// copied to shared memory with cp.async and read with ldmatrix.trans. Long K
// is split across CTAs; partial tiles go to fp32 scratch and are summed in a
// fixed order (deterministic).
constexpr int WM_BM = 128, WM_BN = 128, WM_BK = 32, WM_STAGES = 3, WM_LD = WM_BM + 8;

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N_>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N_) : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(256) wgrad_mma_kernel(WgradArgs a, int splits, int kchunk) {
  extern __shared__ __align__(128) unsigned char wm_smem[];
  typedef __nv_bfloat16 Slab[WM_BK][WM_LD];
  Slab* As = (Slab*)wm_smem;                       // [WM_STAGES]
  Slab* Bs = (Slab*)(wm_smem + WM_STAGES * sizeof(Slab));
  const int D = a.D, N = a.N, T = a.T, G = a.G;
  const int j0 = blockIdx.x * WM_BN, i0 = blockIdx.y * WM_BM;
  const int gn = blockIdx.z / splits, split = blockIdx.z - gn * splits;
  const int g = gn / N, n = gn - g * N;
  const int K = a.B * T;
  const int kbeg = split * kchunk, kend = min(K, kbeg + kchunk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 2, wn = warp & 3;  // 2 x 4 warps, 64 x 32 each
  const __nv_bfloat16* states = (const __nv_bfloat16*)a.states;
  const __nv_bfloat16* s0 = (const __nv_bfloat16*)a.s0;
  const __nv_bfloat16* dr = (const __nv_bfloat16*)a.dr;

  auto load_stage = [&](int stage, int k0) {
    // 32 rows x 128 columns of each operand = 512 chunks of 16 bytes each
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int c = tid + r * 256;
      const int row = c >> 4, col = (c & 15) * 8;
      const int k = k0 + row;
      // A: h_{t-1}[b, n, i0 + col ..]
      const __nv_bfloat16* srcA = states;
      int bytesA = 0;
      if (k < kend && i0 + col < D) {
        const int b = k / T, t = k - b * T;
        if (t > 0) {
          srcA = states + (((size_t)b * T + (t - 1)) * N + n) * D + i0 + col;
          bytesA = 16;
        } else if (s0) {
          srcA = s0 + ((size_t)b * N + n) * D + i0 + col;
          bytesA = 16;
        }
      }
      cp_async_16(smem_u32(&As[stage][row][col]), srcA, bytesA);
      const __nv_bfloat16* srcB = dr;
      int bytesB = 0;
      if (k < kend && j0 + col < D) {
        srcB = dr + ((size_t)k * G + g) * N * D + (size_t)n * D + j0 + col;
        bytesB = 16;
      }
      cp_async_16(smem_u32(&Bs[stage][row][col]), srcB, bytesB);
    }
  };

  float acc[4][4][4];
#pragma unroll
  for (int p = 0; p < 4; ++p)
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[p][q][r] = 0.0f;

  const int nk = (kend - kbeg + WM_BK - 1) / WM_BK;
#pragma unroll
  for (int s = 0; s < WM_STAGES - 1; ++s) {
    if (s < nk) load_stage(s, kbeg + s * WM_BK);
    cp_async_commit();
  }
  for (int kt = 0; kt < nk; ++kt) {
    cp_async_wait<WM_STAGES - 2>();
    __syncthreads();
    const int nxt = kt + WM_STAGES - 1;
    if (nxt < nk) load_stage(nxt % WM_STAGES, kbeg + nxt * WM_BK);
    cp_async_commit();
    const int s = kt % WM_STAGES;
#pragma unroll
    for (int kk = 0; kk < WM_BK; kk += 16) {
      uint32_t af[4][4], bfr[4][2];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int m0 = wm * 64 + p * 16;
        const int kr = kk + (lane & 7) + ((lane >> 4) << 3);
        const int mc = m0 + ((lane >> 3) & 1) * 8;
        ldsm_x4_trans(smem_u32(&As[s][kr][mc]), af[p][0], af[p][1], af[p][2], af[p][3]);
      }
#pragma unroll
      for (int q = 0; q < 4; q += 2) {
        const int n0 = wn * 32 + q * 8;
        const int kr = kk + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int nc = n0 + (lane >> 4) * 8;
        ldsm_x4_trans(smem_u32(&Bs[s][kr][nc]), bfr[q][0], bfr[q][1], bfr[q + 1][0], bfr[q + 1][1]);
      }
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q)
          mma16816(acc[p][q], af[p][0], af[p][1], af[p][2], af[p][3], bfr[q][0], bfr[q][1]);
    }
  }
  cp_async_wait<0>();

  // epilogue: fragment (row = lane/4 (+8), col = 2 (lane%4) (+1))
  const int r4 = lane >> 2, c2 = 2 * (lane & 3);
#pragma unroll
  for (int p = 0; p < 4; ++p)
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = i0 + wm * 64 + p * 16 + r4 + h * 8;
        const int j = j0 + wn * 32 + q * 8 + c2;
        if (i >= D || j >= D) continue;
        const float v0 = acc[p][q][2 * h], v1 = acc[p][q][2 * h + 1];
        if (splits == 1) {
          __nv_bfloat16* out = (__nv_bfloat16*)a.dR + (((size_t)g * N + n) * D + i) * D + j;
          *(__nv_bfloat162*)out = __floats2bfloat162_rn(v0, v1);
        } else {
          float* out = a.scratch + ((((size_t)split * G + g) * N + n) * D + i) * D + j;
          *(float2*)out = make_float2(v0, v1);
        }
      }
}

// Sums the split-K partials in order and rounds to bf16.
__global__ void wgrad_reduce_kernel(WgradArgs a, int splits) {
  const size_t total = (size_t)a.G * a.N * a.D * a.D;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t first = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (total % 4 == 0) {  // four elements per thread: 16-byte loads of every partial, all in flight
    const size_t quads = total / 4;
    const float4* p = (const float4*)a.scratch;
    for (size_t e = first; e < quads; e += stride) {
      float4 s = p[e];
      for (int k = 1; k < splits; ++k) {
        const float4 v = p[(size_t)k * quads + e];
        s.x += v.x;
        s.y += v.y;
        s.z += v.z;
        s.w += v.w;
      }
      uint2 o;
      o.x = pack_bf16(__float2bfloat16_rn(s.x), __float2bfloat16_rn(s.y));
      o.y = pack_bf16(__float2bfloat16_rn(s.z), __float2bfloat16_rn(s.w));
      ((uint2*)a.dR)[e] = o;
    }
    return;
  }
  for (size_t e = first; e < total; e += stride) {
    float s = 0.0f;
    for (int k = 0; k < splits; ++k) s += a.scratch[(size_t)k * total + e];
    ((__nv_bfloat16*)a.dR)[e] = __float2bfloat16_rn(s);
  }
}

static int wgrad_splits(int B, int T, int N, int D, int G) {
  const int tiles = ((D + WM_BN - 1) / WM_BN) * ((D + WM_BM - 1) / WM_BM) * G * N;
  const int K = B * T;
  int splits = (2 * device_sms() + tiles - 1) / tiles;  // aim at two CTAs per SM
  const int max_by_k = (K + 255) / 256;           // keep >= 256 rows of K per split
  if (splits > max_by_k) splits = max_by_k;
  if (splits > 32) splits = 32;
  return splits < 1 ? 1 : splits;
}

size_t wgrad_scratch_bytes(int B, int T, int N, int D, int G, int dtype) {
  if (dtype != 1 || D % 8) return 0;
  int s = wgrad_splits(B, T, N, D, G);
  const int su = wgrad_umma_splits(B, T, N, D, G);
  if (su > s) s = su;
  const size_t dR_part = s > 1 ? (size_t)s * G * N * D * D * sizeof(float) : 0;
  // the db partials reuse the region after the dR partials have been reduced
  const size_t db_part = colsum_scratch_bytes(B * T, G * N * D);
  return dR_part > db_part ? dR_part : db_part;
}

// db from the backward scan kernel's per-batch-block sums, added in block order.
__global__ void db_blocks_kernel(const float* __restrict__ dbp, int blocks, int cols, __nv_bfloat16* __restrict__ db) {
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < cols; c += gridDim.x * blockDim.x) {
    float v = 0.0f;
    for (int k = 0; k < blocks; ++k) v += dbp[(size_t)k * cols + c];
    db[c] = __float2bfloat16_rn(v);
  }
}

// db after the tensor-core dR: the sum of the scan kernel's block partials
// when it left them, else the column sums of dr (two passes when the scratch
// and alignment allow, else one block per 32 columns).
static cudaError_t bgrad_launch(const WgradArgs& a, cudaStream_t st) {
  if (!a.db) return cudaSuccess;
  if (a.dbp && a.dbp_blocks > 0) {
    const int cols = a.G * a.N * a.D;
    db_blocks_kernel<<<(cols + 255) / 256, 256, 0, st>>>(a.dbp, a.dbp_blocks, cols, (__nv_bfloat16*)a.db);
    note_launch();
    return cudaGetLastError();
  }
  const int K = a.B * a.T, Cn = a.G * a.N * a.D;
  if (colsum_bf16((const __nv_bfloat16*)a.dr, (__nv_bfloat16*)a.db, K, Cn, a.scratch, a.scratch_bytes, st)) {
    // dr is [K rows][G N D columns]; db[g, n, j] is column (g, n, j)
  } else {
    dim3 g2((a.D + 31) / 32, a.G * a.N);
    bgrad_kernel<__nv_bfloat16><<<g2, 32 * BG_KS, 0, st>>>(a);
    note_launch();
  }
  return cudaGetLastError();
}

cudaError_t wgrad_sum_partials(const WgradArgs& a, int parts, cudaStream_t st) {
  if (a.dR) {
    wgrad_reduce_kernel<<<2 * device_sms(), 256, 0, st>>>(a, parts);
    note_launch();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return bgrad_launch(a, st);
}

cudaError_t wgrad_run(int dtype, const WgradArgs& a, cudaStream_t st) {
  if (dtype != 1 || a.D % 8 || !a.dR) return dtype == 1 ? wgrad_launch<__nv_bfloat16>(a, st) : wgrad_launch<float>(a, st);
  if (wgrad_umma_supported(a)) {  // tcgen05 GEMM, accumulator in tensor memory
    int su = wgrad_umma_splits(a.B, a.T, a.N, a.D, a.G);
    const size_t need = (size_t)su * a.G * a.N * a.D * a.D * sizeof(float);
    if (su > 1 && (!a.scratch || a.scratch_bytes < need)) su = 1;
    const cudaError_t e = wgrad_umma_run(a, su, st);
    if (e == cudaSuccess) {
      if (su > 1) {
        wgrad_reduce_kernel<<<2 * device_sms(), 256, 0, st>>>(a, su);
        note_launch();
      }
      return bgrad_launch(a, st);
    }
    if (e != cudaErrorInvalidValue && e != cudaErrorNotSupported) return e;
    (void)cudaGetLastError();  // the operands do not fit the TMA boxes: the mma.sync GEMM below
  }
  int splits = wgrad_splits(a.B, a.T, a.N, a.D, a.G);
  const size_t need = (size_t)splits * a.G * a.N * a.D * a.D * sizeof(float);
  if (splits > 1 && (!a.scratch || a.scratch_bytes < need)) splits = 1;
  const int K = a.B * a.T;
  int kchunk = (K + splits - 1) / splits;
  kchunk = (kchunk + WM_BK - 1) / WM_BK * WM_BK;
  splits = (K + kchunk - 1) / kchunk;
  if (splits < 1) splits = 1;
  dim3 grid((a.D + WM_BN - 1) / WM_BN, (a.D + WM_BM - 1) / WM_BM, a.G * a.N * splits);
  const int smem = 2 * WM_STAGES * WM_BK * WM_LD * (int)sizeof(__nv_bfloat16);
  cudaError_t e = set_smem_attr((const void*)wgrad_mma_kernel, (size_t)smem);
  if (e != cudaSuccess) return e;
  wgrad_mma_kernel<<<grid, 256, smem, st>>>(a, splits, kchunk);
  note_launch();
  if (splits > 1) {
    wgrad_reduce_kernel<<<2 * device_sms(), 256, 0, st>>>(a, splits);
    note_launch();
  }
  return bgrad_launch(a, st);
}

}  // namespace rnn
