// Alternating path: one kernel launch per time step, replayed as a CUDA graph.
//
// The FlashRNN announcement names two designs: "fused" (matrix product and
// pointwise cell in one persistent kernel, recurrent weights on chip) and
// "alternating" (a matrix product and a pointwise step per time step, for
// hidden sizes whose weights do not fit on chip). Here the alternating step is
// one kernel that streams its slice of R from L2 / HBM, runs the step's product
// on the tensor cores (mma.sync m16n8k16, bf16 operands, fp32 accumulation) and
// applies the cell in its epilogue: the pointwise work never leaves the CTA that
// produced the pre-activations. The T launches of a sequence are captured once
// into a CUDA graph and replayed, keyed on the call's shapes and pointers.
//
// Forward step t (grid: unit tiles x heads x batch tiles):
//   rec[b, (g, u)] = sum_i h_{t-1}[b, n, i] R[g, n, i, u0 + u]   (K = D, split over warps)
//   cell update of (b, u0 + u) with Wx[b, t], b, and the carried states (fp32,
//   workspace) -> states[:, b, t], tape[t], h_t (bf16 ping-pong buffer).
// Backward step t (grid: unit tiles x heads x batch tiles, reverse order):
//   dh_t[b, i] = sum_{g, j} dr_{t+1}[b, g, n, j] R[g, n, i, j]  (K = G D, split over warps)
//   cell derivative of (b, i) from the tape -> dWx[b, t], dr_t (bf16 ping-pong
//   and, for the weight gradients, the [B,T,G,N,D] buffer), carried gradients.
// A last backward launch (t = -1) turns dr_0 into dstates0.
#include <mutex>
#include <vector>

#include "kernels.cuh"
#include "ptx.cuh"

namespace rnn {

namespace {

constexpr int ALT_BK = 16;    // k per pipeline chunk (one m16n8k16 step)
constexpr int ALT_NSTG = 4;   // cp.async stages per warp

__device__ __forceinline__ void cpa16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N_>
__device__ __forceinline__ void cpa_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N_) : "memory");
}
// Programmatic dependent launch: let the next step's grid start while this one
// runs (it only prefetches R before its own dependency wait), and wait for the
// previous step's grid (complete, memory visible) before touching its outputs.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Columns a CTA owns: the forward takes all G gates of UT units (the cell
// needs them together), the backward UB units.
template <int FN> struct AltFwdTile {
  static constexpr int G = FnInfo<FN>::G;
  static constexpr int UT = FN == ELMAN ? 64 : 16;
  static constexpr int NC = G * UT;  // 64, 48, 64, 64
};
constexpr int ALT_UB = 16;

// Shared memory of one warp's pipeline stage: a k-chunk of the B operand and of
// the A operand (bf16, rows padded by 16 bytes against ldmatrix bank conflicts).
template <int NCOLS, int BROWS, int MT>
struct AltStage {
  static constexpr int BSTR = NCOLS + 8;  // forward: [16 k][NC] ; backward: [UB cols][16 k] uses BROWS
  static constexpr int B_ELEMS = BROWS * BSTR;
  static constexpr int ASTR = ALT_BK + 8;
  static constexpr int A_ELEMS = 16 * MT * ASTR;
  static constexpr int ELEMS = B_ELEMS + A_ELEMS;
};

// ---- forward step -----------------------------------------------------------
// 8 warps split the D/16 k-chunks (unevenly when they do not divide); after
// the product the partial sums meet in shared memory and the 256 threads take
// PPT (batch row, unit) pairs each through the cell.
constexpr int ALT_WARPS = 8, ALT_THREADS = 32 * ALT_WARPS;

template <int FN, int MT>
__global__ void __launch_bounds__(ALT_THREADS) alt_fwd_step(AltArgs a, int t) {
  constexpr int G = FnInfo<FN>::G, S = FnInfo<FN>::S, P = FnInfo<FN>::P, K = P + S;
  constexpr int UT = AltFwdTile<FN>::UT, NC = AltFwdTile<FN>::NC, NNT = NC / 8;
  constexpr int BM = 16 * MT, PPT = BM * UT / ALT_THREADS;
  using Stg = AltStage<NC, ALT_BK, MT>;  // B chunk [16 k][NC cols]
  constexpr int RSTR = NC + 8;            // fp32 row stride of the K-split partials
  const int D = a.D, N = a.N, B = a.B, T = a.T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u0 = blockIdx.x * UT, n = blockIdx.y, b0 = blockIdx.z * BM;
  const int nb = min(BM, B - b0);
  const int nchunk_all = D / ALT_BK;
  const int cbeg = warp * nchunk_all / ALT_WARPS, nchunk = (warp + 1) * nchunk_all / ALT_WARPS - cbeg;

  extern __shared__ __align__(128) unsigned char alt_smem[];
  __nv_bfloat16* wbase = (__nv_bfloat16*)alt_smem + (size_t)warp * ALT_NSTG * Stg::ELEMS;
  const __nv_bfloat16* R = (const __nv_bfloat16*)a.R;
  const __nv_bfloat16* hin = (const __nv_bfloat16*)a.xbuf + (size_t)(t & 1) * B * N * D;

  auto load_r = [&](int c) {
    __nv_bfloat16* st = wbase + (c % ALT_NSTG) * Stg::ELEMS;
    const int k0 = (cbeg + c) * ALT_BK;
    // B: rows k0..k0+15 of R[g, n, :, u0 .. u0 + UT), UT/8 pieces of 16 bytes per gate
    constexpr int PPR = G * (UT / 8);  // pieces per row
    for (int e = lane; e < ALT_BK * PPR; e += 32) {
      const int r = e / PPR, q = e - r * PPR, g = q / (UT / 8), p8 = q - g * (UT / 8);
      const __nv_bfloat16* src = R + ((size_t)(g * N + n) * D + k0 + r) * D + u0 + p8 * 8;
      cpa16(smem_u32(st + r * Stg::BSTR + g * UT + p8 * 8), src, true);
    }
  };
  auto load_h = [&](int c) {
    __nv_bfloat16* as = wbase + (c % ALT_NSTG) * Stg::ELEMS + Stg::B_ELEMS;
    const int k0 = (cbeg + c) * ALT_BK;
    // A: h_{t-1}[b0 + b, n, k0 .. k0 + 15], two pieces per row, zero rows past nb
    for (int e = lane; e < BM * 2; e += 32) {
      const int r = e >> 1, p8 = e & 1;
      const bool ok = r < nb;
      const __nv_bfloat16* src = hin + ((size_t)(b0 + (ok ? r : 0)) * N + n) * D + k0 + p8 * 8;
      cpa16(smem_u32(as + r * Stg::ASTR + p8 * 8), src, ok);
    }
  };

  float acc[MT][NNT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int j = 0; j < NNT; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[m][j][q] = 0.0f;

  // Nothing before the dependency wait depends on the previous step: R of the
  // first stages, and this step's Wx and bias for the thread's pairs, are in
  // flight while the previous step finishes. cp.async groups: R0 .. R(NS-2),
  // then h0 .. h(NS-2), then one group per later chunk; waiting for all but
  // the newest NS - 2 groups at chunk c always covers chunk c's R and h.
#pragma unroll
  for (int c = 0; c < ALT_NSTG - 1; ++c) {
    if (c < nchunk) load_r(c);
    cpa_commit();
  }
  const __nv_bfloat16* Wx = (const __nv_bfloat16*)a.Wx;
  const __nv_bfloat16* bias = (const __nv_bfloat16*)a.bias;
  float xk[PPT][G], bk[PPT][G];
#pragma unroll
  for (int k = 0; k < PPT; ++k) {
    const int e = threadIdx.x + k * ALT_THREADS, b = e / UT, u = e - b * UT, j = u0 + u;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      xk[k][g] = b < nb ? __bfloat162float(Wx[((((size_t)(b0 + b) * T + t) * G + g) * N + n) * D + j]) : 0.0f;
      bk[k][g] = __bfloat162float(bias[((size_t)g * N + n) * D + j]);
    }
  }
  pdl_wait();
#pragma unroll
  for (int c = 0; c < ALT_NSTG - 1; ++c) {
    if (c < nchunk) load_h(c);
    cpa_commit();
  }
  for (int c = 0; c < nchunk; ++c) {
    cpa_wait<ALT_NSTG - 2>();
    __syncwarp();
    if (c + ALT_NSTG - 1 < nchunk) {
      load_r(c + ALT_NSTG - 1);
      load_h(c + ALT_NSTG - 1);
    }
    cpa_commit();
    const __nv_bfloat16* st = wbase + (c % ALT_NSTG) * Stg::ELEMS;
    const __nv_bfloat16* as = st + Stg::B_ELEMS;
    uint32_t af[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
      ldmatrix_x4(smem_u32(as + (m * 16 + (lane & 15)) * Stg::ASTR + (lane >> 4) * 8), af[m][0], af[m][1], af[m][2],
                  af[m][3]);
#pragma unroll
    for (int j = 0; j < NNT; j += 2) {
      uint32_t b00, b01, b10, b11;
      const int kr = (lane & 7) + ((lane >> 3) & 1) * 8, cc = (j + (lane >> 4)) * 8;
      ldsm_x4_t(smem_u32(st + kr * Stg::BSTR + cc), b00, b01, b10, b11);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        mma_bf16_16816(acc[m][j], af[m], b00, b01);
        mma_bf16_16816(acc[m][j + 1], af[m], b10, b11);
      }
    }
  }
  cpa_wait<0>();
  // the next step may now start its own prefetch
  pdl_launch_dependents();
  __syncthreads();  // every warp is done with its pipeline: the region becomes the partial sums
  float* red = (float*)alt_smem;  // [ALT_WARPS][BM][RSTR]
  {
    float* rw = red + (size_t)warp * BM * RSTR;
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int j = 0; j < NNT; ++j) {
        const int r = m * 16 + (lane >> 2), col = j * 8 + 2 * (lane & 3);
        rw[r * RSTR + col] = acc[m][j][0];
        rw[r * RSTR + col + 1] = acc[m][j][1];
        rw[(r + 8) * RSTR + col] = acc[m][j][2];
        rw[(r + 8) * RSTR + col + 1] = acc[m][j][3];
      }
  }
  __syncthreads();

  __nv_bfloat16* states = (__nv_bfloat16*)a.states;
  __nv_bfloat16* last = (__nv_bfloat16*)a.last;
  __nv_bfloat16* hout = (__nv_bfloat16*)a.xbuf + (size_t)((t + 1) & 1) * B * N * D;
#pragma unroll
  for (int k = 0; k < PPT; ++k) {
    const int e = threadIdx.x + k * ALT_THREADS, b = e / UT, u = e - b * UT, bg = b0 + b, j = u0 + u;
    if (b >= nb) break;
    float rc[G], sp[S], sn[S], pre[P];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float v = bk[k][g];
#pragma unroll
      for (int w = 0; w < ALT_WARPS; ++w) v += red[((size_t)w * BM + b) * RSTR + g * UT + u];
      rc[g] = v;
    }
#pragma unroll
    for (int s = 0; s < S; ++s) sp[s] = a.cst[(((size_t)s * B + bg) * N + n) * D + j];
    cell_fwd<FN, true>(xk[k], rc, sp, sn, pre);
#pragma unroll
    for (int s = 0; s < S; ++s) {
      a.cst[(((size_t)s * B + bg) * N + n) * D + j] = sn[s];
      if (states) states[(((size_t)s * B + bg) * T + t) * N * D + (size_t)n * D + j] = __float2bfloat16_rn(sn[s]);
      if (last && t == T - 1) last[(((size_t)s * B + bg) * N + n) * D + j] = __float2bfloat16_rn(sn[s]);
    }
    hout[((size_t)bg * N + n) * D + j] = __float2bfloat16_rn(sn[0]);
    if (a.tape) {
      float* tp = a.tape + (((size_t)t * B + bg) * N + n) * K * D + j;
#pragma unroll
      for (int k2 = 0; k2 < P; ++k2) tp[k2 * D] = pre[k2];
#pragma unroll
      for (int s = 0; s < S; ++s) tp[(P + s) * D] = sn[s];
    }
  }
}

// h_{-1} into the ping-pong buffer, carried states (fp32) from states0.
template <int FN>
__global__ void alt_fwd_init(AltArgs a) {
  constexpr int S = FnInfo<FN>::S;
  const size_t per = (size_t)a.B * a.N * a.D;
  const __nv_bfloat16* s0 = (const __nv_bfloat16*)a.s0;
  __nv_bfloat16* h = (__nv_bfloat16*)a.xbuf;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < per; e += (size_t)gridDim.x * blockDim.x) {
#pragma unroll
    for (int s = 0; s < S; ++s) {
      const float v = s0 ? __bfloat162float(s0[s * per + e]) : 0.0f;
      a.cst[s * per + e] = v;
      if (s == 0) h[e] = __float2bfloat16_rn(v);
    }
  }
}

// ---- backward step ------------------------------------------------------------
template <int FN, int MT>
__global__ void __launch_bounds__(ALT_THREADS) alt_bwd_step(AltArgs a, int t) {
  constexpr int G = FnInfo<FN>::G, S = FnInfo<FN>::S, P = FnInfo<FN>::P, K = P + S;
  constexpr int UB = ALT_UB, NNT = UB / 8;
  constexpr int BM = 16 * MT, PPT = BM * UB / ALT_THREADS;
  // B chunk stored [UB cols (units i)][16 k]: each column's k values contiguous
  using Stg = AltStage<ALT_BK, UB, MT>;
  constexpr int RSTR = UB + 4;
  const int D = a.D, N = a.N, B = a.B, T = a.T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i0 = blockIdx.x * UB, n = blockIdx.y, b0 = blockIdx.z * BM;
  const int nb = min(BM, B - b0);
  const int nchunk_all = G * D / ALT_BK;
  const int cbeg = warp * nchunk_all / ALT_WARPS, nchunk = (warp + 1) * nchunk_all / ALT_WARPS - cbeg;
  const bool have_rec = t < T - 1;  // dr_{t+1} exists

  extern __shared__ __align__(128) unsigned char alt_smem[];
  __nv_bfloat16* wbase = (__nv_bfloat16*)alt_smem + (size_t)warp * ALT_NSTG * Stg::ELEMS;
  const __nv_bfloat16* R = (const __nv_bfloat16*)a.R;
  const size_t drsz = (size_t)B * G * N * D;
  const __nv_bfloat16* drin = (const __nv_bfloat16*)a.xbuf + (size_t)((t + 1) & 1) * drsz;

  // the gate of 16-wide chunk kc of the G D inputs, by comparison (G <= 4)
  // rather than a division by D
  const int d16 = D / ALT_BK;
  auto chunk_gate = [&](int kc) {
    int g = 0;
#pragma unroll
    for (int q = 1; q < G; ++q) g += kc >= q * d16;
    return g;
  };
  auto load_r = [&](int c) {
    __nv_bfloat16* st = wbase + (c % ALT_NSTG) * Stg::ELEMS;
    const int kc = cbeg + c, g = chunk_gate(kc), j0 = (kc - g * d16) * ALT_BK;
    // B: R[g, n, i0 + i, j0 .. j0 + 15] for the UB units i, two pieces each
    const int i = lane >> 1, p8 = lane & 1;  // UB * 2 = 32 pieces
    const __nv_bfloat16* src = R + ((size_t)(g * N + n) * D + i0 + i) * D + j0 + p8 * 8;
    cpa16(smem_u32(st + i * Stg::BSTR + p8 * 8), src, true);
  };
  auto load_dr = [&](int c) {
    __nv_bfloat16* st = wbase + (c % ALT_NSTG) * Stg::ELEMS;
    const int kc = cbeg + c, g = chunk_gate(kc), j0 = (kc - g * d16) * ALT_BK;
    // A: dr_{t+1}[b0 + b, g, n, j0 .. j0 + 15]
    __nv_bfloat16* as = st + Stg::B_ELEMS;
    for (int e = lane; e < BM * 2; e += 32) {
      const int r = e >> 1, p8 = e & 1;
      const bool ok = r < nb;
      const __nv_bfloat16* src = drin + (((size_t)(b0 + (ok ? r : 0)) * G + g) * N + n) * D + j0 + p8 * 8;
      cpa16(smem_u32(as + r * Stg::ASTR + p8 * 8), src, ok);
    }
  };

  float acc[MT][NNT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int j = 0; j < NNT; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[m][j][q] = 0.0f;
  if (have_rec) {  // R first, the previous step's dr after the dependency wait
#pragma unroll
    for (int c = 0; c < ALT_NSTG - 1; ++c) {
      if (c < nchunk) load_r(c);
      cpa_commit();
    }
  }
  // the tape and the upstream gradients of this step come from earlier work:
  // loaded before the dependency wait too
  const __nv_bfloat16* s0 = (const __nv_bfloat16*)a.s0;
  const __nv_bfloat16* dstates = (const __nv_bfloat16*)a.dstates;
  const __nv_bfloat16* dlast = (const __nv_bfloat16*)a.dlast;
  float prek[PPT][P], snk[PPT][S], spk[PPT][S], upk[PPT][S];
  if (t >= 0) {
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
      const int e = threadIdx.x + k * ALT_THREADS, b = e / UB, u = e - b * UB, j = i0 + u;
      const int bg = b0 + (b < nb ? b : 0);
      const float* tp = a.tape + (((size_t)t * B + bg) * N + n) * K * D + j;
#pragma unroll
      for (int k2 = 0; k2 < P; ++k2) prek[k][k2] = tp[k2 * D];
#pragma unroll
      for (int s = 0; s < S; ++s) {
        snk[k][s] = tp[(P + s) * D];
        if (t > 0)
          spk[k][s] = a.tape[(((size_t)(t - 1) * B + bg) * N + n) * K * D + (size_t)(P + s) * D + j];
        else
          spk[k][s] = s0 ? __bfloat162float(s0[(((size_t)s * B + bg) * N + n) * D + j]) : 0.0f;
        float d = 0.0f;
        if (dstates) d += __bfloat162float(dstates[(((size_t)s * B + bg) * T + t) * N * D + (size_t)n * D + j]);
        if (dlast && t == T - 1) d += __bfloat162float(dlast[(((size_t)s * B + bg) * N + n) * D + j]);
        upk[k][s] = d;
      }
    }
  }
  pdl_wait();
  if (have_rec) {
#pragma unroll
    for (int c = 0; c < ALT_NSTG - 1; ++c) {
      if (c < nchunk) load_dr(c);
      cpa_commit();
    }
    for (int c = 0; c < nchunk; ++c) {
      cpa_wait<ALT_NSTG - 2>();
      __syncwarp();
      if (c + ALT_NSTG - 1 < nchunk) {
        load_r(c + ALT_NSTG - 1);
        load_dr(c + ALT_NSTG - 1);
      }
      cpa_commit();
      const __nv_bfloat16* st = wbase + (c % ALT_NSTG) * Stg::ELEMS;
      const __nv_bfloat16* as = st + Stg::B_ELEMS;
      uint32_t af[MT][4];
#pragma unroll
      for (int m = 0; m < MT; ++m)
        ldmatrix_x4(smem_u32(as + (m * 16 + (lane & 15)) * Stg::ASTR + (lane >> 4) * 8), af[m][0], af[m][1],
                    af[m][2], af[m][3]);
      // B fragments of both n8 tiles: rows = units, 8 k values per row
      uint32_t b00, b01, b10, b11;
      ldmatrix_x4(smem_u32(st + ((lane >> 4) * 8 + (lane & 7)) * Stg::BSTR + ((lane >> 3) & 1) * 8), b00, b01, b10,
                  b11);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        mma_bf16_16816(acc[m][0], af[m], b00, b01);
        mma_bf16_16816(acc[m][1], af[m], b10, b11);
      }
    }
    cpa_wait<0>();
  }
  pdl_launch_dependents();
  __syncthreads();
  float* red = (float*)alt_smem;  // [ALT_WARPS][BM][RSTR]
  {
    float* rw = red + (size_t)warp * BM * RSTR;
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int j = 0; j < NNT; ++j) {
        const int r = m * 16 + (lane >> 2), col = j * 8 + 2 * (lane & 3);
        rw[r * RSTR + col] = acc[m][j][0];
        rw[r * RSTR + col + 1] = acc[m][j][1];
        rw[(r + 8) * RSTR + col] = acc[m][j][2];
        rw[(r + 8) * RSTR + col + 1] = acc[m][j][3];
      }
  }
  __syncthreads();

  __nv_bfloat16* dWx = (__nv_bfloat16*)a.dWx;
  __nv_bfloat16* dro = (__nv_bfloat16*)a.dr;
  const bool write_dr = dro && (FN == GRU || (void*)dro != (void*)dWx);
  __nv_bfloat16* drout = (__nv_bfloat16*)a.xbuf + (size_t)(t & 1) * drsz;
#pragma unroll
  for (int k = 0; k < PPT; ++k) {
    const int e = threadIdx.x + k * ALT_THREADS, b = e / UB, u = e - b * UB, bg = b0 + b, j = i0 + u;
    if (b >= nb) break;
    float dh = 0.0f;
#pragma unroll
    for (int w = 0; w < ALT_WARPS; ++w) dh += red[((size_t)w * BM + b) * RSTR + u];
    if (t < 0) {  // dstates0: carried gradients plus the product of dr_0
      __nv_bfloat16* ds0 = (__nv_bfloat16*)a.ds0;
#pragma unroll
      for (int s = 0; s < S; ++s) {
        float v = a.cst[(((size_t)s * B + bg) * N + n) * D + j];
        if (s == 0) v += dh;
        ds0[(((size_t)s * B + bg) * N + n) * D + j] = __float2bfloat16_rn(v);
      }
      continue;
    }
    float dsn[S], dx[G], dr[G], dsp[S];
#pragma unroll
    for (int s = 0; s < S; ++s) {
      float d = a.cst[(((size_t)s * B + bg) * N + n) * D + j] + upk[k][s];
      if (s == 0) d += dh;
      dsn[s] = d;
    }
    cell_bwd<FN, true>(prek[k], spk[k], snk[k], dsn, dx, dr, dsp);
    const size_t o = (((size_t)bg * T + t) * G) * N * D + (size_t)n * D + j;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (dWx) dWx[o + (size_t)g * N * D] = __float2bfloat16_rn(dx[g]);
      if (write_dr) dro[o + (size_t)g * N * D] = __float2bfloat16_rn(dr[g]);
      drout[(((size_t)bg * G + g) * N + n) * D + j] = __float2bfloat16_rn(dr[g]);
    }
#pragma unroll
    for (int s = 0; s < S; ++s) a.cst[(((size_t)s * B + bg) * N + n) * D + j] = dsp[s];
  }
}

__global__ void alt_zero(float* p, size_t n) {
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x)
    p[e] = 0.0f;
}

template <int FN, int MT>
size_t alt_fwd_smem() {
  constexpr int NC = AltFwdTile<FN>::NC;
  const size_t pipe = (size_t)ALT_WARPS * ALT_NSTG * AltStage<NC, ALT_BK, MT>::ELEMS * 2;
  const size_t red = (size_t)ALT_WARPS * 16 * MT * (NC + 8) * 4;
  return pipe > red ? pipe : red;
}
template <int FN, int MT>
size_t alt_bwd_smem() {
  const size_t pipe = (size_t)ALT_WARPS * ALT_NSTG * AltStage<ALT_BK, ALT_UB, MT>::ELEMS * 2;
  const size_t red = (size_t)ALT_WARPS * 16 * MT * (ALT_UB + 4) * 4;
  return pipe > red ? pipe : red;
}

// ---- graph capture and replay -----------------------------------------------------
struct GraphKey {
  int dev, fn, bwd, B, T, N, D;
  const void* p[14];
  bool operator==(const GraphKey& o) const {
    if (dev != o.dev || fn != o.fn || bwd != o.bwd || B != o.B || T != o.T || N != o.N || D != o.D) return false;
    for (int k = 0; k < 14; ++k)
      if (p[k] != o.p[k]) return false;
    return true;
  }
};
std::mutex g_graph_mu;
std::vector<std::pair<GraphKey, cudaGraphExec_t>> g_graphs;  // most recent last
constexpr size_t kMaxGraphs = 8;
cudaStream_t g_capture_stream[64] = {};

GraphKey key_of(int fn, bool bwd, const AltArgs& a) {
  GraphKey k{};
  cudaGetDevice(&k.dev);
  k.fn = fn; k.bwd = bwd; k.B = a.B; k.T = a.T; k.N = a.N; k.D = a.D;
  const void* p[14] = {a.Wx, a.R, a.bias, a.s0, a.states, a.last, a.tape, a.dstates,
                       a.dlast, a.dWx, a.dr, a.ds0, a.xbuf, a.cst};
  for (int i = 0; i < 14; ++i) k.p[i] = p[i];
  return k;
}

// Launch with programmatic stream serialisation: the kernel may begin while
// its predecessor in the stream still runs; it orders itself with
// griddepcontrol.wait.
template <typename... Args>
cudaError_t launch_pdl(void (*k)(Args...), dim3 grid, int threads, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

template <int FN, int MT>
cudaError_t enqueue_fwd(const AltArgs& a, cudaStream_t st) {
  constexpr int UT = AltFwdTile<FN>::UT;
  const size_t smem = alt_fwd_smem<FN, MT>();
  cudaError_t e = set_smem_attr((const void*)alt_fwd_step<FN, MT>, smem);
  if (e != cudaSuccess) return e;
  const size_t per = (size_t)a.B * a.N * a.D;
  alt_fwd_init<FN><<<(unsigned)((per + 255) / 256 < 1184 ? (per + 255) / 256 : 1184), 256, 0, st>>>(a);
  const dim3 grid(a.D / UT, a.N, (a.B + 16 * MT - 1) / (16 * MT));
  for (int t = 0; t < a.T && e == cudaSuccess; ++t) e = launch_pdl(alt_fwd_step<FN, MT>, grid, ALT_THREADS, smem, st, a, t);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int FN, int MT>
cudaError_t enqueue_bwd(const AltArgs& a, cudaStream_t st) {
  constexpr int S = FnInfo<FN>::S;
  const size_t smem = alt_bwd_smem<FN, MT>();
  cudaError_t e = set_smem_attr((const void*)alt_bwd_step<FN, MT>, smem);
  if (e != cudaSuccess) return e;
  const size_t n = (size_t)S * a.B * a.N * a.D;
  alt_zero<<<(unsigned)((n + 255) / 256 < 1184 ? (n + 255) / 256 : 1184), 256, 0, st>>>(a.cst, n);
  const dim3 grid(a.D / ALT_UB, a.N, (a.B + 16 * MT - 1) / (16 * MT));
  for (int t = a.T - 1; t >= 0 && e == cudaSuccess; --t)
    e = launch_pdl(alt_bwd_step<FN, MT>, grid, ALT_THREADS, smem, st, a, t);
  if (a.ds0 && e == cudaSuccess) e = launch_pdl(alt_bwd_step<FN, MT>, grid, ALT_THREADS, smem, st, a, -1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int FN>
cudaError_t enqueue(const AltArgs& a, bool bwd, cudaStream_t st) {
  if (a.B <= 16) return bwd ? enqueue_bwd<FN, 1>(a, st) : enqueue_fwd<FN, 1>(a, st);
  return bwd ? enqueue_bwd<FN, 2>(a, st) : enqueue_fwd<FN, 2>(a, st);
}

cudaError_t enqueue_any(int fn, const AltArgs& a, bool bwd, cudaStream_t st) {
  switch (fn) {
    case LSTM: return enqueue<LSTM>(a, bwd, st);
    case GRU: return enqueue<GRU>(a, bwd, st);
    case ELMAN: return enqueue<ELMAN>(a, bwd, st);
    case SLSTM: return enqueue<SLSTM>(a, bwd, st);
    case SLSTM_LS: return enqueue<SLSTM_LS>(a, bwd, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t alt_run(int fn, const AltArgs& a, bool bwd, cudaStream_t st) {
  const GraphKey key = key_of(fn, bwd, a);
  std::lock_guard<std::mutex> lock(g_graph_mu);
  cudaGraphExec_t exec = nullptr;
  for (size_t i = 0; i < g_graphs.size(); ++i)
    if (g_graphs[i].first == key) {
      exec = g_graphs[i].second;
      auto item = g_graphs[i];
      g_graphs.erase(g_graphs.begin() + i);
      g_graphs.push_back(item);
      break;
    }
  if (!exec) {
    if (key.dev < 0 || key.dev >= 64) return cudaErrorInvalidDevice;
    cudaStream_t& cs = g_capture_stream[key.dev];
    cudaError_t e = cudaSuccess;
    if (!cs) e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
    e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return e;
    const cudaError_t le = enqueue_any(fn, a, bwd, cs);
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(cs, &graph);
    if (le != cudaSuccess) {
      if (graph) cudaGraphDestroy(graph);
      return le;
    }
    if (e != cudaSuccess) return e;
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return e;
    if (g_graphs.size() >= kMaxGraphs) {
      cudaGraphExecDestroy(g_graphs.front().second);
      g_graphs.erase(g_graphs.begin());
    }
    g_graphs.push_back({key, exec});
  }
  note_launch(1 + (bwd ? a.T + (a.ds0 ? 1 : 0) : a.T));
  return cudaGraphLaunch(exec, st);
}

}  // namespace

size_t alt_scratch_bytes(int fn, int B, int N, int D, bool bwd) {
  const size_t per = (size_t)B * N * D;
  const size_t x = bwd ? 2 * per * fn_gates(fn) * 2 : 2 * per * 2;  // bf16 ping-pong
  const size_t c = (size_t)fn_states(fn) * per * 4;                 // fp32 carried values
  return ((x + 255) & ~(size_t)255) + ((c + 255) & ~(size_t)255);
}

int alt_supported(int fn, int D) {
  const int UT = fn == ELMAN ? 64 : 16;
  return D % 16 == 0 && D % UT == 0 && D % ALT_UB == 0;
}

cudaError_t alt_fwd_run(int fn, const AltArgs& a, cudaStream_t st) { return alt_run(fn, a, false, st); }
cudaError_t alt_bwd_run(int fn, const AltArgs& a, cudaStream_t st) { return alt_run(fn, a, true, st); }

}  // namespace rnn
