// Persistent thread-block-cluster backward scan (bf16 storage, fp32 arithmetic).
//
// Reverse-time counterpart of the forward cluster kernel. One cluster of C
// CTAs runs one head and batch group from t = T-1 down to 0; CTA c owns units
// [c*U, (c+1)*U) and carries their state gradients (fp32, registers).
// Per step:
//   0. the tape, the upstream gradients and the gate activations of the
//      CTA's (row, unit) pairs, which do not depend on dh_t, while its
//      partial products are still arriving;
//   1. dh_t[own units] = sum over the C CTAs of the fp32 partial products
//      received for this step (plus dstates[:, t] and the carried terms);
//   2. the cell derivative gives dWx[:, t] and the recurrent-branch gradient
//      dr_t of the CTA's units (written out for the weight gradients);
//   3. the CTA multiplies its own dr_t (bf16) with its resident slice of R,
//        partial[i, b] = sum_{g, j in own units} R[g, n, i, j] dr_t[b, g, j],
//      for ALL rows i (M = D, K = G*U, N = batch) on the tensor cores, and
//   4. pushes each 16-row block of partials to the CTA owning those rows with
//      st.async (a reduce-scatter; the owner's mbarrier counts the bytes).
// tape[t] and dstates[:, t] stream in through a TMA ring several steps ahead.
#pragma once
#include <cuda.h>

#include "kernels.cuh"
#include "layout.h"
#include "ptx.cuh"

namespace rnn {

template <int FN, int NT, int MT>
__global__ void __launch_bounds__(256, 1)
    fused_bwd_kernel(const __grid_constant__ CUtensorMap tapemap, const __grid_constant__ CUtensorMap dstmap,
                     FusedArgs a) {
  constexpr int G = FnInfo<FN>::G, S = FnInfo<FN>::S, P = FnInfo<FN>::P, K = P + S;
  constexpr int BC = 8 * NT;
  constexpr int KTM = FUSED_BWD_MAX_KTA;
  const int C = a.C, U = a.U, D = a.D, TT = a.T, N = a.N, B = a.B;
  const int KTA = G * U / 16;  // k-tiles of the CTA's own gradient block
  const int KB = G * U + 8;    // row stride (elements) of the gradient operand
  const uint32_t rank = cluster_ctarank();
  const int grp = blockIdx.x / C;
  const int n = grp % N;
  const int b0 = (grp / N) * BC;
  const int nb = min(BC, B - b0);
  const int u0 = (int)rank * U;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;

  extern __shared__ __align__(128) unsigned char smem[];
  const FusedBwdSmem L = FusedBwdSmem::make(G, S, K, U, BC, C);
  uint64_t* bars = (uint64_t*)(smem + L.bars);  // [0,1]: partials full; [2..]: ring
  unsigned char* ring = smem + L.ring;
  // [2][C][U][BC]; within a unit's row the 16-byte groups of batch columns are
  // XOR-swizzled by the unit (column b is stored at b ^ 4 swz(u)), so that
  // readers of one batch column across 16 consecutive units meet at most
  // two-way bank conflicts while each sender's pair of lanes still fills
  // whole aligned 32-byte sectors
  float* recv = (float*)(smem + L.recv);
  auto swz = [](int u) { return NT == 1 ? ((u >> 2) & 1) : ((u >> 1) & 3); };
  __nv_bfloat16* drb = (__nv_bfloat16*)(smem + L.drb);  // [2][BC][KB]
  float* s0s = (float*)(smem + L.s0);   // [S][BC][U]
  float* dbs = (float*)(smem + L.dbs);  // [G][BC][U]: the pairs' sums of dr, gathered at the end
  const bool with_db = a.dbp != nullptr;
  const uint32_t recv_bar0 = smem_u32(&bars[0]);
  const uint32_t ring_bar0 = smem_u32(&bars[2]);
  const uint32_t rbytes = (uint32_t)C * U * BC * 4;  // payload bytes (padding not sent)
  const bool has_dst = a.dstates != nullptr;
  const uint32_t stage_bytes = (uint32_t)(L.tape_bytes + (has_dst ? (size_t)S * BC * U * 2 : 0));

  const __nv_bfloat16* R = (const __nv_bfloat16*)a.R;
  const __nv_bfloat16* s0 = (const __nv_bfloat16*)a.s0;
  const __nv_bfloat16* dlast = (const __nv_bfloat16*)a.dlast;
  __nv_bfloat16* dWx = (__nv_bfloat16*)a.dWx;
  __nv_bfloat16* dro = (__nv_bfloat16*)a.dr;
  const bool write_dr = dro && (FN == GRU || (void*)dro != (void*)dWx);

  // ---- prologue --------------------------------------------------------------
  if (tid == 0) {
    mbar_init(recv_bar0, 1);
    mbar_init(recv_bar0 + 8, 1);
    for (int s = 0; s < FUSED_NS; ++s) mbar_init(ring_bar0 + 8 * s, 1);
    fence_mbar_init_cluster();
    prefetch_tensormap(&tapemap);
    if (has_dst) prefetch_tensormap(&dstmap);
  }
  for (int e = tid; e < 2 * BC * KB; e += nthr) drb[e] = __float2bfloat16_rn(0.0f);
  for (int e = tid; e < S * BC * U; e += nthr) {
    const int s = e / (BC * U), r = e - s * BC * U, b = r / U, u = r - b * U;
    float v = 0.0f;
    if (b < nb && s0) v = __bfloat162float(s0[(((size_t)s * B + b0 + b) * N + n) * D + u0 + u]);
    s0s[e] = v;
  }
  // carried state gradients of this thread's (batch row, unit) pairs
  // e = tid + k * blockDim (k < FUSED_PPT), in registers for the whole scan
  // and their (row, unit) coordinates, divided once here rather than every step
  float dsr[FUSED_PPT][S];
  int prow[FUSED_PPT], punit[FUSED_PPT];
#pragma unroll
  for (int k = 0; k < FUSED_PPT; ++k) {
    prow[k] = (tid + k * nthr) / U;
    punit[k] = tid + k * nthr - prow[k] * U;
#pragma unroll
    for (int s = 0; s < S; ++s) dsr[k][s] = 0.0f;
  }
  // resident R fragments: A[m = row i][k = (g, j)] = R[g, n, i, u0 + j]
  uint32_t afr[MT][KTM][4];
  {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int ir = (warp * MT + mt) * 16 + (lane >> 2);
#pragma unroll
      for (int kt = 0; kt < KTM; ++kt) {
        if (kt < KTA) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int i = ir + ((q & 1) ? 8 : 0);
            const int k = kt * 16 + 2 * (lane & 3) + ((q & 2) ? 8 : 0);
            const int g = k / U, j = k - g * U;
            afr[mt][kt][q] = *(const uint32_t*)(R + ((size_t)(g * N + n) * D + i) * D + u0 + j);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) afr[mt][kt][q] = 0u;
        }
      }
    }
  }
  __syncthreads();
  cluster_sync_all();

  auto issue_stage = [&](int k) {  // processing index k <-> time step T-1-k
    const int t = TT - 1 - k, s = k % FUSED_NS;
    unsigned char* st = ring + (size_t)s * L.ring_stage;
    mbar_arrive_expect_tx(ring_bar0 + 8 * s, stage_bytes);
    tma_load_5d(smem_u32(st), &tapemap, ring_bar0 + 8 * s, u0, 0, n, b0, t);
    if (has_dst) tma_load_5d(smem_u32(st + L.dst_off), &dstmap, ring_bar0 + 8 * s, u0, n, t, b0, 0);
  };
  if (tid == 0) {
    mbar_arrive_expect_tx(recv_bar0 + 8 * ((TT - 2) & 1), rbytes);
    if (TT >= 2) mbar_arrive_expect_tx(recv_bar0 + 8 * ((TT - 3) & 1), rbytes);
    for (int k = 0; k < FUSED_NS && k < TT; ++k) issue_stage(k);
  }

  bool failed = false;
  float dbv[FUSED_PPT][G];      // the pairs' running sums of dr over the steps (db)
#pragma unroll
  for (int kp = 0; kp < FUSED_PPT; ++kp)
#pragma unroll
    for (int g = 0; g < G; ++g) dbv[kp][g] = 0.0f;
  uint32_t ph0 = 0u, ph1 = 0u;  // phase parity of the two partial-sum barriers
  const int q4 = lane & 3, r8 = lane >> 2;
  // each lane always sends row i = (warp*MT + mt)*16 + r8 (+8 on odd lanes):
  // its owner CTA and the cluster addresses there are fixed for the kernel
  uint32_t send_base0[MT], send_base1[MT], send_bar0[MT], send_bar1[MT];
  int send_row[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int i = (warp * MT + mt) * 16 + r8 + ((q4 & 1) ? 8 : 0);
    const int owner = i / U;
    send_row[mt] = i - owner * U;
    send_base0[mt] = mapa_shared(smem_u32(recv + (size_t)rank * U * BC), (uint32_t)owner);
    send_base1[mt] = mapa_shared(smem_u32(recv + ((size_t)C + rank) * U * BC), (uint32_t)owner);
    send_bar0[mt] = mapa_shared(recv_bar0, (uint32_t)owner);
    send_bar1[mt] = mapa_shared(recv_bar0 + 8, (uint32_t)owner);
  }

  const bool tracer = a.trace && blockIdx.x == 0 && tid == 0;
#define RNN_TRACE(p)                                                                    \
  if (tracer && k >= a.trace_t0 && k < a.trace_t0 + a.trace_steps)                      \
    a.trace[(size_t)(k - a.trace_t0) * 16 + (p)] = (unsigned long long)clock64();

  // ---- reverse time loop ---------------------------------------------------------
  for (int k = 0; k < TT; ++k) {
    const int t = TT - 1 - k;
    const int pb = t & 1;  // gradient-operand buffer of this step
    RNN_TRACE(0)
    const int sc = k % FUSED_NS, sn_ = (k + 1) % FUSED_NS;
    const float* tp = (const float*)(ring + (size_t)sc * L.ring_stage);
    const __nv_bfloat16* dstage = (const __nv_bfloat16*)(ring + (size_t)sc * L.ring_stage + L.dst_off);
    const float* tq = (const float*)(ring + (size_t)sn_ * L.ring_stage);
    if (k == 0 && tid < nb * U) {  // later steps: waited for one step ahead, below
      mbar_wait_bounded<false>(ring_bar0 + 8 * sc, (k / FUSED_NS) & 1, a.wait_limit_ns, a.status, failed);
      if (t > 0)
        mbar_wait_bounded<false>(ring_bar0 + 8 * sn_, ((k + 1) / FUSED_NS) & 1, a.wait_limit_ns, a.status, failed);
    }
    // The tape, the upstream gradients and the gate activations of the step
    // do not depend on dh_t: they are evaluated while its partial sums are
    // still arriving.
    float pre[FUSED_PPT][P], sp[FUSED_PPT][S], sn[FUSED_PPT][S], dsn[FUSED_PPT][S];
    float act[FUSED_PPT][CELL_BWD_ACT];
#pragma unroll
    for (int kp = 0; kp < FUSED_PPT; ++kp) {
      if (tid + kp * nthr < nb * U) {
        const int b = prow[kp], u = punit[kp];
#pragma unroll
        for (int kk = 0; kk < P; ++kk) pre[kp][kk] = tp[(b * K + kk) * U + u];
#pragma unroll
        for (int s = 0; s < S; ++s) {
          sn[kp][s] = tp[(b * K + P + s) * U + u];
          sp[kp][s] = t > 0 ? tq[(b * K + P + s) * U + u] : s0s[(s * BC + b) * U + u];
          float d = dsr[kp][s];
          if (has_dst) d += __bfloat162float(dstage[(s * BC + b) * U + u]);
          if (dlast && t == TT - 1) d += __bfloat162float(dlast[(((size_t)s * B + b0 + b) * N + n) * D + u0 + u]);
          dsn[kp][s] = d;
        }
        cell_bwd_act<FN, true>(pre[kp], sp[kp], sn[kp], act[kp]);
      }
    }
    RNN_TRACE(1)
    if (t < TT - 1) {  // partial sums for dh_t arrived
      const int bi = t & 1;
      mbar_wait_bounded(recv_bar0 + 8 * bi, bi ? ph1 : ph0, a.wait_limit_ns, a.status, failed);
      if (bi) ph1 ^= 1u; else ph0 ^= 1u;
      if (tid == 0 && t - 2 >= -1) mbar_arrive_expect_tx(recv_bar0 + 8 * bi, rbytes);
    }
    RNN_TRACE(2)
    const float* rv = recv + (size_t)(t & 1) * C * U * BC;
    __nv_bfloat16* drw = drb + (size_t)pb * BC * KB;
#pragma unroll
    for (int kp = 0; kp < FUSED_PPT; ++kp) {
      if (tid + kp * nthr < nb * U) {
        const int b = prow[kp], u = punit[kp];
        float dx[G], dr[G], dsp[S];
        if (t < TT - 1) {  // the C partial sums, loaded together
          float part[FUSED_MAX_C];
          const int bs = b ^ (4 * swz(u));
#pragma unroll
          for (int c = 0; c < FUSED_MAX_C; ++c) part[c] = c < C ? rv[(c * U + u) * BC + bs] : 0.0f;
          float acc = 0.0f;
#pragma unroll
          for (int c = 0; c < FUSED_MAX_C; ++c) acc += part[c];
          dsn[kp][0] += acc;
        }
        cell_bwd_grad<FN, true>(act[kp], pre[kp], sp[kp], dsn[kp], dx, dr, dsp);
        const size_t o = (((size_t)(b0 + b) * TT + t) * G) * N * D + (size_t)n * D + u0 + u;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          if (dWx) dWx[o + (size_t)g * N * D] = __float2bfloat16_rn(dx[g]);
          if (write_dr) dro[o + (size_t)g * N * D] = __float2bfloat16_rn(dr[g]);
          drw[b * KB + g * U + u] = __float2bfloat16_rn(dr[g]);
        }
        if (with_db)  // db: the pair's running sum (the pair stays with this thread)
#pragma unroll
          for (int g = 0; g < G; ++g) dbv[kp][g] += dr[g];
#pragma unroll
        for (int s = 0; s < S; ++s) dsr[kp][s] = dsp[s];
      }
    }
    // one thread observes the TMA completion of the two stages the next step
    // reads (loaded NS - 2 or more steps ago); the barrier below orders them
    // for every thread
    if (tid == nthr - 1 && k + 1 < TT) {
      mbar_wait_bounded<false>(ring_bar0 + 8 * ((k + 1) % FUSED_NS), ((k + 1) / FUSED_NS) & 1, a.wait_limit_ns,
                               a.status, failed);
      if (k + 2 < TT)
        mbar_wait_bounded<false>(ring_bar0 + 8 * ((k + 2) % FUSED_NS), ((k + 2) / FUSED_NS) & 1, a.wait_limit_ns,
                                 a.status, failed);
    }
    RNN_TRACE(3)
    __syncthreads();
    RNN_TRACE(4)

    // partial[i, b] = sum_k A[i][k] drb[b][k] for this warp's MT m-tiles
    float acc[MT][NT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[mt][nt][q] = 0.0f;
    const uint32_t hb = smem_u32(drw);
#pragma unroll
    for (int kt = 0; kt < KTM; ++kt) {
      if (kt < KTA) {
        const int k0 = kt * 16;
        uint32_t bf[NT][2];
        if constexpr (NT == 1) {
          const uint32_t addr = hb + (uint32_t)(((lane & 7) * KB + k0 + ((lane >> 3) & 1) * 8) * 2);
          ldmatrix_x2(addr, bf[0][0], bf[0][1]);
        } else {
#pragma unroll
          for (int np = 0; np < NT; np += 2) {
            const int q = lane >> 3;
            const uint32_t addr =
                hb + (uint32_t)((((np + (q >> 1)) * 8 + (lane & 7)) * KB + k0 + (q & 1) * 8) * 2);
            ldmatrix_x4(addr, bf[np][0], bf[np][1], bf[np + 1][0], bf[np + 1][1]);
          }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[mt][nt], afr[mt][kt], bf[nt][0], bf[nt][1]);
      }
    }
    RNN_TRACE(5)
    // reduce-scatter: each lane assembles 4 consecutive batch columns of one row
    {
      const int bi = (t - 1) & 1;  // consumption t-1 (t = 0 feeds the final dh_{-1})
      const bool even = (q4 & 1) == 0;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float* v = acc[mt][nt];
          const float sa = even ? v[2] : v[0];
          const float sb = even ? v[3] : v[1];
          const float ra = __shfl_xor_sync(0xffffffffu, sa, 1);
          const float rb = __shfl_xor_sync(0xffffffffu, sb, 1);
          uint4 out;
          int bcol;
          if (even) {
            out = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(ra), __float_as_uint(rb));
            bcol = nt * 8 + 2 * q4;
          } else {
            out = make_uint4(__float_as_uint(ra), __float_as_uint(rb), __float_as_uint(v[2]), __float_as_uint(v[3]));
            bcol = nt * 8 + 2 * q4 - 2;
          }
          const uint32_t off = (uint32_t)((send_row[mt] * BC + (bcol ^ (4 * swz(send_row[mt])))) * 4);
          st_async_16((bi ? send_base1[mt] : send_base0[mt]) + off, out, bi ? send_bar1[mt] : send_bar0[mt]);
        }
    }
    RNN_TRACE(6)
    // tape and upstream gradients of step k + NS into the ring slot this
    // step's derivative has finished reading
    if (tid == nthr - 32 && k + FUSED_NS < TT) issue_stage(k + FUSED_NS);
  }
#undef RNN_TRACE

  // ---- dstates0: the carried gradients after step 0 ------------------------------
  {
    const int bi = 1;  // consumption -1
    mbar_wait_bounded(recv_bar0 + 8 * bi, ph1, a.wait_limit_ns, a.status, failed);  // bi == 1
    const float* rv = recv + (size_t)bi * C * U * BC;
    __nv_bfloat16* ds0 = (__nv_bfloat16*)a.ds0;
    if (ds0) {
#pragma unroll
      for (int kp = 0; kp < FUSED_PPT; ++kp) {
        const int e = tid + kp * nthr;
        if (e >= nb * U) break;
        const int b = e / U, u = e - b * U;
#pragma unroll
        for (int s = 0; s < S; ++s) {
          float v = dsr[kp][s];
          if (s == 0)
            for (int c = 0; c < C; ++c) v += rv[((size_t)c * U + u) * BC + (b ^ (4 * swz(u)))];
          ds0[(((size_t)s * B + b0 + b) * N + n) * D + u0 + u] = __float2bfloat16_rn(v);
        }
      }
    }
  }
  if (with_db)
#pragma unroll
    for (int kp = 0; kp < FUSED_PPT; ++kp)
      if (tid + kp * nthr < nb * U)
#pragma unroll
        for (int g = 0; g < G; ++g) dbs[(g * BC + prow[kp]) * U + punit[kp]] = dbv[kp][g];
  __syncthreads();
  // db partial of the batch block: the column sums over its rows, in row order
  if (with_db)
    for (int e = tid; e < G * U; e += nthr) {
      const int g = e / U, u = e - g * U;
      float v = 0.0f;
      for (int b = 0; b < nb; ++b) v += dbs[(g * BC + b) * U + u];
      a.dbp[(((size_t)(grp / N) * G + g) * N + n) * D + u0 + u] = v;
    }
  cluster_sync_all();
}

template <int FN>
cudaError_t fused_bwd_launch(const FusedShape& sh, const FusedArgs& a, cudaStream_t st) {
  constexpr int G = FnInfo<FN>::G, S = FnInfo<FN>::S, K = FnInfo<FN>::P + FnInfo<FN>::S;
  void (*k)(const CUtensorMap, const CUtensorMap, FusedArgs) = nullptr;
#define RNN_FUSED_BWD_PICK(NT_, MT_) \
  if (sh.NT == NT_ && sh.MT == MT_) k = fused_bwd_kernel<FN, NT_, MT_>;
  RNN_FUSED_BWD_PICK(1, 1) RNN_FUSED_BWD_PICK(1, 2) RNN_FUSED_BWD_PICK(2, 1) RNN_FUSED_BWD_PICK(2, 2)
#undef RNN_FUSED_BWD_PICK
  if (!k) return cudaErrorInvalidValue;
  const unsigned BC = 8u * sh.NT;
  CUtensorMap tmap, dmap;
  {
    const unsigned long long dims[5] = {(unsigned long long)a.D, (unsigned long long)K,
                                        (unsigned long long)a.N, (unsigned long long)a.B,
                                        (unsigned long long)a.T};
    const unsigned int box[5] = {(unsigned)sh.U, (unsigned)K, 1u, BC, 1u};
    cudaError_t e = encode_tensor_map(&tmap, a.tape, 4, 5, dims, box);
    if (e != cudaSuccess) return e;
  }
  if (a.dstates) {
    const unsigned long long dims[5] = {(unsigned long long)a.D, (unsigned long long)a.N,
                                        (unsigned long long)a.T, (unsigned long long)a.B,
                                        (unsigned long long)S};
    const unsigned int box[5] = {(unsigned)sh.U, 1u, 1u, BC, (unsigned)S};
    cudaError_t e = encode_tensor_map(&dmap, a.dstates, 2, 5, dims, box);
    if (e != cudaSuccess) return e;
  } else {
    dmap = tmap;  // unused
  }
  (void)G;
  cudaError_t e = set_smem_attr((const void*)k, (size_t)sh.smem);
  if (e != cudaSuccess) return e;
  if (sh.C > 8) {
    e = set_nonportable_cluster((const void*)k);
    if (e != cudaSuccess) return e;
  }
  const int groups = a.N * ((a.B + (int)BC - 1) / (int)BC);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(groups * sh.C);
  cfg.blockDim = dim3(sh.warps * 32);
  cfg.dynamicSmemBytes = sh.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = sh.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, k, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  e = cudaLaunchKernelEx(&cfg, k, tmap, dmap, a);
  note_launch();
  return e;
}

// Clusters of the backward cluster kernel of shape `sh` that the current
// device holds at once, -1 if the device cannot be asked.
template <int FN>
int fused_bwd_capacity(const FusedShape& sh) {
  void (*k)(const CUtensorMap, const CUtensorMap, FusedArgs) = nullptr;
#define RNN_FUSED_BWD_PICK(NT_, MT_) \
  if (sh.NT == NT_ && sh.MT == MT_) k = fused_bwd_kernel<FN, NT_, MT_>;
  RNN_FUSED_BWD_PICK(1, 1) RNN_FUSED_BWD_PICK(1, 2) RNN_FUSED_BWD_PICK(2, 1) RNN_FUSED_BWD_PICK(2, 2)
#undef RNN_FUSED_BWD_PICK
  if (!k) return 0;
  return cluster_capacity_of((const void*)k, sh);
}

}  // namespace rnn
