// Persistent thread-block-cluster forward scan (bf16 storage, fp32 arithmetic).
//
// The "fused" design of the FlashRNN announcement (matrix product and
// pointwise cell in one kernel, recurrent weights kept in registers),
// re-planned for sm_103a:
//  - one cluster of C CTAs runs one head n for a group of up to BC = 8*NT batch
//    rows over the whole sequence; CTA c owns units [c*U, (c+1)*U), U = D/C;
//  - its slice of R (all G gates of its U units, all D inputs) lives in
//    registers as mma.sync A fragments for the whole kernel; the step's
//    contraction is the transposed product  rec^T[(g,j), b] = R[g,:,j]^T h[b,:],
//    M = G*U, N = batch, K = D, split over warps along M (16-unit groups) and K;
//  - h_{t-1} (bf16, all D units) sits in shared memory; after the pointwise
//    update every CTA pushes its U-slice of h_t into every peer's buffer with
//    one bulk copy (shared::cta -> shared::cluster) per peer, whose mbarrier
//    transaction count is the step's only synchronisation (no cluster-wide
//    barrier inside the time loop);
//  - Wx[:, t] for the CTA's slice streams in through a TMA ring NS steps ahead;
//  - the cell update runs in the epilogue with c, n, m carried in fp32 in
//    registers; states and the backward's tape are written straight out.
#pragma once
#include <cuda.h>

#include "kernels.cuh"
#include "grid_place.cuh"
#include "layout.h"
#include "ptx.cuh"

namespace rnn {

// GRIDX = true is the grid variant for R too large for one cluster: C CTAs of a
// cooperative launch share a head and batch group, and h_t goes through L2 (a
// bf16 exchange buffer plus a per-group step counter) instead of DSMEM.
template <int FN, int NT, int KT, bool ALLG, bool GRIDX>
__global__ void __launch_bounds__(256, 1)
    fused_fwd_kernel(const __grid_constant__ CUtensorMap wxmap, FusedArgs a) {
  constexpr int G = FnInfo<FN>::G, S = FnInfo<FN>::S, P = FnInfo<FN>::P, K = P + S;
  constexpr int BC = 8 * NT;
  const int C = a.C, U = a.U, D = a.D, KS = a.KS, TT = a.T, N = a.N, B = a.B;
  const int UP = U + 8;  // row stride (elements) of one source CTA's block of h
  // one h buffer: [C][BC][UP] blocks per source CTA in a cluster; the grid
  // variant gathers whole rows, [BC][D + 8] (one block, within the same space)
  const int RS = GRIDX ? D + 8 : UP;
  const int HB = GRIDX ? BC * (D + 8) : C * BC * UP;
  extern __shared__ __align__(128) unsigned char smem[];
  int2 place = make_int2((int)(blockIdx.x / C), 0);
  if constexpr (GRIDX) {
    place = grid_place(a, C, (int*)smem);
    if (place.x < 0) return;  // a spare CTA of a die-placed launch
  }
  const uint32_t rank = GRIDX ? (uint32_t)place.y : cluster_ctarank();
  const int grp = place.x;
  const int n = grp % N;
  const int b0 = (grp / N) * BC;
  const int nb = min(BC, B - b0);
  const int u0 = (int)rank * U;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  // warp -> (16-unit group mg, gate group gq of GW gates, K slice ks): GW
  // 16 x (8 NT) tiles over KT k-tiles; the KS partial tiles are summed in the
  // cell update
  constexpr int GW = ALLG ? G : 1, GQ = G / GW;
  // accumulator chains per tile (four where the registers allow)
  constexpr int CH = GW == 1 ? ((KT >= 4 && KT * NT <= 32) ? 4 : (KT >= 2 ? 2 : 1)) : 1;
  const int mg = warp / (GQ * KS), wrem = warp - mg * (GQ * KS);
  const int gq = wrem / KS, ks = wrem - gq * KS;

  const FusedSmem L = FusedSmem::make(G, S, D, U, BC, KS);
  uint64_t* bars = (uint64_t*)(smem + L.bars);  // [0,1]: h full; [2..]: Wx ring
  __nv_bfloat16* wxs = (__nv_bfloat16*)(smem + L.wx);
  __nv_bfloat16* hbuf = (__nv_bfloat16*)(smem + L.hbuf);
  float* red = (float*)(smem + L.red);
  __nv_bfloat16* stage = (__nv_bfloat16*)(smem + L.stage);
  const uint32_t full_bar0 = smem_u32(&bars[0]);
  const uint32_t wx_bar0 = smem_u32(&bars[2]);
  const uint32_t slice_bytes = (uint32_t)nb * UP * 2;  // one CTA's h slice, as sent
  const uint32_t hbytes = (uint32_t)C * slice_bytes;    // what a CTA receives per step
  const uint32_t wxbytes = (uint32_t)BC * G * U * 2;
  const size_t wx_stage_elems = (size_t)BC * G * U;

  const __nv_bfloat16* Wx = (const __nv_bfloat16*)a.Wx;
  const __nv_bfloat16* R = (const __nv_bfloat16*)a.R;
  const __nv_bfloat16* bias = (const __nv_bfloat16*)a.bias;
  const __nv_bfloat16* s0 = (const __nv_bfloat16*)a.s0;
  __nv_bfloat16* states = (__nv_bfloat16*)a.states;
  (void)Wx;

  // ---- prologue ------------------------------------------------------------
  if (tid == 0) {
    mbar_init(full_bar0, 1);
    mbar_init(full_bar0 + 8, 1);
    mbar_init(full_bar0 + 8 * (2 + FUSED_NS), 1);  // fault injection: nothing arrives on it
    for (int s = 0; s < FUSED_NS; ++s) mbar_init(wx_bar0 + 8 * s, 1);
    fence_mbar_init_cluster();
    prefetch_tensormap(&wxmap);
  }
  for (int e = tid; e < 2 * HB; e += nthr) hbuf[e] = __float2bfloat16_rn(0.0f);
  for (int e = tid; e < 2 * BC * UP; e += nthr) stage[e] = __float2bfloat16_rn(0.0f);
  __syncthreads();
  for (int e = tid; e < nb * D; e += nthr) {
    const int b = e / D, i = e - b * D, src = i / U;
    float v = s0 ? __bfloat162float(s0[((size_t)(b0 + b) * N + n) * D + i]) : 0.0f;
    hbuf[GRIDX ? b * RS + i : (src * BC + b) * UP + i - src * U] = __float2bfloat16_rn(v);
  }
  // Each thread owns the (batch row, unit) pairs e = tid + k * blockDim
  // (k < FUSED_PPT) for the whole sequence: their carried states (fp32) and
  // biases live in registers.
  // The pairs' (row, unit) coordinates are fixed for the kernel: divided
  // once here, not every step.
  float csr[FUSED_PPT][S], bsr[FUSED_PPT][G];
  int pb[FUSED_PPT], pu[FUSED_PPT];
#pragma unroll
  for (int k = 0; k < FUSED_PPT; ++k) {
    const int e = tid + k * nthr, b = e / U, u = e - b * U;
    pb[k] = b;
    pu[k] = u;
    const bool own = e < nb * U;
#pragma unroll
    for (int s = 0; s < S; ++s)
      csr[k][s] = (own && s0) ? __bfloat162float(s0[(((size_t)s * B + b0 + b) * N + n) * D + u0 + u]) : 0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g)
      bsr[k][g] = own ? __bfloat162float(bias[((size_t)g * N + n) * D + u0 + u]) : 0.0f;
  }

  // per pair, fixed for the kernel: the offset of its K-split partial sums
  // (k2 = 0, g = 0) in red, of its Wx in a ring stage, of its h in the grid's
  // exchange buffer, and its states / tape output pointers at t = 0 (advanced
  // by a fixed stride per step): no index arithmetic inside the time loop
  const int red_sk = G * BC * FUSED_RED_STRIDE;  // red stride of the K slice k2
  constexpr int RED_SG = BC * FUSED_RED_STRIDE;   // red stride of the gate g
  const int groups = N * ((B + BC - 1) / BC);
  const size_t hx_par = (size_t)groups * BC * D;  // grid exchange buffer stride of the step parity
  int red_off[FUSED_PPT], hx_off[FUSED_PPT];
  __nv_bfloat16* st_ptr[FUSED_PPT];
  float* tp_ptr[FUSED_PPT];
  const size_t st_sstride = (size_t)B * TT * N * D, tp_tstride = (size_t)B * N * K * D;
#pragma unroll
  for (int k = 0; k < FUSED_PPT; ++k) {
    const int b = pb[k], u = pu[k], bg = b0 + b, j = u0 + u;
    red_off[k] = (((u >> 4) * KS * G) * BC + b) * FUSED_RED_STRIDE + (u & 15);
    hx_off[k] = (grp * BC + b) * D + j;
    st_ptr[k] = states ? states + ((size_t)bg * TT) * N * D + (size_t)n * D + j : nullptr;
    tp_ptr[k] = a.tape ? a.tape + ((size_t)bg * N + n) * K * D + j : nullptr;
  }

  // the first k-tile of this warp's K slice: source block and column group
  // (the grid variant's one block holds all D inputs)
  const int U16 = GRIDX ? D / 16 : U / 16;
  const int ktile_sblk0 = (ks * KT) / U16, ktile_j0 = ks * KT - ktile_sblk0 * U16;

  // resident R fragments: A[m = unit j][k = input i] = R[g, n, i, j]. Warps
  // past the (U/16) * KS that the product needs only join the cell update.
  const bool mma_warp = warp < (U / 16) * GQ * KS;
  uint32_t afr[GW][KT][4];
  if (mma_warp) {
    const int jr = u0 + mg * 16 + (lane >> 2);
#pragma unroll
    for (int gi = 0; gi < GW; ++gi) {
      const __nv_bfloat16* Rg = R + (size_t)((gq * GW + gi) * N + n) * D * D;
#pragma unroll
      for (int kt = 0; kt < KT; ++kt) {
        const int k0 = (ks * KT + kt) * 16 + 2 * (lane & 3);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j = jr + ((q & 1) ? 8 : 0);
          const int k = k0 + ((q & 2) ? 8 : 0);
          afr[gi][kt][q] = pack_bf16(Rg[(size_t)k * D + j], Rg[(size_t)(k + 1) * D + j]);
        }
      }
    }
  }
  __syncthreads();
  if constexpr (!GRIDX) cluster_sync_all();  // every CTA's barriers are initialised before any peer signals them

  if (tid == 0) {
    if (!GRIDX && TT > 1) mbar_arrive_expect_tx(full_bar0 + 8, hbytes);  // step 1
    if (!GRIDX && TT > 2) mbar_arrive_expect_tx(full_bar0, hbytes);      // step 2
    for (int s = 0; s < FUSED_NS && s < TT; ++s) {
      mbar_arrive_expect_tx(wx_bar0 + 8 * s, wxbytes);
      tma_load_5d(smem_u32(wxs + s * wx_stage_elems), &wxmap, wx_bar0 + 8 * s, u0, n, 0, s, b0);
    }
  }

  bool failed = false;
  uint32_t ph0 = 0, ph1 = 0;
  // lane q of warp w sends this CTA's slice to the peer rank + w + q warps
  // (mod C), one bulk copy each: the copies of a step leave side by side, one
  // instruction per warp, rather than one after another. Each sender's
  // cluster addresses (the peer's h buffer and barrier, for both parities)
  // are fixed for the kernel.
  const int nwarps = nthr >> 5;
  const int my_c = warp + lane * nwarps;
  const bool sender = !GRIDX && lane < (C + nwarps - 1) / nwarps && my_c < C;
  uint32_t rdst0 = 0, rdst1 = 0, rbar0 = 0, rbar1 = 0;
  if (sender) {
    int peer = (int)rank + my_c;
    if (peer >= C) peer -= C;
    rdst0 = mapa_shared(smem_u32(hbuf + (size_t)rank * BC * UP), (uint32_t)peer);
    rdst1 = mapa_shared(smem_u32(hbuf + HB + (size_t)rank * BC * UP), (uint32_t)peer);
    rbar0 = mapa_shared(full_bar0, (uint32_t)peer);
    rbar1 = mapa_shared(full_bar0 + 8, (uint32_t)peer);
  }

  float prk[FUSED_PPT][P];  // pre-activations kept for the tape, written after the exchange
  // the states and tape of a step, off the exchange's critical path
  auto store_pair_outputs = [&]() {
#pragma unroll
    for (int kp = 0; kp < FUSED_PPT; ++kp) {
      const int e = tid + kp * nthr;
      if (e >= nb * U) break;
      if (st_ptr[kp]) {
#pragma unroll
        for (int s = 0; s < S; ++s) st_ptr[kp][s * st_sstride] = __float2bfloat16_rn(csr[kp][s]);
        st_ptr[kp] += (size_t)N * D;
      }
      if (tp_ptr[kp]) {
        float* tp = tp_ptr[kp];
#pragma unroll
        for (int k2 = 0; k2 < P; ++k2) tp[k2 * D] = prk[kp][k2];
#pragma unroll
        for (int s = 0; s < S; ++s) tp[(P + s) * D] = csr[kp][s];
        tp_ptr[kp] += tp_tstride;
      }
    }
  };
  // the grid variant's thread 0 observes the step counter: it writes its own
  // pairs' states and tape of step t - 1 after issuing step t's pull
  const bool defer_stores = GRIDX && tid == 0;

  const bool tracer = a.trace && grp == 0 && rank == 0 && tid == 0;
#define RNN_TRACE(k)                                                                    \
  if (tracer && t >= a.trace_t0 && t < a.trace_t0 + a.trace_steps)                      \
    a.trace[(size_t)(t - a.trace_t0) * 16 + (k)] = (unsigned long long)clock64();

  // ---- time loop -------------------------------------------------------------
  for (int t = 0; t < TT; ++t) {
    const int p = t & 1;
    RNN_TRACE(0)
    if (t > 0) {
      if constexpr (GRIDX) {
        // every CTA of the group published h_{t-1}: one thread observes the
        // step counter and pulls the nb rows from L2 with one bulk copy each;
        // every thread waits for the bytes
        if (tid == 0) {
          counter_wait_bounded(group_counter(a, grp), (unsigned)(C * t), a.wait_limit_ns, a.status, failed);
          if (!failed) {
            const __nv_bfloat16* src = (const __nv_bfloat16*)a.hx + p * hx_par + (size_t)grp * BC * D;
            fence_proxy_async_global();  // the peers' stores, acquired above, before the bulk reads
            fence_proxy_async_smem();    // the last reads of this buffer (ordered by the barrier) before the writes
            mbar_arrive_expect_tx(full_bar0, (uint32_t)(nb * D * 2));
            for (int b = 0; b < nb; ++b)
              bulk_load_global(smem_u32(hbuf + p * HB + b * RS), src + (size_t)b * D, (uint32_t)(D * 2), full_bar0);
          }
          store_pair_outputs();  // step t - 1's, while the rows are in flight
        }
        mbar_wait_bounded<false>(full_bar0, ph0, a.wait_limit_ns, a.status, failed);
        ph0 ^= 1u;
      } else {
        const uint32_t par = p ? ph1 : ph0;
        mbar_wait_bounded(full_bar0 + 8 * p, par, a.wait_limit_ns, a.status, failed);
        if (p) ph1 ^= 1; else ph0 ^= 1;
        if (tid == 0 && t + 2 <= TT - 1) mbar_arrive_expect_tx(full_bar0 + 8 * p, hbytes);
      }
    }
    RNN_TRACE(1)
    const int ws = t % FUSED_NS;
    // Wx[:, t] (loaded NS - 1 steps ahead): one thread observes the TMA
    // completion; the barrier after the product orders it for every thread
    if (tid == nthr - 1)
      mbar_wait_bounded<false>(wx_bar0 + 8 * ws, (t / FUSED_NS) & 1, a.wait_limit_ns, a.status, failed);
    if (t == a.inject_step && grp == 0 && rank == 0) {
      // injected fault: a wait that nothing ends runs out and records
      // STATUS_TIMEOUT; the exchange protocol itself is left untouched
      bool inj_failed = false;
      mbar_wait_bounded<false>(full_bar0 + 8 * (2 + FUSED_NS), 0, a.inject_limit_ns, a.status, inj_failed);
    }

    // rec^T = R_slice^T h_{t-1}: this warp's gate tile over KT k-tiles, in
    // CH accumulator chains (k-tile kt feeds chain kt % CH) to shorten the
    // dependent MMA sequence
    if (mma_warp) {
    float acc[GW][CH][NT][4];
#pragma unroll
    for (int gi = 0; gi < GW; ++gi)
#pragma unroll
      for (int c2 = 0; c2 < CH; ++c2)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[gi][c2][nt][q] = 0.0f;
    const uint32_t hb = smem_u32(hbuf + p * HB);
    // k-tile kt holds inputs 16 (ks KT + kt) .. + 15, in the block of source
    // CTA sblk at column 16 jj; both advance without a division
    int sblk = ktile_sblk0, jj = ktile_j0;
#pragma unroll
    for (int kt = 0; kt < KT; ++kt) {
      const uint32_t blk = hb + (uint32_t)((sblk * BC * UP + 16 * jj) * 2);
      if (++jj == U16) {
        jj = 0;
        ++sblk;
      }
      uint32_t bf[NT][2];
      if constexpr (NT == 1) {
        const uint32_t addr = blk + (uint32_t)(((lane & 7) * RS + ((lane >> 3) & 1) * 8) * 2);
        ldmatrix_x2(addr, bf[0][0], bf[0][1]);
      } else {
#pragma unroll
        for (int np = 0; np < NT; np += 2) {
          const int q = lane >> 3;
          const uint32_t addr = blk + (uint32_t)((((np + (q >> 1)) * 8 + (lane & 7)) * RS + (q & 1) * 8) * 2);
          ldmatrix_x4(addr, bf[np][0], bf[np][1], bf[np + 1][0], bf[np + 1][1]);
        }
      }
#pragma unroll
      for (int gi = 0; gi < GW; ++gi)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma_bf16_16816(acc[gi][kt % CH][nt], afr[gi][kt], bf[nt][0], bf[nt][1]);
    }
    {
      const int r = lane >> 2, bc = 2 * (lane & 3);
#pragma unroll
      for (int gi = 0; gi < GW; ++gi) {
        float* rp = red + ((mg * KS + ks) * G + gq * GW + gi) * BC * FUSED_RED_STRIDE;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if constexpr (CH == 4)
              v[q] = (acc[gi][0][nt][q] + acc[gi][1][nt][q]) + (acc[gi][2][nt][q] + acc[gi][3][nt][q]);
            else if constexpr (CH == 2)
              v[q] = acc[gi][0][nt][q] + acc[gi][1][nt][q];
            else
              v[q] = acc[gi][0][nt][q];
          }
          const int b = nt * 8 + bc;
          rp[b * FUSED_RED_STRIDE + r] = v[0];
          rp[(b + 1) * FUSED_RED_STRIDE + r] = v[1];
          rp[b * FUSED_RED_STRIDE + r + 8] = v[2];
          rp[(b + 1) * FUSED_RED_STRIDE + r + 8] = v[3];
        }
      }
    }
    }  // mma_warp
    RNN_TRACE(2)
    __syncthreads();
    RNN_TRACE(3)

    // ---- epilogue: gate assembly and cell update, one (batch row, unit) pair per thread
    const __nv_bfloat16* wxt = wxs + ws * wx_stage_elems;
    RNN_TRACE(4)
#pragma unroll
    for (int kp = 0; kp < FUSED_PPT; ++kp) {
      const int e = tid + kp * nthr;
      if (e >= nb * U) break;
      const int u = pu[kp];
      float x[G], rc[G], sn[S], pre[P];
      // all K-split partials are loaded before any is summed (independent loads)
      float part[G][FUSED_MAX_KS];
      const float* rp = red + red_off[kp];
#pragma unroll
      for (int k2 = 0; k2 < FUSED_MAX_KS; ++k2) {
#pragma unroll
        for (int g = 0; g < G; ++g) part[g][k2] = k2 < KS ? rp[g * RED_SG] : 0.0f;
        rp += red_sk;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float v = bsr[kp][g];
#pragma unroll
        for (int k2 = 0; k2 < FUSED_MAX_KS; ++k2) v += part[g][k2];
        rc[g] = v;
        x[g] = __bfloat162float(wxt[(pb[kp] * G + g) * U + u]);
      }
      cell_fwd<FN, true>(x, rc, csr[kp], sn, pre);
#pragma unroll
      for (int s = 0; s < S; ++s) csr[kp][s] = sn[s];
#pragma unroll
      for (int k2 = 0; k2 < P; ++k2) prk[kp][k2] = pre[k2];
      if constexpr (GRIDX) {
        if (t + 1 < TT)
          ((__nv_bfloat16*)a.hx)[(size_t)hx_off[kp] + (p ^ 1) * hx_par] = __float2bfloat16_rn(sn[0]);
      } else {
        stage[(p * BC + pb[kp]) * UP + u] = __float2bfloat16_rn(sn[0]);
      }
    }
    RNN_TRACE(5)
    if constexpr (!GRIDX) fence_proxy_async_smem();  // the staged slice is read by bulk copies
    __syncthreads();
    RNN_TRACE(6)

    // ---- exchange: push this CTA's slice of h_t into every CTA's next buffer.
    // The staged slice stage[p] is not rewritten before step t + 2, whose wait
    // needs every peer's h_{t+1}, which in turn needed this step's copies to
    // have landed (so their reads of stage[p] are over).
    if (GRIDX) {
      if (t + 1 < TT && tid == 0) counter_publish(group_counter(a, grp));
    } else if (t + 1 < TT && sender) {  // into the peer's buffer p ^ 1
      bulk_copy_to_peer(p ? rdst0 : rdst1, smem_u32(stage + p * BC * UP), slice_bytes, p ? rbar0 : rbar1);
    }
    RNN_TRACE(7)
    // Wx[:, t + NS] into the ring slot this step's update has finished reading
    if (tid == nthr - 32 && t + FUSED_NS < TT) {
      const int ts = t + FUSED_NS;
      mbar_arrive_expect_tx(wx_bar0 + 8 * ws, wxbytes);
      tma_load_5d(smem_u32(wxs + ws * wx_stage_elems), &wxmap, wx_bar0 + 8 * ws, u0, n, 0, ts, b0);
    }
    // states and tape of this step (thread 0 of the grid variant: at the next
    // step, after its pull is issued)
    if (!defer_stores || t + 1 == TT) store_pair_outputs();
    RNN_TRACE(11)
  }
#undef RNN_TRACE

  // ---- epilogue of the sequence ---------------------------------------------
  if (a.last) {
    __nv_bfloat16* last = (__nv_bfloat16*)a.last;
#pragma unroll
    for (int kp = 0; kp < FUSED_PPT; ++kp) {
      const int e = tid + kp * nthr;
      if (e >= nb * U) break;
      const int b = e / U, u = e - b * U;
#pragma unroll
      for (int s = 0; s < S; ++s)
        last[(((size_t)s * B + b0 + b) * N + n) * D + u0 + u] = __float2bfloat16_rn(csr[kp][s]);
    }
  }
  __syncthreads();
  if constexpr (!GRIDX) cluster_sync_all();  // no CTA leaves while a peer may still write into its shared memory
}

// Host launcher for one cell type; the TMA descriptor covers Wx as the 5-D
// tensor (D, N, G, T, B) with a (U, 1, G, 1, BC) box. GRIDX selects the
// cooperative grid variant (no cluster; co-residency guaranteed by the launch).
template <int FN, bool GRIDX>
cudaError_t fwd_launch(const FusedShape& sh, const FusedArgs& a, cudaStream_t st) {
  constexpr int G = FnInfo<FN>::G;
  void (*k)(const CUtensorMap, FusedArgs) = nullptr;
#define RNN_FUSED_PICK(NT_, KT_, AG_) \
  if (sh.NT == NT_ && sh.KT == KT_ && sh.allg == AG_) k = fused_fwd_kernel<FN, NT_, KT_, AG_, GRIDX>;
  if constexpr (GRIDX) {
    RNN_FUSED_PICK(1, 8, false) RNN_FUSED_PICK(1, 16, false) RNN_FUSED_PICK(1, 32, false)
    RNN_FUSED_PICK(2, 8, false) RNN_FUSED_PICK(2, 16, false) RNN_FUSED_PICK(2, 32, false)
  } else {
    // one gate per warp (long K per warp, few partial sums) ...
    RNN_FUSED_PICK(1, 4, false) RNN_FUSED_PICK(1, 6, false) RNN_FUSED_PICK(1, 8, false)
    RNN_FUSED_PICK(1, 12, false) RNN_FUSED_PICK(1, 16, false)
    // ... or all G gates per warp (wide slices, short K per warp)
    RNN_FUSED_PICK(1, 2, true) RNN_FUSED_PICK(1, 3, true) RNN_FUSED_PICK(1, 4, true)
    RNN_FUSED_PICK(2, 2, true) RNN_FUSED_PICK(2, 3, true) RNN_FUSED_PICK(2, 4, true)
  }
#undef RNN_FUSED_PICK
  if (!k) return cudaErrorInvalidValue;
  CUtensorMap map;
  const unsigned long long dims[5] = {(unsigned long long)a.D, (unsigned long long)a.N,
                                      (unsigned long long)G, (unsigned long long)a.T,
                                      (unsigned long long)a.B};
  const unsigned int box[5] = {(unsigned)sh.U, 1u, (unsigned)G, 1u, (unsigned)(8 * sh.NT)};
  cudaError_t e = encode_tensor_map_bf16(&map, a.Wx, 5, dims, box);
  if (e != cudaSuccess) return e;
  e = set_smem_attr((const void*)k, (size_t)sh.smem);
  if (e != cudaSuccess) return e;
  if (!GRIDX && sh.C > 8) {
    e = set_nonportable_cluster((const void*)k);
    if (e != cudaSuccess) return e;
  }
  const int groups = a.N * ((a.B + 8 * sh.NT - 1) / (8 * sh.NT));
  FusedArgs args = a;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(groups * sh.C);
  cfg.blockDim = dim3(sh.warps * 32);
  cfg.dynamicSmemBytes = sh.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (GRIDX) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    int per_sm = 0, dev = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, (int)cfg.blockDim.x, sh.smem);
    if (e != cudaSuccess) return e;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (per_sm * sms < groups * sh.C) return cudaErrorCooperativeLaunchTooLarge;
    // die placement holds one CTA per SM, so that each die's ticket counts
    // exactly its SMs; otherwise groups by block index
    if (args.die_of_sm && per_sm == 1 && args.launch_ctas == sms) cfg.gridDim = dim3(sms);
    else args.die_of_sm = nullptr;
  } else {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = sh.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!GRIDX) {
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, k, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
  }
  e = cudaLaunchKernelEx(&cfg, k, map, args);
  note_launch();
  return e;
}

template <int FN>
cudaError_t fused_fwd_launch(const FusedShape& sh, const FusedArgs& a, cudaStream_t st) {
  return fwd_launch<FN, false>(sh, a, st);
}

// Clusters of the forward cluster kernel of shape `sh` that the current device
// holds at once (cudaOccupancyMaxActiveClusters), -1 if the device cannot be
// asked. The planner's co-residency constraint.
template <int FN>
int fused_fwd_capacity(const FusedShape& sh) {
  void (*k)(const CUtensorMap, FusedArgs) = nullptr;
#define RNN_FUSED_PICK(NT_, KT_, AG_) \
  if (sh.NT == NT_ && sh.KT == KT_ && sh.allg == AG_) k = fused_fwd_kernel<FN, NT_, KT_, AG_, false>;
  RNN_FUSED_PICK(1, 4, false) RNN_FUSED_PICK(1, 6, false) RNN_FUSED_PICK(1, 8, false)
  RNN_FUSED_PICK(1, 12, false) RNN_FUSED_PICK(1, 16, false)
  RNN_FUSED_PICK(1, 2, true) RNN_FUSED_PICK(1, 3, true) RNN_FUSED_PICK(1, 4, true)
  RNN_FUSED_PICK(2, 2, true) RNN_FUSED_PICK(2, 3, true) RNN_FUSED_PICK(2, 4, true)
#undef RNN_FUSED_PICK
  if (!k) return 0;
  return cluster_capacity_of((const void*)k, sh);
}
template <int FN>
cudaError_t grid_fwd_launch(const FusedShape& sh, const FusedArgs& a, cudaStream_t st) {
  return fwd_launch<FN, true>(sh, a, st);
}

}  // namespace rnn
