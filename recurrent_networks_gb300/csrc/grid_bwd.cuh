// Persistent cooperative-grid backward scan for R too large for one cluster
// (bf16 storage, fp32 arithmetic).
//
// C CTAs of one cooperative launch share a head and batch group; CTA c owns
// units [c*U, (c+1)*U) and keeps R[g, n, i, :] for its rows i (all gates, all
// columns j) as mma.sync A fragments in registers. Per step, from t = T-1
// down to 0:
//   1. wait until every CTA of the group published dr_{t+1} (a per-group step
//      counter in global memory) and copy all of it (bf16, B x G*D) from L2;
//   2. dh^rec_t[b, i] = sum_{g, j} R[g, n, i, j] dr_{t+1}[b, g, j] for the own
//      rows i: M = U, N = batch, K = G*D split over the warps, reduced in
//      shared memory;
//   3. the cell derivative (tape[t], dstates[:, t] from a TMA ring) gives dWx,
//      the recurrent-branch gradient dr_t (written for the weight gradients
//      and published to L2 for the other CTAs) and the carried gradients.
// A last gather-and-multiply after t = 0 yields dstates0.
#pragma once
#include <cuda.h>

#include "kernels.cuh"
#include "dr_beside.cuh"
#include "grid_place.cuh"
#include "layout.h"
#include "ptx.cuh"

namespace rnn {

template <int FN, int NT, int KT>
__global__ void __launch_bounds__(256, 1)
    grid_bwd_kernel(const __grid_constant__ CUtensorMap tapemap, const __grid_constant__ CUtensorMap dstmap,
                    FusedArgs a, const __grid_constant__ UmmaMaps dmaps) {
  constexpr int G = FnInfo<FN>::G, S = FnInfo<FN>::S, P = FnInfo<FN>::P, K = P + S;
  constexpr int BC = 8 * NT;
  const int C = a.C, U = a.U, D = a.D, KS = a.KS, TT = a.T, N = a.N, B = a.B;
  const int KG = G * D, KB = KG + 8;
  extern __shared__ __align__(128) unsigned char smem[];
  const int2 place = grid_place(a, C, (int*)smem);
  if (place.x < 0) {  // a spare CTA: dR beside the scan, when asked for
    dr_beside(a, dmaps, G, smem);
    return;
  }
  const int rank = place.y, grp = place.x, groups = N * ((B + BC - 1) / BC);
  const int n = grp % N;
  const int b0 = (grp / N) * BC;
  const int nb = min(BC, B - b0);
  const int u0 = rank * U;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int mg = warp / KS, ks = warp - mg * KS;

  const GridBwdSmem L = GridBwdSmem::make(G, S, K, D, U, BC, KS);
  uint64_t* bars = (uint64_t*)(smem + L.bars);
  unsigned char* ring = smem + L.ring;
  __nv_bfloat16* dbuf = (__nv_bfloat16*)(smem + L.dbuf);  // [BC][KB]
  float* red = (float*)(smem + L.red);
  float* ds = (float*)(smem + L.ds);
  float* s0s = (float*)(smem + L.s0);
  float* dbs = (float*)(smem + L.dbs);  // [G][BC][U]: the pairs' sums of dr over the steps
  const bool with_db = a.dbp != nullptr;
  const uint32_t ring_bar0 = smem_u32(&bars[0]);
  const uint32_t gath_bar = smem_u32(&bars[FUSED_NS]);  // the gather of the group's dr
  const bool has_dst = a.dstates != nullptr;
  const uint32_t stage_bytes = (uint32_t)(L.tape_bytes + (has_dst ? (size_t)S * BC * U * 2 : 0));

  const __nv_bfloat16* R = (const __nv_bfloat16*)a.R;
  const __nv_bfloat16* s0 = (const __nv_bfloat16*)a.s0;
  const __nv_bfloat16* dlast = (const __nv_bfloat16*)a.dlast;
  __nv_bfloat16* dWx = (__nv_bfloat16*)a.dWx;
  __nv_bfloat16* dro = (__nv_bfloat16*)a.dr;
  __nv_bfloat16* dx = (__nv_bfloat16*)a.hx;  // [2][groups][BC][G*D]
  const bool write_dr = dro && (FN == GRU || (void*)dro != (void*)dWx);

  if (tid == 0) {
    for (int s = 0; s < FUSED_NS; ++s) mbar_init(ring_bar0 + 8 * s, 1);
    mbar_init(gath_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tensormap(&tapemap);
    if (has_dst) prefetch_tensormap(&dstmap);
  }
  for (int e = tid; e < BC * KB; e += nthr) dbuf[e] = __float2bfloat16_rn(0.0f);
  for (int e = tid; e < S * BC * U; e += nthr) {
    const int s = e / (BC * U), r = e - s * BC * U, b = r / U, u = r - b * U;
    float v = 0.0f;
    if (b < nb && s0) v = __bfloat162float(s0[(((size_t)s * B + b0 + b) * N + n) * D + u0 + u]);
    s0s[e] = v;
    ds[e] = 0.0f;
  }
  if (with_db)
    for (int e = tid; e < G * BC * U; e += nthr) dbs[e] = 0.0f;
  // resident fragments: A[m = own row i][k = (g, j)] = R[g, n, i, j]
  uint32_t afr[KT][4];
  {
    const int ir = u0 + mg * 16 + (lane >> 2);
#pragma unroll
    for (int kt = 0; kt < KT; ++kt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = ir + ((q & 1) ? 8 : 0);
        const int k = (ks * KT + kt) * 16 + 2 * (lane & 3) + ((q & 2) ? 8 : 0);
        const int g = k / D, j = k - g * D;
        afr[kt][q] = *(const uint32_t*)(R + ((size_t)(g * N + n) * D + i) * D + j);
      }
  }
  __syncthreads();

  // per-thread starting coordinates and strides of the per-step cell loop
  // over the pairs e = b U + u
  const int c_b0 = tid / U, c_u0 = tid - c_b0 * U, c_db = nthr / U, c_du = nthr - c_db * U;
  uint32_t gath_par = 0u;
  // the thread's first pair, fixed for the kernel: the offset of its K-split
  // partial sums in red and of its gradients in dWx / dr at t = 0 (a step
  // moves them by G N D): no index arithmetic in the time loop for it
  const int red_off0 = ((c_u0 >> 4) * KS * BC + c_b0) * FUSED_RED_STRIDE + (c_u0 & 15);
  const int red_sk = BC * FUSED_RED_STRIDE;
  const size_t o_first = ((size_t)(b0 + c_b0) * TT * G) * N * D + (size_t)n * D + u0 + c_u0;
  const size_t o_step = (size_t)G * N * D;

  auto issue_stage = [&](int k) {
    const int t = TT - 1 - k, s = k % FUSED_NS;
    unsigned char* st = ring + (size_t)s * L.ring_stage;
    mbar_arrive_expect_tx(ring_bar0 + 8 * s, stage_bytes);
    tma_load_5d(smem_u32(st), &tapemap, ring_bar0 + 8 * s, u0, 0, n, b0, t);
    if (has_dst) tma_load_5d(smem_u32(st + L.dst_off), &dstmap, ring_bar0 + 8 * s, u0, n, t, b0, 0);
  };
  if (tid == 0)
    for (int k = 0; k < FUSED_NS - 1 && k < TT; ++k) issue_stage(k);

  bool failed = false;
  float dbv[G];  // the first pair's dr of the step, for db
  const bool tracer = a.trace && grp == 0 && rank == 0 && tid == 0;
#define RNN_TRACE(p)                                                                    \
  if (tracer && kk >= a.trace_t0 && kk < a.trace_t0 + a.trace_steps)                    \
    a.trace[(size_t)(kk - a.trace_t0) * 16 + (p)] = (unsigned long long)clock64();
  for (int kk = 0; kk <= TT; ++kk) {
    const int t = TT - 1 - kk;
    const bool have_rec = kk > 0;
    RNN_TRACE(0)
    const int sc = kk % FUSED_NS, sn_ = (kk + 1) % FUSED_NS;
    const float* tp = (const float*)(ring + (size_t)sc * L.ring_stage);
    const __nv_bfloat16* dstage = (const __nv_bfloat16*)(ring + (size_t)sc * L.ring_stage + L.dst_off);
    const float* tq = (const float*)(ring + (size_t)sn_ * L.ring_stage);
    // The first pair's tape, upstream gradients and gate activations do not
    // depend on dh: evaluated while the step counter and the gathered dr are
    // still outstanding (thread 0 after issuing the gather).
    float f_pre[P], f_sp[S], f_dsn[S], f_act[CELL_BWD_ACT];
    auto first_pair_inputs = [&]() {
      if (kk < TT && tid < nb * U) {
        mbar_wait_bounded<false>(ring_bar0 + 8 * sc, (kk / FUSED_NS) & 1, a.wait_limit_ns, a.status, failed);
        if (t > 0)
          mbar_wait_bounded<false>(ring_bar0 + 8 * sn_, ((kk + 1) / FUSED_NS) & 1, a.wait_limit_ns, a.status,
                                   failed);
        const int b = c_b0, u = c_u0;
        float f_sn[S];
#pragma unroll
        for (int k2 = 0; k2 < P; ++k2) f_pre[k2] = tp[(b * K + k2) * U + u];
#pragma unroll
        for (int s = 0; s < S; ++s) {
          f_sn[s] = tp[(b * K + P + s) * U + u];
          f_sp[s] = t > 0 ? tq[(b * K + P + s) * U + u] : s0s[(s * BC + b) * U + u];
          float d = ds[(s * BC + b) * U + u];
          if (has_dst) d += __bfloat162float(dstage[(s * BC + b) * U + u]);
          if (dlast && t == TT - 1) d += __bfloat162float(dlast[(((size_t)s * B + b0 + b) * N + n) * D + u0 + u]);
          f_dsn[s] = d;
        }
        cell_bwd_act<FN, true>(f_pre, f_sp, f_sn, f_act);
      }
    };
    if (!have_rec) first_pair_inputs();
    if (have_rec) {
      // gather dr_{t+1} of the whole group, multiply by the resident rows of R
      // one thread observes the group's step counter, then pulls the nb rows
      // of dr (G D bf16 each) with one bulk copy per row; every thread waits
      // for the bytes on the gather barrier
      if (tid == 0) {
        counter_wait_bounded(group_counter(a, grp), (unsigned)(C * kk), a.wait_limit_ns, a.status, failed);
        if (!failed) {
          const __nv_bfloat16* src = dx + ((size_t)((kk - 1) & 1) * groups + grp) * BC * KG;
          fence_proxy_async_global();  // the peers' stores, acquired above, before the bulk reads
          fence_proxy_async_smem();    // the last step's reads of dbuf (ordered by the barrier) before the writes
          mbar_arrive_expect_tx(gath_bar, (uint32_t)(nb * KG * 2));
          for (int b = 0; b < nb; ++b)
            bulk_load_global(smem_u32(dbuf + b * KB), src + (size_t)b * KG, (uint32_t)(KG * 2), gath_bar);
        }
      }
      RNN_TRACE(1)
      first_pair_inputs();
      mbar_wait_bounded<false>(gath_bar, gath_par, a.wait_limit_ns, a.status, failed);
      gath_par ^= 1u;
      RNN_TRACE(2)
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[nt][q] = 0.0f;
      const uint32_t hb = smem_u32(dbuf);
#pragma unroll
      for (int kt = 0; kt < KT; ++kt) {
        const int k0 = (ks * KT + kt) * 16;
        uint32_t bf[NT][2];
        if constexpr (NT == 1) {
          ldmatrix_x2(hb + (uint32_t)(((lane & 7) * KB + k0 + ((lane >> 3) & 1) * 8) * 2), bf[0][0], bf[0][1]);
        } else {
#pragma unroll
          for (int np = 0; np < NT; np += 2) {
            const int q = lane >> 3;
            ldmatrix_x4(hb + (uint32_t)((((np + (q >> 1)) * 8 + (lane & 7)) * KB + k0 + (q & 1) * 8) * 2),
                        bf[np][0], bf[np][1], bf[np + 1][0], bf[np + 1][1]);
          }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[nt], afr[kt], bf[nt][0], bf[nt][1]);
      }
      {
        const int r = lane >> 2, bc = 2 * (lane & 3);
        float* rp = red + (size_t)(mg * KS + ks) * BC * FUSED_RED_STRIDE;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int b = nt * 8 + bc;
          rp[b * FUSED_RED_STRIDE + r] = acc[nt][0];
          rp[(b + 1) * FUSED_RED_STRIDE + r] = acc[nt][1];
          rp[b * FUSED_RED_STRIDE + r + 8] = acc[nt][2];
          rp[(b + 1) * FUSED_RED_STRIDE + r + 8] = acc[nt][3];
        }
      }
      __syncthreads();
      RNN_TRACE(3)
    }

    if (kk == TT) {  // dstates0 = carried gradients after step 0
      __nv_bfloat16* ds0 = (__nv_bfloat16*)a.ds0;
      if (ds0)
        for (int e = tid; e < nb * U; e += nthr) {
          const int b = e / U, u = e - b * U, q = u >> 4, r = u & 15;
#pragma unroll
          for (int s = 0; s < S; ++s) {
            float v = ds[(s * BC + b) * U + u];
            if (s == 0 && have_rec)
              for (int k2 = 0; k2 < KS; ++k2) v += red[((size_t)(q * KS + k2) * BC + b) * FUSED_RED_STRIDE + r];
            ds0[(((size_t)s * B + b0 + b) * N + n) * D + u0 + u] = __float2bfloat16_rn(v);
          }
        }
      break;
    }

    // ---- the cell derivative of step t -----------------------------------------
    if (tid == 0 && kk + FUSED_NS - 1 < TT) issue_stage(kk + FUSED_NS - 1);
    RNN_TRACE(4)
    __nv_bfloat16* dxw = dx + ((size_t)(kk & 1) * groups + grp) * BC * KG;
    // pair e = b U + u, stepped without a division
    for (int e = tid, b = c_b0, u = c_u0; e < nb * U; e += nthr, b += c_db + (u + c_du >= U), u = u + c_du >= U ? u + c_du - U : u + c_du) {
      const bool first = e == tid;
      float pre[P], sp[S], sn[S], dsn[S], dxg[G], dr[G], dsp[S], act[CELL_BWD_ACT];
      if (first) {  // evaluated at the start of the step
#pragma unroll
        for (int k2 = 0; k2 < P; ++k2) pre[k2] = f_pre[k2];
#pragma unroll
        for (int s = 0; s < S; ++s) sp[s] = f_sp[s], dsn[s] = f_dsn[s];
#pragma unroll
        for (int k2 = 0; k2 < CELL_BWD_ACT; ++k2) act[k2] = f_act[k2];
      } else {
#pragma unroll
        for (int k2 = 0; k2 < P; ++k2) pre[k2] = tp[(b * K + k2) * U + u];
#pragma unroll
        for (int s = 0; s < S; ++s) {
          sn[s] = tp[(b * K + P + s) * U + u];
          sp[s] = t > 0 ? tq[(b * K + P + s) * U + u] : s0s[(s * BC + b) * U + u];
          float d = ds[(s * BC + b) * U + u];
          if (has_dst) d += __bfloat162float(dstage[(s * BC + b) * U + u]);
          if (dlast && t == TT - 1) d += __bfloat162float(dlast[(((size_t)s * B + b0 + b) * N + n) * D + u0 + u]);
          dsn[s] = d;
        }
        cell_bwd_act<FN, true>(pre, sp, sn, act);
      }
      if (have_rec) {  // the K-split partials, loaded together
        float part[FUSED_MAX_KS];
        const float* rp = red + (first ? red_off0 : (((u >> 4) * KS * BC + b) * FUSED_RED_STRIDE + (u & 15)));
#pragma unroll
        for (int k2 = 0; k2 < FUSED_MAX_KS; ++k2) part[k2] = k2 < KS ? rp[k2 * red_sk] : 0.0f;
#pragma unroll
        for (int k2 = 0; k2 < FUSED_MAX_KS; ++k2) dsn[0] += part[k2];
      }
      cell_bwd_grad<FN, true>(act, pre, sp, dsn, dxg, dr, dsp);
      const size_t o = first ? o_first + (size_t)t * o_step
                             : (((size_t)(b0 + b) * TT + t) * G) * N * D + (size_t)n * D + u0 + u;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (dWx) dWx[o + (size_t)g * N * D] = __float2bfloat16_rn(dxg[g]);
        if (write_dr) dro[o + (size_t)g * N * D] = __float2bfloat16_rn(dr[g]);
        dxw[(size_t)b * KG + g * D + u0 + u] = __float2bfloat16_rn(dr[g]);
      }
      // db: the pair's own running sum (the pair stays with this thread); the
      // first pair's is added after the step is published, off the step's path
      if (with_db) {
        if (first) {
#pragma unroll
          for (int g = 0; g < G; ++g) dbv[g] = dr[g];
        } else {
#pragma unroll
          for (int g = 0; g < G; ++g) dbs[(g * BC + b) * U + u] += dr[g];
        }
      }
#pragma unroll
      for (int s = 0; s < S; ++s) ds[(s * BC + b) * U + u] = dsp[s];
    }
    RNN_TRACE(5)
    __syncthreads();
    if (tid == 0) counter_publish(group_counter(a, grp));
    RNN_TRACE(6)
    if (with_db && tid < nb * U)
#pragma unroll
      for (int g = 0; g < G; ++g) dbs[(g * BC + c_b0) * U + c_u0] += dbv[g];
  }
#undef RNN_TRACE
  // db partial of the batch block: the column sums over its rows, in row order
  // (every pair's last update was ordered before the last step's barrier)
  if (with_db)
    for (int e = tid; e < G * U; e += nthr) {
      const int g = e / U, u = e - g * U;
      float v = 0.0f;
      for (int b = 0; b < nb; ++b) v += dbs[(g * BC + b) * U + u];
      a.dbp[(((size_t)(grp / N) * G + g) * N + n) * D + u0 + u] = v;
    }
  if (a.drw.nc > 0) {  // the scan is over: take the dR units still left
    __syncthreads();   // every thread is done with the shared memory the worker reuses
    dr_beside(a, dmaps, G, smem);
  }
}

// dmaps: the dR operand maps when a.drw.nc > 0 (dR beside the scan, which
// needs one CTA per SM: cudaErrorNotSupported, before any launch, otherwise).
template <int FN>
cudaError_t grid_bwd_launch(const FusedShape& sh, const FusedArgs& a, cudaStream_t st, const UmmaMaps* dmaps) {
  constexpr int S = FnInfo<FN>::S, K = FnInfo<FN>::P + FnInfo<FN>::S;
  void (*k)(const CUtensorMap, const CUtensorMap, FusedArgs, const UmmaMaps) = nullptr;
#define RNN_GRID_BWD_PICK(NT_, KT_) \
  if (sh.NT == NT_ && sh.KT == KT_) k = grid_bwd_kernel<FN, NT_, KT_>;
  RNN_GRID_BWD_PICK(1, 8) RNN_GRID_BWD_PICK(1, 16) RNN_GRID_BWD_PICK(1, 24) RNN_GRID_BWD_PICK(1, 32)
  RNN_GRID_BWD_PICK(2, 8) RNN_GRID_BWD_PICK(2, 16) RNN_GRID_BWD_PICK(2, 24) RNN_GRID_BWD_PICK(2, 32)
#undef RNN_GRID_BWD_PICK
  if (!k) return cudaErrorInvalidValue;
  const unsigned BC = 8u * sh.NT;
  CUtensorMap tmap, dmap;
  {
    const unsigned long long dims[5] = {(unsigned long long)a.D, (unsigned long long)K, (unsigned long long)a.N,
                                        (unsigned long long)a.B, (unsigned long long)a.T};
    const unsigned int box[5] = {(unsigned)sh.U, (unsigned)K, 1u, BC, 1u};
    cudaError_t e = encode_tensor_map(&tmap, a.tape, 4, 5, dims, box);
    if (e != cudaSuccess) return e;
  }
  if (a.dstates) {
    const unsigned long long dims[5] = {(unsigned long long)a.D, (unsigned long long)a.N, (unsigned long long)a.T,
                                        (unsigned long long)a.B, (unsigned long long)S};
    const unsigned int box[5] = {(unsigned)sh.U, 1u, 1u, BC, (unsigned)S};
    cudaError_t e = encode_tensor_map(&dmap, a.dstates, 2, 5, dims, box);
    if (e != cudaSuccess) return e;
  } else {
    dmap = tmap;
  }
  // dR beside the scan needs room for its TMA ring: the launch then holds at
  // least that much shared memory (the scan uses its own part of it)
  const size_t smem = a.drw.nc > 0 && sh.smem < (size_t)DRB_MIN_SMEM ? (size_t)DRB_MIN_SMEM : (size_t)sh.smem;
  cudaError_t e = set_smem_attr((const void*)k, smem);
  if (e != cudaSuccess) return e;
  const int groups = a.N * ((a.B + (int)BC - 1) / (int)BC);
  int per_sm = 0, dev = 0, sms = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, sh.warps * 32, smem);
  if (e != cudaSuccess) return e;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (per_sm * sms < groups * sh.C) return cudaErrorCooperativeLaunchTooLarge;
  FusedArgs args = a;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(groups * sh.C);
  // die placement holds one CTA per SM, so that each die's ticket counts
  // exactly its SMs; otherwise groups by block index
  if (args.die_of_sm && per_sm == 1 && args.launch_ctas == sms) cfg.gridDim = dim3(sms);
  else args.die_of_sm = nullptr;
  // dR beside the scan runs on the spare CTAs of a launch of one CTA per SM
  if (args.drw.nc > 0) {
    if (per_sm != 1 || !dmaps || sms <= groups * sh.C) return cudaErrorNotSupported;
    cfg.gridDim = dim3(sms);
  }
  args.groups = groups;
  cfg.blockDim = dim3(sh.warps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  UmmaMaps none;
  memset(&none, 0, sizeof(none));
  e = cudaLaunchKernelEx(&cfg, k, tmap, dmap, args, dmaps ? *dmaps : none);
  note_launch();
  return e;
}

}  // namespace rnn
