// Latency floor of the cluster h exchange: the steps of the forward cluster
// kernel with the product and the cell update taken out. Each step: wait for
// the C slices of the previous step (mbarrier transaction count, bounded),
// order the staged slice for the async proxy, a CTA barrier, then one bulk
// copy per peer (shared::cta -> shared::cluster) into the peer's next buffer,
// issued as in the forward kernel: lane q of warp w sends to peer
// rank + w + q warps, with the cluster addresses computed once.
#include <stdio.h>

#include "grid_place.cuh"
#include "kernels.cuh"
#include "plan.h"
#include "ptx.cuh"
#include "rnn.h"

namespace rnn {

namespace {

__global__ void __launch_bounds__(256, 1) exchange_floor_kernel(int slice_bytes, int steps, unsigned long long* out) {
  extern __shared__ __align__(128) unsigned char fl_smem[];
  const int C = (int)gridDim.x;  // the grid is one cluster
  uint64_t* bars = (uint64_t*)fl_smem;
  unsigned char* hbuf = fl_smem + 128;                          // [2][C][slice]
  unsigned char* stage = hbuf + (size_t)2 * C * slice_bytes;    // [2][slice]
  const uint32_t rank = cluster_ctarank();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
  const uint32_t bar0 = smem_u32(&bars[0]);
  unsigned int* status = (unsigned int*)(out + 1);
  const unsigned long long limit = 2000000000ull;
  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    fence_mbar_init_cluster();
  }
  for (int e = tid; e < 2 * slice_bytes; e += blockDim.x) stage[e] = (unsigned char)e;
  __syncthreads();
  cluster_sync_all();
  const uint32_t hbytes = (uint32_t)C * slice_bytes;
  if (tid == 0) {
    if (steps > 1) mbar_arrive_expect_tx(bar0 + 8, hbytes);
    if (steps > 2) mbar_arrive_expect_tx(bar0, hbytes);
  }
  const int my_c = warp + lane * nwarps;
  const bool sender = lane < (C + nwarps - 1) / nwarps && my_c < C;
  uint32_t rdst0 = 0, rdst1 = 0, rbar0 = 0, rbar1 = 0;
  if (sender) {
    int peer = (int)rank + my_c;
    if (peer >= C) peer -= C;
    rdst0 = mapa_shared(smem_u32(hbuf + (size_t)rank * slice_bytes), (uint32_t)peer);
    rdst1 = mapa_shared(smem_u32(hbuf + (size_t)C * slice_bytes + (size_t)rank * slice_bytes), (uint32_t)peer);
    rbar0 = mapa_shared(bar0, (uint32_t)peer);
    rbar1 = mapa_shared(bar0 + 8, (uint32_t)peer);
  }
  bool failed = false;
  uint32_t ph0 = 0, ph1 = 0;
  const long long t0 = clock64();
  for (int t = 0; t < steps; ++t) {
    const int p = t & 1;
    if (t > 0) {
      mbar_wait_bounded(bar0 + 8 * p, p ? ph1 : ph0, limit, status, failed);
      if (p) ph1 ^= 1u; else ph0 ^= 1u;
      if (tid == 0 && t + 2 <= steps - 1) mbar_arrive_expect_tx(bar0 + 8 * p, hbytes);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (t + 1 < steps && sender)  // into the peer's buffer p ^ 1
      bulk_copy_to_peer(p ? rdst0 : rdst1, smem_u32(stage + (size_t)p * slice_bytes), (uint32_t)slice_bytes,
                        p ? rbar0 : rbar1);
  }
  const long long t1 = clock64();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while a peer may still write into its shared memory
  if (rank == 0 && tid == 0) out[0] = (unsigned long long)((t1 - t0) / steps);
}

// Latency floor of the grid kernels' L2 exchange: the forward grid kernel's
// steps with the product and the cell taken out. C CTAs per group, `groups`
// groups, one CTA per SM (cooperative launch). Each step t > 0: one thread
// waits until the group's step counter reaches C t (acquire), fences the
// proxies and pulls the group's `rows` rows of h_{t-1} (D bf16 each) from L2
// with one bulk copy per row; every thread waits for the bytes. Then every
// CTA stores its U = D / C units of h_t for each row (2-byte stores, as the
// cell does), a CTA barrier, and one release increment of the counter.
__global__ void __launch_bounds__(256, 1) grid_floor_kernel(int D, int rows, int steps, int groups, unsigned short* hx,
                                                          FusedArgs pl, unsigned long long* out) {
  extern __shared__ __align__(128) unsigned char gf_smem[];
  const int C = pl.C;
  const int2 place = grid_place(pl, C, (int*)gf_smem);  // as the grid kernels place their CTAs
  if (place.x < 0) return;
  const int U = D / C, grp = place.x, r = place.y;
  unsigned int* ctr = group_counter(pl, grp);
  const int tid = threadIdx.x;
  uint64_t* bar = (uint64_t*)gf_smem;
  unsigned short* hbuf = (unsigned short*)(gf_smem + 128);  // [rows][D + 8]
  unsigned int* status = (unsigned int*)(out + 1);
  const unsigned long long limit = 2000000000ull;
  const uint32_t bar0 = smem_u32(bar);
  if (tid == 0) {
    mbar_init(bar0, 1);
    fence_mbar_init_cluster();
  }
  __syncthreads();
  bool failed = false;
  uint32_t ph = 0;
  unsigned x = 0;
  const long long t0 = clock64();
  for (int t = 0; t < steps; ++t) {
    const int p = t & 1;
    if (t > 0) {
      if (tid == 0) {
        counter_wait_bounded(ctr, (unsigned)(C * t), limit, status, failed);
        if (!failed) {
          const unsigned short* src = hx + ((size_t)(p * groups + grp) * rows) * D;
          fence_proxy_async_global();
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(bar0, (uint32_t)(rows * D * 2));
          for (int b = 0; b < rows; ++b)
            bulk_load_global(smem_u32(hbuf + b * (D + 8)), src + (size_t)b * D, (uint32_t)(D * 2), bar0);
        }
      }
      mbar_wait_bounded<false>(bar0, ph, limit, status, failed);
      ph ^= 1u;
      x += hbuf[tid % (rows * (D + 8))];  // the pulled row is read, as the product reads it
    }
    if (t + 1 < steps) {
      unsigned short* dst = hx + ((size_t)((p ^ 1) * groups + grp) * rows) * D;
      for (int e = tid; e < rows * U; e += blockDim.x) {
        const int b = e / U, u = e - b * U;
        dst[(size_t)b * D + r * U + u] = (unsigned short)(t + x);
      }
    }
    __syncthreads();
    if (t + 1 < steps && tid == 0) counter_publish(ctr);
  }
  const long long t1 = clock64();
  if (grp == 0 && r == 0 && tid == 0) out[0] = (unsigned long long)((t1 - t0) / steps) + (x == 0xffffffffu);
}

}  // namespace

}  // namespace rnn

using namespace rnn;

extern "C" int rnn_exchange_floor_grid(int C, int groups, int rows, int D, int steps, void* scratch,
                                       size_t scratch_bytes, void* out, void* stream) {
  if (C < 1 || groups < 1 || rows < 1 || rows > 32 || D < 8 || D > 4096 || D % 8 || D % C || steps < 2 ||
      steps > 1000000 || !scratch || ((uintptr_t)scratch & 255u) || !out || ((uintptr_t)out & 7u))
    return RNN_EINVAL;
  const size_t hx_bytes = ((size_t)2 * groups * rows * D * 2 + 255) & ~(size_t)255;
  if (scratch_bytes < hx_bytes + GRID_CTR_BYTES) return RNN_ENOSPC;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned short* hx = (unsigned short*)scratch;
  FusedArgs pl{};
  pl.C = C;
  pl.counters = (unsigned int*)(((uintptr_t)scratch + hx_bytes + 1023) & ~(uintptr_t)1023);
  // the grid kernels' die placement, when they would use it
  DiePlan dp;
  const bool die = die_plan(groups, C, pl.counters, st, &dp);
  if (die) {
    for (int g = 0; g < groups; ++g) pl.ctr_word[g] = dp.ctr_word[g];
    pl.die_of_sm = dp.table;
    pl.tickets = pl.counters + GRID_CTR_BLOCKS * 256;
    for (int d = 0; d < 2; ++d) {
      pl.die_grp0[d] = dp.grp0[d];
      pl.die_ngrp[d] = dp.ngrp[d];
    }
  }
  // at least as much shared memory as the forward grid kernel, so one CTA runs per SM
  size_t smem = 128 + (size_t)rows * (D + 8) * 2;
  if (smem < 100 * 1024) smem = 100 * 1024;
  const size_t ctr_bytes = (groups > GRID_CTR_BLOCKS * 256 ? (size_t)groups : (size_t)GRID_CTR_BLOCKS * 256) * 4 + 256;
  cudaError_t e = cudaMemsetAsync(out, 0, 16, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(pl.counters, 0, ctr_bytes, st);
  if (e == cudaSuccess) e = set_smem_attr((const void*)grid_floor_kernel, smem);
  int per_sm = 0;
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, grid_floor_kernel, 256, smem);
  if (e == cudaSuccess && per_sm * device_sms() < groups * C) return RNN_EUNSUPPORTED;
  if (e == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(groups * C);
    if (die && per_sm == 1 && dp.sms == device_sms()) cfg.gridDim = dim3(dp.sms);
    else pl.die_of_sm = nullptr;
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, grid_floor_kernel, D, rows, steps, groups, hx, pl, (unsigned long long*)out);
    note_launch();
  }
  if (e != cudaSuccess) {
    fprintf(stderr, "librnn_gb300: CUDA error: %s\n", cudaGetErrorString(e));
    return RNN_ECUDA;
  }
  return RNN_OK;
}

extern "C" int rnn_exchange_floor(int C, int slice_bytes, int steps, void* out, void* stream) {
  if (C < 1 || C > 16 || slice_bytes < 16 || slice_bytes > 4096 || slice_bytes % 16 || steps < 2 ||
      steps > 1000000 || !out || ((uintptr_t)out & 7u))
    return RNN_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t smem = 128 + (size_t)2 * C * slice_bytes + (size_t)2 * slice_bytes;
  cudaError_t e = cudaMemsetAsync(out, 0, 16, st);
  if (e == cudaSuccess) e = set_smem_attr((const void*)exchange_floor_kernel, (size_t)smem);
  if (e == cudaSuccess && C > 8) e = set_nonportable_cluster((const void*)exchange_floor_kernel);
  if (e == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, exchange_floor_kernel, slice_bytes, steps, (unsigned long long*)out);
    note_launch();
  }
  if (e != cudaSuccess) {
    fprintf(stderr, "librnn_gb300: CUDA error: %s\n", cudaGetErrorString(e));
    return RNN_ECUDA;
  }
  return RNN_OK;
}
