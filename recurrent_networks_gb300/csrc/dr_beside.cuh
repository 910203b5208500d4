// dR computed beside the grid backward scan.
//
// The grid backward is a cooperative launch of one CTA per SM in which only
// groups x C CTAs run the scan; the rest (24 on a GB300 for the LSTM D = 1024
// workload) would leave at once. Here they compute the weight gradient
//   dR[g, n] = sum_{b, t} h_{t-1}[b, n, :]^T dr_t[b, g, n, :]
// while the scan runs: the steps are cut into chunks (runs of 64-step tiles,
// in the scan's order, from t = T-1 down), and a chunk's dR tiles become work
// units once every group's step counter shows the scan past the chunk's first
// step. A unit is one 128 x 256 tile of one chunk on the tensor cores (the
// same TMA boxes and tcgen05 MMAs as the stand-alone dR GEMM), its fp32
// result written to the chunk's partial slot; after the launch one kernel
// adds the slots in chunk order. Units are taken from one atomic counter in
// order, so each is done once and the result does not depend on which CTA
// did it. The scan's CTAs take units too once their own scan is over, which
// shortens the last chunk. Every wait is bounded; a failure anywhere ends the
// loop on every thread of the CTA.
#pragma once
#include <cuda.h>

#include "grid_place.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace rnn {

constexpr int DRB_BN = 256;                                    // tile columns
constexpr int DRB_STAGE = (2 + DRB_BN / 64) * UM_BOX_BYTES;     // 48 KB: A two slabs, B four
constexpr int DRB_MAX_STAGES = 4;
// dynamic shared memory the worker needs: a 1 KB gap (the scan's barrier
// words), 1 KB of alignment slack, two stages, 256 bytes of barriers
constexpr int DRB_MIN_SMEM = 2048 + 2 * DRB_STAGE + 256;

// Waits until *ctr >= target, with 1 us sleeps between polls (the scan's own
// CTAs poll the same line); bounded and reporting like counter_wait_bounded.
__device__ __forceinline__ bool counter_wait_sleepy(const unsigned int* ctr, unsigned int target, uint64_t limit_ns,
                                                    unsigned int* status, bool& failed) {
  if (failed) return false;
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_gpu(ctr) < target) {
    if (globaltimer_ns() - t0 > limit_ns) {
      if (status) atomicExch(status, 1u);
      failed = true;
      return false;
    }
    __nanosleep(1000);
  }
  return true;
}

// Barrier 1 over the worker's 128 threads, returning whether any of them
// passed `flag` set.
__device__ __forceinline__ bool worker_sync_or(bool flag) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred q, p;\n setp.ne.u32 q, %1, 0;\n"
      " bar.red.or.pred p, 1, 128, q;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(r)
      : "r"((uint32_t)flag)
      : "memory");
  return r != 0;
}

// Threads 0..127 of the CTA take and compute units until none is left; the
// others return at once. smem: the kernel's dynamic shared memory, free to
// reuse from its second KB on (every thread is done with it).
static __device__ __noinline__ void dr_beside(const FusedArgs& a, const UmmaMaps& mp, int G, unsigned char* smem) {
  const int tid = threadIdx.x;
  if (a.drw.nc <= 0) return;
  if (blockDim.x < 128) {  // the host asks for workers only with four warps or more
    if (tid == 0 && a.status) atomicExch(a.status, 1u);
    return;
  }
  if (tid >= 128) return;
  uint32_t smem_bytes;
  asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(smem_bytes));
  const int warp = tid >> 5, lane = tid & 31;
  unsigned char* sm = (unsigned char*)(((uintptr_t)smem + 1024 + 1023) & ~(uintptr_t)1023);
  int stages = ((int)smem_bytes - (int)(sm - smem) - 256) / DRB_STAGE;
  if (stages > DRB_MAX_STAGES) stages = DRB_MAX_STAGES;
  if (stages < 2) {  // the host checks the size; a unit left undone is reported, not skipped silently
    if (tid == 0 && a.status) atomicExch(a.status, 1u);
    return;
  }
  uint64_t* bars = (uint64_t*)(sm + (size_t)stages * DRB_STAGE);  // full[4], empty[4], acc, tmem slot, unit
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[DRB_MAX_STAGES]),
                 accb = smem_u32(&bars[2 * DRB_MAX_STAGES]);
  uint32_t* tslot = (uint32_t*)(bars + 2 * DRB_MAX_STAGES + 1);
  int* unit_slot = (int*)(bars + 2 * DRB_MAX_STAGES + 2);
  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(accb, 1);
    fence_mbar_init_cluster();
    fence_proxy_async_smem();  // earlier generic use of this memory before the TMA writes into it
    prefetch_tensormap(&mp.amain);
    prefetch_tensormap(&mp.bmain);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "n"(DRB_BN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  worker_sync_or(false);
  tc_fence_after();
  const uint32_t tmem = *tslot;

  const int D = a.D, N = a.N, B = a.B, TT = a.T, C = a.C;
  const int tx = (D + DRB_BN - 1) / DRB_BN, ty = (D + UM_TILE - 1) / UM_TILE;
  const int upc = tx * ty * G * N;  // units per chunk
  const int total = upc * a.drw.nc;
  // kind::f16: f32 accumulator, bf16 A and B, both MN-major, M = 128, N = 256
  const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) |
                         ((uint32_t)(DRB_BN >> 3) << 17) | ((uint32_t)(UM_TILE >> 4) << 24);
  bool failed = false;
  int gi = 0, done = 0, nissued = 0;
  for (;;) {
    if (tid == 0) *unit_slot = (int)atomicAdd(a.drw.next, 1u);
    worker_sync_or(false);
    const int u = *unit_slot;
    if (u >= total) break;
    const int c = u / upc, tile = u - c * upc;
    const int xx = tile % tx, yy = (tile / tx) % ty, gn = tile / (tx * ty);
    const int j0 = xx * DRB_BN, i0 = yy * UM_TILE, g = gn / N, n = gn - g * N;
    const int ttlo = a.drw.tt_lo[c], ntt = a.drw.tt_n[c];
    const int nmain = B * ntt;
    const int nq = nmain + (c == a.drw.nc - 1 ? a.drw.s0_tiles : 0);
    if (tid == 0) {  // ---- producer: the chunk's steps are done, then its boxes
      const unsigned need = (unsigned)C * (unsigned)(TT - ttlo * UM_BK);
      for (int gg = 0; gg < a.groups; ++gg)
        counter_wait_sleepy(group_counter(a, gg), need, a.wait_limit_ns, a.status, failed);
      fence_proxy_async_global();  // the scan's dr stores, acquired above, before the TMA reads
      for (int it = 0; it < nq && !failed; ++it) {
        const int gq = gi + it, s = gq % stages;
        if (gq >= stages &&
            !mbar_wait_bounded<false>(empty0 + 8 * s, ((gq / stages) - 1) & 1, a.wait_limit_ns, a.status, failed))
          break;
        nissued = gq + 1;
        const uint32_t fb = full0 + 8 * s;
        const uint32_t As = smem_u32(sm + (size_t)s * DRB_STAGE), Bs = As + 2 * UM_BOX_BYTES;
        mbar_arrive_expect_tx(fb, DRB_STAGE);
        if (it < nmain) {
          const int b = it / ntt, t0 = (ttlo + it - b * ntt) * UM_BK;
          tma_load_5d(As, &mp.amain, fb, 0, t0 - 1, i0 / 64, n, b);
          tma_load_5d(Bs, &mp.bmain, fb, 0, t0, j0 / 64, g * N + n, b);
        } else {
          const int bb = (it - nmain) * UM_BK;
          tma_load_5d(As, &mp.as0, fb, 0, bb, i0 / 64, n, 0);
          tma_load_5d(Bs, &mp.bs0, fb, 0, bb, j0 / 64, g * N + n, 0);
        }
      }
    } else if (tid == 32) {  // ---- MMA issuer
      for (int it = 0; it < nq; ++it) {
        const int gq = gi + it, s = gq % stages;
        mbar_wait_bounded<false>(full0 + 8 * s, (gq / stages) & 1, a.wait_limit_ns, a.status, failed);
        tc_fence_after();
        const uint32_t As = smem_u32(sm + (size_t)s * DRB_STAGE), Bs = As + 2 * UM_BOX_BYTES;
        if (!failed) {
#pragma unroll
          for (int k = 0; k < UM_BK / 16; ++k)
            umma_bf16(tmem, umma_desc_sw128(As + k * 2048), umma_desc_sw128(Bs + k * 2048), idesc,
                      (it | k) ? 1u : 0u);
        }
        umma_commit(empty0 + 8 * s);
      }
      umma_commit(accb);
    }
    gi += nq;
    // ---- epilogue: TMEM lanes 32 w .. 32 w + 31 are rows i0 + 32 w + lane
    mbar_wait_bounded<false>(accb, done & 1, a.wait_limit_ns, a.status, failed);
    tc_fence_after();
    const int i = i0 + warp * 32 + lane;
    float* slot = a.drw.slots + (((size_t)c * G + g) * N + n) * D * D;
    for (int c0 = 0; c0 < DRB_BN; c0 += 32) {
      uint32_t r[32];
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
          "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
          : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
            "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
            "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
            "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
            "=r"(r[30]), "=r"(r[31])
          : "r"(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      const int j = j0 + c0;
      if (i >= D || failed) continue;
      float* out = slot + (size_t)i * D + j;
      if (j + 32 <= D) {
#pragma unroll
        for (int v = 0; v < 8; ++v)
          *(float4*)(out + 4 * v) = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                                __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
      } else {
        for (int cc = 0; cc < 32; ++cc)
          if (j + cc < D) out[cc] = __uint_as_float(r[cc]);
      }
    }
    ++done;
    // the accumulator is read before the next unit's first MMA overwrites it;
    // a failure anywhere stops every thread
    tc_fence_before();
    const bool any_failed = worker_sync_or(failed);
    tc_fence_after();
    if (any_failed) {
      failed = true;
      break;
    }
  }
  // every TMA load issued has landed before the CTA leaves
  if (tid == 0 && failed)
    for (int it = nissued - stages > 0 ? nissued - stages : 0; it < nissued; ++it) {
      bool f2 = false;
      mbar_wait_bounded<false>(full0 + 8 * (it % stages), (it / stages) & 1, a.wait_limit_ns, nullptr, f2);
    }
  tc_fence_before();
  worker_sync_or(false);
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(DRB_BN) : "memory");
}

}  // namespace rnn
