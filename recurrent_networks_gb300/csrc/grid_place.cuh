// Placement of a CTA of the cooperative grid kernels in its batch group.
#pragma once
#include "kernels.cuh"

namespace rnn {

// (group, rank) of this CTA: by block index, or, with die placement on
// (a.die_of_sm), from a ticket of the CTA's die, so that each group's C CTAs
// share a die; {-1, -1} for a spare CTA, which takes part in nothing and
// leaves. `scratch` is 8 bytes of shared memory not yet in use; every thread
// must call this (it ends with a block barrier).
__device__ __forceinline__ int2 grid_place(const FusedArgs& a, int C, int* scratch) {
  if (threadIdx.x == 0) {
    int2 p = make_int2((int)(blockIdx.x / C), (int)(blockIdx.x % C));
    if (a.groups > 0 && (int)blockIdx.x >= a.groups * C) p = make_int2(-1, -1);  // a spare CTA
    if (a.die_of_sm) {
      unsigned sm;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
      const int d = a.die_of_sm[sm & 255u];
      p = make_int2(-1, -1);
      if (d == 0 || d == 1) {
        const unsigned r = atomicAdd(a.tickets + d, 1u);
        if (r < (unsigned)(a.die_ngrp[d] * C)) p = make_int2(a.die_grp0[d] + (int)(r / C), (int)(r % C));
      }
    }
    scratch[0] = p.x;
    scratch[1] = p.y;
  }
  __syncthreads();
  const int2 p = make_int2(scratch[0], scratch[1]);
  __syncthreads();  // the scratch words are free again
  return p;
}

// The step counter of group g.
__device__ __forceinline__ unsigned int* group_counter(const FusedArgs& a, int g) {
  return a.counters + (g < FUSED_MAX_GROUP_CTR ? a.ctr_word[g] : g);
}

}  // namespace rnn
