// tcgen05 building blocks of the weight-gradient GEMM (dR = Hprev^T dr):
// tile geometry, shared-memory descriptors of the 128-byte-swizzled MN-major
// operands, the MMA / commit / fence instructions, and the tensor maps of the
// operands (encoded by umma_encode_maps in wgrad_umma.cu). Written from the
// PTX ISA.
#pragma once
#include <cuda.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace rnn {

constexpr int UM_TILE = 128, UM_BK = 64;           // tile rows (i), k-rows per stage
constexpr int UM_BOX_BYTES = 64 * 128;              // one 64 x 64 bf16 box, 128-byte rows

// The tile width for head size D: the columns rounded up to 64, at most 256.
inline int um_bn(int D) { return D <= 128 ? 128 : (D <= 192 ? 192 : 256); }

template <int BN>
struct UmCfg {
  static constexpr int NB = BN / 64;                            // B boxes per stage
  static constexpr int STAGE_BYTES = (2 + NB) * UM_BOX_BYTES;   // A: two 64-unit halves, B: NB
  static constexpr int STAGES = (192 * 1024) / STAGE_BYTES;
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + 256;  // + alignment slack, barriers
  static constexpr int TCOLS = BN <= 128 ? 128 : 256;           // tensor-memory columns (a power of two)
};

__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t addr) {
  // start address, leading byte offset = stride of the 64-unit halves (8 KB),
  // stride byte offset = stride of the 8-row groups (1 KB), version 1,
  // layout: 128-byte swizzle
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)(UM_BOX_BYTES >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem),
      "l"(ad), "l"(bd), "r"(idesc), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }


// The four operand maps of one dR problem: h_{t-1} rows (states[0]), the
// initial-state rows (states0[0]), dr rows over t and dr rows over the batch
// at t = 0; with gathered boxes when D % 64 == 0.
struct UmmaMaps {
  CUtensorMap amain, as0, bmain, bs0;
};
// Encodes them for a's problem with tiles BN columns wide (blk: gathered
// boxes, which needs D % 64 == 0).
cudaError_t umma_encode_maps(const WgradArgs& a, int bn, bool blk, UmmaMaps* m);

}  // namespace rnn
