// Weight gradient of the recurrent branch on the 5th-generation tensor cores:
//   dR[g, n] (D x D) = Hprev^T dr,   K = B T (+ B rows for the initial state)
// one 128 x 128 output tile per CTA, the fp32 accumulator in tensor memory.
//
// Operands stream in by TMA with the 128-byte swizzle, k-rows of 64 units
// (128 bytes) per box, which is the MN-major canonical layout tcgen05 reads
// (atoms of 8 k-rows x 128 bytes; consecutive 8-row groups 1 KB apart, the two
// 64-unit halves of a tile 8 KB apart). The k-tiles are runs of 64 steps of
// one batch row b:
//   A rows: h_{t-1}[b, n, i0 .. i0+127] for t = t0 .. t0+63, i.e. states[0, b,
//           t0-1 .. t0+62] (a TMA box starting at t = -1 reads zeros there);
//   B rows: dr[b, t0 .. t0+63, g, n, j0 .. j0+127];
// rows past T read zeros on both sides. The initial state enters as extra
// k-tiles whose rows run over b: A = states0[0, b, n, :], B = dr[b, 0, g, n, :].
//
// Warp roles: thread 0 issues the TMA loads into a ring of 4 stages, thread 32
// issues the MMAs (4 per stage, K = 16 each) and releases each stage with
// tcgen05.commit; after the last stage all four warps read the accumulator
// (warp w owns TMEM lanes 32w .. 32w+31 = tile rows) and write dR, or fp32
// split-K partials that wgrad_reduce_kernel sums in a fixed order.
#include "kernels.cuh"
#include "ptx.cuh"

namespace rnn {

namespace {

constexpr int UM_TILE = 128, UM_BK = 64, UM_STAGES = 4;
constexpr int UM_BOX_BYTES = 64 * 128;              // one 64 x 64 bf16 box, 128-byte rows
constexpr int UM_STAGE_BYTES = 4 * UM_BOX_BYTES;    // A: two unit halves, B: two unit halves
constexpr int UM_SMEM = UM_STAGES * UM_STAGE_BYTES + 1024 + 256;  // + alignment slack, barriers

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

__global__ void __launch_bounds__(128, 1)
    wgrad_umma_kernel(const __grid_constant__ CUtensorMap amain, const __grid_constant__ CUtensorMap as0,
                      const __grid_constant__ CUtensorMap bmain, const __grid_constant__ CUtensorMap bs0,
                      WgradArgs a, int splits, int kps, int tpb, int s0_tiles) {
  extern __shared__ unsigned char um_raw[];
  unsigned char* sm = (unsigned char*)(((uintptr_t)um_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(sm + UM_STAGES * UM_STAGE_BYTES);  // full[4], empty[4], acc
  uint32_t* tslot = (uint32_t*)(bars + 2 * UM_STAGES + 1);
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[UM_STAGES]),
                 accb = smem_u32(&bars[2 * UM_STAGES]);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int D = a.D, N = a.N, G = a.G;
  const int j0 = blockIdx.x * UM_TILE, i0 = blockIdx.y * UM_TILE;
  const int gn = blockIdx.z / splits, split = blockIdx.z - gn * splits;
  const int g = gn / N, n = gn - g * N;
  const int Q = a.B * tpb + s0_tiles;
  const int q0 = split * kps, nq = min(Q, q0 + kps) - q0;

  if (tid == 0) {
    for (int s = 0; s < UM_STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(accb, 1);
    fence_mbar_init_cluster();
    prefetch_tensormap(&amain);
    prefetch_tensormap(&bmain);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 128;" ::"r"(smem_u32(tslot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  bool failed = false;

  int nissued = 0;
  if (tid == 0) {  // ---- TMA producer
    for (int it = 0; it < nq; ++it) {
      const int s = it % UM_STAGES;
      if (it >= UM_STAGES &&
          !mbar_wait_bounded<false>(empty0 + 8 * s, ((it / UM_STAGES) - 1) & 1, a.wait_limit_ns, a.status, failed))
        break;
      nissued = it + 1;
      const uint32_t fb = full0 + 8 * s;
      unsigned char* As = sm + (size_t)s * UM_STAGE_BYTES;
      unsigned char* Bs = As + 2 * UM_BOX_BYTES;
      mbar_arrive_expect_tx(fb, UM_STAGE_BYTES);
      const int q = q0 + it;
      if (q < a.B * tpb) {
        const int b = q / tpb, t0 = (q - b * tpb) * UM_BK;
        for (int h = 0; h < 2; ++h) {
          tma_load_5d(smem_u32(As + h * UM_BOX_BYTES), &amain, fb, i0 + 64 * h, n, t0 - 1, b, 0);
          tma_load_5d(smem_u32(Bs + h * UM_BOX_BYTES), &bmain, fb, j0 + 64 * h, n, g, t0, b);
        }
      } else {
        const int bb = (q - a.B * tpb) * UM_BK;
        for (int h = 0; h < 2; ++h) {
          tma_load_5d(smem_u32(As + h * UM_BOX_BYTES), &as0, fb, i0 + 64 * h, n, bb, 0, 0);
          tma_load_5d(smem_u32(Bs + h * UM_BOX_BYTES), &bs0, fb, j0 + 64 * h, n, g, 0, bb);
        }
      }
    }
  } else if (tid == 32) {  // ---- MMA issuer
    // kind::f16 descriptor: f32 accumulator, bf16 A and B, both MN-major, N = M = 128
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) |
                           ((uint32_t)(UM_TILE >> 3) << 17) | ((uint32_t)(UM_TILE >> 4) << 24);
    for (int it = 0; it < nq; ++it) {
      const int s = it % UM_STAGES;
      mbar_wait_bounded<false>(full0 + 8 * s, (it / UM_STAGES) & 1, a.wait_limit_ns, a.status, failed);
      tc_fence_after();
      const uint32_t As = smem_u32(sm + (size_t)s * UM_STAGE_BYTES), Bs = As + 2 * UM_BOX_BYTES;
      if (!failed) {
#pragma unroll
        for (int k = 0; k < UM_BK / 16; ++k)  // K = 16 per instruction: two 8-row groups, 2 KB
          umma_bf16(tmem, umma_desc_sw128(As + k * 2048), umma_desc_sw128(Bs + k * 2048), idesc,
                    (it | k) ? 1u : 0u);
      }
      umma_commit(empty0 + 8 * s);  // the stage is free once these MMAs have read it
    }
    umma_commit(accb);
  }

  // ---- epilogue: TMEM lanes 32 w .. 32 w + 31 are rows i0 + 32 w + lane
  mbar_wait_bounded<false>(accb, 0, a.wait_limit_ns, a.status, failed);
  tc_fence_after();
  const int i = i0 + warp * 32 + lane;
  for (int c0 = 0; c0 < UM_TILE; c0 += 32) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    if (i >= D || failed) continue;
    const int j = j0 + c0;
    if (splits == 1) {
      __nv_bfloat16* out = (__nv_bfloat16*)a.dR + (((size_t)g * N + n) * D + i) * D + j;
      if (j + 32 <= D) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_bf16(__float2bfloat16_rn(__uint_as_float(r[8 * v + 0])), __float2bfloat16_rn(__uint_as_float(r[8 * v + 1])));
          w.y = pack_bf16(__float2bfloat16_rn(__uint_as_float(r[8 * v + 2])), __float2bfloat16_rn(__uint_as_float(r[8 * v + 3])));
          w.z = pack_bf16(__float2bfloat16_rn(__uint_as_float(r[8 * v + 4])), __float2bfloat16_rn(__uint_as_float(r[8 * v + 5])));
          w.w = pack_bf16(__float2bfloat16_rn(__uint_as_float(r[8 * v + 6])), __float2bfloat16_rn(__uint_as_float(r[8 * v + 7])));
          *(uint4*)(out + 8 * v) = w;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (j + c < D) out[c] = __float2bfloat16_rn(__uint_as_float(r[c]));
      }
    } else {
      float* out = a.scratch + ((((size_t)split * G + g) * N + n) * D + i) * D + j;
      if (j + 32 <= D) {
#pragma unroll
        for (int v = 0; v < 8; ++v)
          *(float4*)(out + 4 * v) = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                                __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (j + c < D) out[c] = __uint_as_float(r[c]);
      }
    }
  }
  // every TMA load issued has landed before the CTA leaves (its stage was
  // consumed, or, after a time-out, waited for here with the same bound)
  if (tid == 0 && failed) {
    for (int it = nissued - UM_STAGES > 0 ? nissued - UM_STAGES : 0; it < nissued; ++it) {
      bool f2 = false;
      mbar_wait_bounded<false>(full0 + 8 * (it % UM_STAGES), (it / UM_STAGES) & 1, a.wait_limit_ns, nullptr, f2);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 128;" ::"r"(tmem) : "memory");
}

}  // namespace

bool wgrad_umma_supported(const WgradArgs& a) { return a.dR && a.D % 8 == 0 && a.D >= 64 && a.B * a.T > 0; }

int wgrad_umma_splits(int B, int T, int N, int D, int G) {
  const int tiles = ((D + UM_TILE - 1) / UM_TILE) * ((D + UM_TILE - 1) / UM_TILE) * G * N;
  const int Q = B * ((T + UM_BK - 1) / UM_BK) + (B + UM_BK - 1) / UM_BK;
  int splits = (device_sms() + tiles - 1) / tiles;  // about one wave of the SMs
  if (splits > Q / 4) splits = Q / 4;      // keep at least 4 k-tiles per split
  if (splits > 32) splits = 32;
  return splits < 1 ? 1 : splits;
}

cudaError_t wgrad_umma_run(const WgradArgs& a, int splits, cudaStream_t st) {
  const int tpb = (a.T + UM_BK - 1) / UM_BK;
  const int s0_tiles = a.s0 ? (a.B + UM_BK - 1) / UM_BK : 0;
  const int Q = a.B * tpb + s0_tiles;
  const int kps = (Q + splits - 1) / splits;
  splits = (Q + kps - 1) / kps;  // every split has at least one k-tile
  CUtensorMap amain, as0, bmain, bs0;
  const unsigned long long D = a.D, N = a.N, T = a.T, B = a.B, G = a.G;
  {  // states[0] as (D, N, T, B): rows of 64 steps of one batch row
    const unsigned long long dims[5] = {D, N, T, B, 1};
    const unsigned int box[5] = {64, 1, UM_BK, 1, 1};
    cudaError_t e = encode_tensor_map_sw128(&amain, a.states, 5, dims, box);
    if (e != cudaSuccess) return e;
  }
  {  // states0[0] as (D, N, B): rows over the batch
    const unsigned long long dims[5] = {D, N, B, 1, 1};
    const unsigned int box[5] = {64, 1, UM_BK, 1, 1};
    cudaError_t e = encode_tensor_map_sw128(&as0, a.s0 ? a.s0 : a.states, 5, dims, box);
    if (e != cudaSuccess) return e;
  }
  {  // dr as (D, N, G, T, B): rows of 64 steps, or rows over the batch at t = 0
    const unsigned long long dims[5] = {D, N, G, T, B};
    const unsigned int box_t[5] = {64, 1, 1, UM_BK, 1};
    const unsigned int box_b[5] = {64, 1, 1, 1, UM_BK};
    cudaError_t e = encode_tensor_map_sw128(&bmain, a.dr, 5, dims, box_t);
    if (e != cudaSuccess) return e;
    e = encode_tensor_map_sw128(&bs0, a.dr, 5, dims, box_b);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = set_smem_attr((const void*)wgrad_umma_kernel, (size_t)UM_SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid((a.D + UM_TILE - 1) / UM_TILE, (a.D + UM_TILE - 1) / UM_TILE, a.G * a.N * splits);
  wgrad_umma_kernel<<<grid, 128, UM_SMEM, st>>>(amain, as0, bmain, bs0, a, splits, kps, tpb, s0_tiles);
  note_launch();
  return cudaGetLastError();
}

}  // namespace rnn
