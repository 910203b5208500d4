// Weight gradient of the recurrent branch on the 5th-generation tensor cores:
//   dR[g, n] (D x D) = Hprev^T dr,   K = B T (+ B rows for the initial state)
// one 128 x BN output tile per CTA (BN = 128, 192 or 256 columns: the head
// size rounded up to 64, at most 256), the fp32 accumulator in tensor memory.
// Wider tiles read each row block of h once per BN columns instead of per 128,
// and a head of 192 units needs no padded columns.
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
// Warp roles: thread 0 issues the TMA loads into a ring of stages (as many as
// 192 KB hold: 6 for BN = 128, 4 for 192 and 256), thread 32
// issues the MMAs (4 per stage, K = 16 each) and releases each stage with
// tcgen05.commit; after the last stage all four warps read the accumulator
// (warp w owns TMEM lanes 32w .. 32w+31 = tile rows) and write dR, or fp32
// split-K partials that wgrad_reduce_kernel sums in a fixed order.
#include "kernels.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace rnn {

namespace {

template <int BN, bool BLK>
__global__ void __launch_bounds__(128, 1)
    wgrad_umma_kernel(const __grid_constant__ CUtensorMap amain, const __grid_constant__ CUtensorMap as0,
                      const __grid_constant__ CUtensorMap bmain, const __grid_constant__ CUtensorMap bs0,
                      WgradArgs a, int splits, int kps, int tpb, int s0_tiles) {
  using Cfg = UmCfg<BN>;
  constexpr int UM_STAGES = Cfg::STAGES, UM_STAGE_BYTES = Cfg::STAGE_BYTES, NB = Cfg::NB;
  extern __shared__ unsigned char um_raw[];
  unsigned char* sm = (unsigned char*)(((uintptr_t)um_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(sm + UM_STAGES * UM_STAGE_BYTES);  // full[4], empty[4], acc
  uint32_t* tslot = (uint32_t*)(bars + 2 * UM_STAGES + 1);
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[UM_STAGES]),
                 accb = smem_u32(&bars[2 * UM_STAGES]);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int D = a.D, N = a.N, G = a.G;
  const int j0 = blockIdx.x * BN, i0 = blockIdx.y * UM_TILE;
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
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "n"(Cfg::TCOLS)
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
        if (BLK) {  // one box per operand: the 64-unit slabs land 8 KB apart
          tma_load_5d(smem_u32(As), &amain, fb, 0, t0 - 1, i0 / 64, n, b);
          tma_load_5d(smem_u32(Bs), &bmain, fb, 0, t0, j0 / 64, g * N + n, b);
        } else {
          for (int h = 0; h < 2; ++h)
            tma_load_5d(smem_u32(As + h * UM_BOX_BYTES), &amain, fb, i0 + 64 * h, n, t0 - 1, b, 0);
          for (int h = 0; h < NB; ++h)
            tma_load_5d(smem_u32(Bs + h * UM_BOX_BYTES), &bmain, fb, j0 + 64 * h, n, g, t0, b);
        }
      } else {
        const int bb = (q - a.B * tpb) * UM_BK;
        if (BLK) {
          tma_load_5d(smem_u32(As), &as0, fb, 0, bb, i0 / 64, n, 0);
          tma_load_5d(smem_u32(Bs), &bs0, fb, 0, bb, j0 / 64, g * N + n, 0);
        } else {
          for (int h = 0; h < 2; ++h)
            tma_load_5d(smem_u32(As + h * UM_BOX_BYTES), &as0, fb, i0 + 64 * h, n, bb, 0, 0);
          for (int h = 0; h < NB; ++h)
            tma_load_5d(smem_u32(Bs + h * UM_BOX_BYTES), &bs0, fb, j0 + 64 * h, n, g, 0, bb);
        }
      }
    }
  } else if (tid == 32) {  // ---- MMA issuer
    // kind::f16 descriptor: f32 accumulator, bf16 A and B, both MN-major, M = 128, N = BN
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) |
                           ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(UM_TILE >> 4) << 24);
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
  for (int c0 = 0; c0 < BN; c0 += 32) {
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
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(Cfg::TCOLS) : "memory");
}

}  // namespace

bool wgrad_umma_supported(const WgradArgs& a) { return a.dR && a.D % 8 == 0 && a.D >= 64 && a.B * a.T > 0; }

int wgrad_umma_splits(int B, int T, int N, int D, int G) {
  // Split K so that the waves of CTAs (one per SM) divide evenly: a split
  // count s costs ceil(tiles s / SMs) / s of the unsplit tile time, plus the
  // fp32 partials written and reduced (s D^2 words per head, each way).
  const int bn = um_bn(D);
  const int tiles = ((D + bn - 1) / bn) * ((D + UM_TILE - 1) / UM_TILE) * G * N;
  const int Q = B * ((T + UM_BK - 1) / UM_BK) + (B + UM_BK - 1) / UM_BK;
  const int sms = device_sms();
  const double tile_s = 2.0 * UM_TILE * bn * UM_BK * (double)Q / 1.0e13;  // one tile, all of K, on one SM
  const double part_s = 2.0 * 4.0 * G * N * (double)D * D / 6.0e12;       // one split's partials, out and back
  int best = 1;
  double best_t = 1e30;
  const int smax = Q / 4 < 32 ? Q / 4 : 32;  // keep at least 4 k-tiles per split
  for (int s = 1; s <= (smax < 1 ? 1 : smax); ++s) {
    const double t = (double)((tiles * s + sms - 1) / sms) * tile_s / s + (s > 1 ? s * part_s + 3e-6 : 0.0);
    if (t < best_t * 0.98) best = s, best_t = t;  // a split must gain 2% to be taken
  }
  return best;
}

cudaError_t umma_encode_maps(const WgradArgs& a, int bn, bool blk, UmmaMaps* m) {
  const unsigned long long D = a.D, N = a.N, T = a.T, B = a.B, G = a.G;
  // With D a multiple of 64, one box per operand and stage gathers the tile's
  // 64-unit slabs (dimension 2, 128 bytes apart in memory) into consecutive
  // 8 KB blocks: 2 TMA copies per stage instead of 2 + BN / 64.
  if (blk) {
    const unsigned int box_a[5] = {64, UM_BK, 2, 1, 1};
    const unsigned int box_b[5] = {64, UM_BK, (unsigned)bn / 64, 1, 1};
    {  // states[0] (B, T, N, D) as (unit, t, slab, n, b)
      const unsigned long long dims[5] = {64, T, D / 64, N, B};
      const unsigned long long str[4] = {N * D * 2, 128, D * 2, T * N * D * 2};
      cudaError_t e = encode_tensor_map_sw128_strided(&m->amain, a.states, 5, dims, str, box_a);
      if (e != cudaSuccess) return e;
    }
    {  // states0[0] (B, N, D) as (unit, b, slab, n)
      const unsigned long long dims[5] = {64, B, D / 64, N, 1};
      const unsigned long long str[4] = {N * D * 2, 128, D * 2, B * N * D * 2};
      cudaError_t e = encode_tensor_map_sw128_strided(&m->as0, a.s0 ? a.s0 : a.states, 5, dims, str, box_a);
      if (e != cudaSuccess) return e;
    }
    {  // dr (B, T, G, N, D) as (unit, t, slab, g n, b), and as (unit, b, slab, g n, t)
      const unsigned long long dims_t[5] = {64, T, D / 64, G * N, B};
      const unsigned long long str_t[4] = {G * N * D * 2, 128, D * 2, T * G * N * D * 2};
      cudaError_t e = encode_tensor_map_sw128_strided(&m->bmain, a.dr, 5, dims_t, str_t, box_b);
      if (e != cudaSuccess) return e;
      const unsigned long long dims_b[5] = {64, B, D / 64, G * N, T};
      const unsigned long long str_b[4] = {T * G * N * D * 2, 128, D * 2, G * N * D * 2};
      e = encode_tensor_map_sw128_strided(&m->bs0, a.dr, 5, dims_b, str_b, box_b);
      if (e != cudaSuccess) return e;
    }
  } else {
    {  // states[0] as (D, N, T, B): rows of 64 steps of one batch row
      const unsigned long long dims[5] = {D, N, T, B, 1};
      const unsigned int box[5] = {64, 1, UM_BK, 1, 1};
      cudaError_t e = encode_tensor_map_sw128(&m->amain, a.states, 5, dims, box);
      if (e != cudaSuccess) return e;
    }
    {  // states0[0] as (D, N, B): rows over the batch
      const unsigned long long dims[5] = {D, N, B, 1, 1};
      const unsigned int box[5] = {64, 1, UM_BK, 1, 1};
      cudaError_t e = encode_tensor_map_sw128(&m->as0, a.s0 ? a.s0 : a.states, 5, dims, box);
      if (e != cudaSuccess) return e;
    }
    {  // dr as (D, N, G, T, B): rows of 64 steps, or rows over the batch at t = 0
      const unsigned long long dims[5] = {D, N, G, T, B};
      const unsigned int box_t[5] = {64, 1, 1, UM_BK, 1};
      const unsigned int box_b[5] = {64, 1, 1, 1, UM_BK};
      cudaError_t e = encode_tensor_map_sw128(&m->bmain, a.dr, 5, dims, box_t);
      if (e != cudaSuccess) return e;
      e = encode_tensor_map_sw128(&m->bs0, a.dr, 5, dims, box_b);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

cudaError_t wgrad_umma_run(const WgradArgs& a, int& splits, cudaStream_t st) {
  const int tpb = (a.T + UM_BK - 1) / UM_BK;
  const int s0_tiles = a.s0 ? (a.B + UM_BK - 1) / UM_BK : 0;
  const int Q = a.B * tpb + s0_tiles;
  const int kps = (Q + splits - 1) / splits;
  splits = (Q + kps - 1) / kps;  // every split has at least one k-tile
  const int bn = um_bn(a.D);
  const bool blk = a.D % 64 == 0;
  UmmaMaps m;
  {
    const cudaError_t e = umma_encode_maps(a, bn, blk, &m);
    if (e != cudaSuccess) return e;
  }
  void (*k)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, WgradArgs, int, int, int, int) =
      blk ? (bn == 128 ? wgrad_umma_kernel<128, true> : bn == 192 ? wgrad_umma_kernel<192, true> : wgrad_umma_kernel<256, true>)
          : (bn == 128 ? wgrad_umma_kernel<128, false> : bn == 192 ? wgrad_umma_kernel<192, false> : wgrad_umma_kernel<256, false>);
  const int smem = bn == 128 ? UmCfg<128>::SMEM : bn == 192 ? UmCfg<192>::SMEM : UmCfg<256>::SMEM;
  cudaError_t e = set_smem_attr((const void*)k, (size_t)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((a.D + bn - 1) / bn, (a.D + UM_TILE - 1) / UM_TILE, a.G * a.N * splits);
  k<<<grid, 128, smem, st>>>(m.amain, m.as0, m.bmain, m.bs0, a, splits, kps, tpb, s0_tiles);
  note_launch();
  return cudaGetLastError();
}

}  // namespace rnn
