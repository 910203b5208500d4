// Input projection of the scan on the 5th-generation tensor cores.
//
// developnotes "deep learning operators", section 5.3 LSTM (MyLSTM.forward)
// computes the input branch of every gate as x_t W_ih^T + b_ih before adding
// the recurrent branch; the FlashRNN announcement's flashrnn() takes that
// product, Wx, as its input. These kernels compute it for a whole sequence at
// once, with W_x in the weight_ih layout [C][I] (C = G N D output columns in
// the order of Wx's last three axes):
//   forward   Wx[m, c]  = sum_i x[m, i] W_x[c, i] (+ bias[c])   m = (b, t), K = I
//   backward  dx[m, i]  = sum_c dWx[m, c] W_x[c, i]              K = C
//             dW_x[c, i] = sum_m dWx[m, c] x[m, i]               K = B T (split-K)
//             dbias[c]  = sum_m dWx[m, c]
// One generic GEMM, D[M][N] = sum_k A(m, k) B(k, n), with either operand stored
// K-major (k contiguous: rows of 64 k per 128-byte TMA box) or MN-major (m / n
// contiguous: boxes of 64 m / n by 64 k), both 128-byte swizzled, in the
// canonical layouts tcgen05 reads; 128 x BN tiles (BN = 128 or 256), the fp32
// accumulator in tensor memory. The kernel is persistent: one CTA per SM walks
// the tiles (and split-K slices), with warp-specialised roles. Warp 0 feeds a
// TMA / mbarrier ring that runs ahead across tile boundaries, warp 1 issues the
// MMAs, and warps 2-5 drain the accumulator. Tensor memory holds two
// accumulators, so one tile's epilogue overlaps the next tile's MMAs. The
// epilogue leaves through shared memory as TMA stores of 64-byte-swizzled
// 32 x 32 boxes, clipped at the matrix edges; split-K partials leave the same
// way and a second kernel adds them in a fixed order. dbias is a two-pass
// column sum.
#include <stdio.h>

#include <cmath>

#include "colsum.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "rnn.h"

namespace rnn {

namespace {

// tiles: 128 rows of M by BN (128 or 256) columns of N, k-chunks of 64
constexpr int GM_TILE = 128, GM_BK = 64;
constexpr int GM_HALF = 64 * 128;                 // a 64 x 64 bf16 box
constexpr int GM_OPERAND = 2 * GM_HALF;           // the A operand's k-chunk of a tile
constexpr int GM_THREADS = 192;                   // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int GM_STAGING = 2 * 2048;              // per epilogue warp: two 32-row x 64-byte store boxes
template <int BN> struct GmTile {
  static constexpr int STAGES = BN == 256 ? 4 : 6;
  static constexpr int B_BYTES = BN / 64 * GM_HALF;    // the B operand's k-chunk
  static constexpr int STAGE = GM_OPERAND + B_BYTES;
  // + alignment slack, each epilogue warp's two 2 KB store staging buffers,
  // barriers (256 B), each epilogue warp's copy of the tile's bias row (fp32)
  static constexpr int SMEM = STAGES * STAGE + 1024 + 4 * GM_STAGING + 256 + 4 * BN * 4;
};

// K-major (128-byte swizzle): 8-row groups 1 KB apart, a 16-element k step is
// 32 bytes further along the 128-byte row. MN-major: the two 64-wide halves of
// the tile 8 KB apart, 8-row k groups 1 KB apart, a 16-row k step is 2 KB.
__device__ __forceinline__ uint64_t gm_desc(uint32_t base, bool kmajor, int k16) {
  const uint32_t addr = base + (uint32_t)(kmajor ? k16 * 32 : k16 * 2048);
  const uint32_t lbo = kmajor ? 16u : (uint32_t)GM_HALF;
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (lane = row)
__device__ __forceinline__ void tmem_ld32(uint32_t* r, uint32_t taddr) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

struct GemmArgs {
  int M, N, K;
  int splits, kps;          // k-chunks of 64 per split
  __nv_bfloat16* C;         // [M][N] bf16 (splits == 1)
  float* partial;           // [splits][M][N] fp32 (splits > 1)
  const __nv_bfloat16* bias;  // [N] or null (splits == 1 only)
  unsigned int* status;
  unsigned long long wait_limit_ns;
};

template <bool AK, bool BK, int BN>
__global__ void __launch_bounds__(GM_THREADS, 1)
    gemm_umma_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                     const __grid_constant__ CUtensorMap cmap, GemmArgs a) {
  constexpr int NS = GmTile<BN>::STAGES, STAGE = GmTile<BN>::STAGE;
  extern __shared__ unsigned char gm_raw[];
  unsigned char* sm = (unsigned char*)(((uintptr_t)gm_raw + 1023) & ~(uintptr_t)1023);
  // full[NS], empty[NS], accumulator full[2], accumulator empty[2], final
  unsigned char* staging = sm + NS * STAGE;  // [4][2][2 KB], 1 KB aligned (64-byte swizzle)
  uint64_t* bars = (uint64_t*)(staging + 4 * GM_STAGING);
  uint32_t* tslot = (uint32_t*)(bars + 2 * NS + 5);
  float* bias_sm = (float*)(staging + 4 * GM_STAGING + 256);  // [4][BN]: the epilogue warps' bias rows
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[NS]);
  const uint32_t accf0 = smem_u32(&bars[2 * NS]), acce0 = accf0 + 16, finb = accf0 + 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mtiles = (a.M + GM_TILE - 1) / GM_TILE, ntiles = (a.N + BN - 1) / BN;
  const int units = mtiles * ntiles * a.splits;
  const int nchunk = (a.K + GM_BK - 1) / GM_BK;
  // unit u: split-K slice u / (mtiles ntiles), then m-tile, then n-tile
  // fastest, so the CTAs working side by side share A tiles through L2
  auto decode = [&](int u, int& m0, int& n0, int& c0, int& nq, int& split) {
    split = u / (mtiles * ntiles);
    const int r = u - split * mtiles * ntiles, mt = r / ntiles;
    m0 = mt * GM_TILE;
    n0 = (r - mt * ntiles) * BN;
    c0 = split * a.kps;
    nq = min(nchunk, c0 + a.kps) - c0;
  };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 4);  // one arrival per epilogue warp
    }
    mbar_init(finb, 1);
    fence_mbar_init_cluster();
    prefetch_tensormap(&amap);
    prefetch_tensormap(&bmap);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "n"(2 * BN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tslot;
  bool failed = false;

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer
      int it = 0, issued = 0;
      for (int u = blockIdx.x; u < units && !failed; u += gridDim.x) {
        int m0, n0, c0, nq, split;
        decode(u, m0, n0, c0, nq, split);
        for (int q = 0; q < nq; ++q, ++it) {
          const int s = it % NS;
          if (it >= NS &&
              !mbar_wait_bounded<false>(empty0 + 8 * s, ((it / NS) - 1) & 1, a.wait_limit_ns, a.status, failed))
            break;
          const uint32_t fb = full0 + 8 * s;
          unsigned char* As = sm + (size_t)s * STAGE;
          unsigned char* Bs = As + GM_OPERAND;
          const int k0 = (c0 + q) * GM_BK;
          mbar_arrive_expect_tx(fb, STAGE);
          if constexpr (AK) {  // rows m0 .. m0+127, k0 .. k0+63
            tma_load_5d(smem_u32(As), &amap, fb, k0, m0, 0, 0, 0);
          } else {             // two 64-wide m halves, k rows k0 .. k0+63
            tma_load_5d(smem_u32(As), &amap, fb, m0, k0, 0, 0, 0);
            tma_load_5d(smem_u32(As + GM_HALF), &amap, fb, m0 + 64, k0, 0, 0, 0);
          }
          if constexpr (BK) {  // BN rows n0 .. n0+BN-1, k0 .. k0+63
            tma_load_5d(smem_u32(Bs), &bmap, fb, k0, n0, 0, 0, 0);
          } else {             // BN/64 column groups of 64, k rows k0 .. k0+63
#pragma unroll
            for (int h = 0; h < BN / 64; ++h)
              tma_load_5d(smem_u32(Bs + h * GM_HALF), &bmap, fb, n0 + 64 * h, k0, 0, 0, 0);
          }
          issued = it + 1;
        }
      }
      if (failed) {  // let the copies in flight land before the CTA exits
        for (int i = issued - NS > 0 ? issued - NS : 0; i < issued; ++i) {
          bool f2 = false;
          mbar_wait_bounded<false>(full0 + 8 * (i % NS), (i / NS) & 1, a.wait_limit_ns, nullptr, f2);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((AK ? 0u : 1u) << 15) | ((BK ? 0u : 1u) << 16) |
                             ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(GM_TILE >> 4) << 24);
      int it = 0, tc = 0;
      for (int u = blockIdx.x; u < units && !failed; u += gridDim.x, ++tc) {
        int m0, n0, c0, nq, split;
        decode(u, m0, n0, c0, nq, split);
        const int b = tc & 1;
        // the epilogue of tile tc - 2 has drained accumulator b
        if (tc >= 2) mbar_wait_bounded<false>(acce0 + 8 * b, ((tc >> 1) - 1) & 1, a.wait_limit_ns, a.status, failed);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t dacc = tmem + (uint32_t)(b * BN);
        for (int q = 0; q < nq; ++q, ++it) {
          const int s = it % NS;
          mbar_wait_bounded<false>(full0 + 8 * s, (it / NS) & 1, a.wait_limit_ns, a.status, failed);
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t As = smem_u32(sm + (size_t)s * STAGE), Bs = As + GM_OPERAND;
          if (!failed) {
#pragma unroll
            for (int k = 0; k < GM_BK / 16; ++k) {
              const uint64_t ad = gm_desc(As, AK, k), bd = gm_desc(Bs, BK, k);
              const uint32_t acc = (q | k) ? 1u : 0u;
              asm volatile(
                  "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                  " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(dacc),
                  "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
                  : "memory");
            }
          }
          asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                           empty0 + 8 * s)
                       : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(accf0 + 8 * b)
                     : "memory");
      }
      // every MMA this thread issued has completed once this arrives
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(finb) : "memory");
      bool f2 = false;
      mbar_wait_bounded<false>(finb, 0, a.wait_limit_ns, nullptr, f2);
    }
  } else {  // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 = tile rows
    const int ew = warp & 3;
    float* bsm = bias_sm + ew * BN;
    unsigned char* stg = staging + ew * GM_STAGING;
    int sbuf = 0, tc = 0;
    // each warp keeps the tile's BN bias values in shared memory (read by
    // every row) and the next tile's in registers (loaded one tile ahead)
    float bv[BN / 32];
    auto load_bias = [&](int nb0) {
#pragma unroll
      for (int q = 0; q < BN / 32; ++q) {
        const int c = nb0 + lane + 32 * q;
        bv[q] = c < a.N ? __bfloat162float(__ldg(a.bias + c)) : 0.0f;
      }
    };
    if (a.bias && (int)blockIdx.x < units) {
      int m1, n1, c1, q1, s1;
      decode(blockIdx.x, m1, n1, c1, q1, s1);
      load_bias(n1);
    }
    for (int u = blockIdx.x; u < units && !failed; u += gridDim.x, ++tc) {
      int m0, n0, c0, nq, split;
      decode(u, m0, n0, c0, nq, split);
      const int b = tc & 1;
      mbar_wait_bounded<false>(accf0 + 8 * b, (tc >> 1) & 1, a.wait_limit_ns, a.status, failed);
      failed = __any_sync(0xffffffffu, failed);  // the warp leaves the loop together
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (a.bias) {
        __syncwarp();  // the previous tile's reads of bsm are done
#pragma unroll
        for (int q = 0; q < BN / 32; ++q) bsm[lane + 32 * q] = bv[q];
        __syncwarp();
        // the next tile's bias, in flight while this tile drains
        const int un = u + gridDim.x;
        if (un < units) {
          int m1, n1, c1, q1, s1;
          decode(un, m1, n1, c1, q1, s1);
          load_bias(n1);
        }
      }
      // Each 32-column chunk of the warp's 32 rows goes out through shared
      // memory as TMA stores (one 32 x 32 bf16 box, or two 32 x 16 fp32 boxes
      // of split-K partials) from alternating staging buffers; TMA clips the
      // boxes at the matrix edges.
      // The TMEM read of the next 32-column chunk is in flight while this one
      // is converted and stored.
      const uint32_t trow = tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)(b * BN);
      auto emit = [&](const uint32_t* r, int cc) {
        if (n0 + cc >= a.N || m0 + ew * 32 >= a.M || failed) return;  // boxes start inside the matrix
        const int nbox = a.splits == 1 ? 1 : 2;
        for (int h = 0; h < nbox; ++h) {
          if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous box has been read
          __syncwarp();
          // this lane's row: 64 bytes, its 16-byte pieces in the 64-byte
          // swizzle the store's tensor map reads (piece v at v ^ (row / 2) % 4)
          uint4* dst = (uint4*)(stg + sbuf * 2048 + lane * 64);
          const int sw = (lane >> 1) & 3;
          if (a.splits == 1) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float f[8];
#pragma unroll
              for (int q = 0; q < 8; ++q) f[q] = __uint_as_float(r[8 * v + q]);
              if (a.bias) {
                const float4 b0 = *(const float4*)(bsm + cc + 8 * v), b1 = *(const float4*)(bsm + cc + 8 * v + 4);
                f[0] += b0.x; f[1] += b0.y; f[2] += b0.z; f[3] += b0.w;
                f[4] += b1.x; f[5] += b1.y; f[6] += b1.z; f[7] += b1.w;
              }
              uint4 w;
              w.x = pack_bf16(__float2bfloat16_rn(f[0]), __float2bfloat16_rn(f[1]));
              w.y = pack_bf16(__float2bfloat16_rn(f[2]), __float2bfloat16_rn(f[3]));
              w.z = pack_bf16(__float2bfloat16_rn(f[4]), __float2bfloat16_rn(f[5]));
              w.w = pack_bf16(__float2bfloat16_rn(f[6]), __float2bfloat16_rn(f[7]));
              dst[v ^ sw] = w;
            }
          } else {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v ^ sw] = h == 0 ? make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3])
                                   : make_uint4(r[16 + 4 * v], r[17 + 4 * v], r[18 + 4 * v], r[19 + 4 * v]);
          }
          fence_proxy_async_smem();  // the generic writes above are read by the TMA store
          __syncwarp();
          if (lane == 0) {
            const uint32_t src = smem_u32(stg + sbuf * 2048);
            if (a.splits == 1)
              tma_store_5d(&cmap, src, n0 + cc, m0 + ew * 32, 0, 0, 0);
            else
              tma_store_5d(&cmap, src, n0 + cc + 16 * h, m0 + ew * 32, split, 0, 0);
            bulk_commit_group();
          }
          sbuf ^= 1;
        }
      };
      uint32_t ra[32], rb[32];
      tmem_ld32(ra, trow);
      tmem_wait_ld();
#pragma unroll 1
      for (int cc = 0; cc < BN; cc += 64) {
        tmem_ld32(rb, trow + (uint32_t)(cc + 32));
        emit(ra, cc);
        tmem_wait_ld();
        if (cc + 64 < BN) tmem_ld32(ra, trow + (uint32_t)(cc + 64));
        emit(rb, cc + 32);
        tmem_wait_ld();
      }
      // accumulator b is free for tile tc + 2
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(acce0 + 8 * b);
    }
    if (lane == 0) bulk_wait_group_all();  // every store has landed before the CTA retires
    __syncwarp();
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(2 * BN) : "memory");
  }
}

// Sum of the split-K partials in a fixed order, rounded to bf16.
__global__ void gemm_reduce_kernel(const float* partial, __nv_bfloat16* C, size_t MN, int splits) {
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < MN; e += (size_t)gridDim.x * blockDim.x) {
    float s = 0.0f;
    for (int k = 0; k < splits; ++k) s += partial[(size_t)k * MN + e];
    C[e] = __float2bfloat16_rn(s);
  }
}

// Column sums of a [rows][cols] bf16 matrix (dbias = sum over m of dWx[m, c]).
__global__ void colsum_kernel(const __nv_bfloat16* X, __nv_bfloat16* out, int rows, int cols) {
  __shared__ float part[32][33];
  const int c = blockIdx.x * 32 + (threadIdx.x & 31), ks = threadIdx.x >> 5;
  float s = 0.0f;
  if (c < cols)
    for (int r = ks; r < rows; r += 32) s += __bfloat162float(X[(size_t)r * cols + c]);
  part[ks][threadIdx.x & 31] = s;
  __syncthreads();
  if (ks == 0 && c < cols) {
    float tot = 0.0f;
    for (int q = 0; q < 32; ++q) tot += part[q][threadIdx.x & 31];
    out[c] = __float2bfloat16_rn(tot);
  }
}


// Tile width and split-K count of one GEMM, from a small cost model of the
// persistent kernel on the device's SMs: the time is the number of waves of work units
// times one unit's MMA cycles (128 x BN x 64 per k-chunk at about 2300 MACs
// per cycle and SM; a 128-wide tile at 85% of a 256-wide one's rate), plus,
// with split-K, the fp32 partials written and read back (8 bytes per output
// and split at about 2900 bytes per cycle).
struct Tiling {
  int BN, splits, kps;
};
Tiling choose_tiling(int M, int N, int K, bool split_ok) {
  const int sms = device_sms(), nchunk = (K + GM_BK - 1) / GM_BK;
  Tiling best{N >= 256 ? 256 : 128, 1, nchunk};
  double best_cost = 1e300;
  for (int BN = 256; BN >= 128; BN -= 128) {
    if (BN == 256 && N < 256) continue;
    const double tiles = (double)((M + GM_TILE - 1) / GM_TILE) * ((N + BN - 1) / BN);
    const int smax = split_ok ? (nchunk / 2 < 32 ? nchunk / 2 : 32) : 1;
    for (int sp = 1; sp <= (smax < 1 ? 1 : smax); ++sp) {
      const int kps = (nchunk + sp - 1) / sp, se = (nchunk + kps - 1) / kps;
      const double waves = std::ceil(tiles * se / sms);
      double cost = waves * GM_TILE * BN * kps * GM_BK / (2300.0 * (BN == 256 ? 1.0 : 0.85));
      if (se > 1) cost += 8.0 * se * M * N / 2900.0;
      if (cost < best_cost * 0.999) {
        best_cost = cost;
        best = Tiling{BN, se, kps};
      }
    }
  }
  return best;
}

// D[M][N] = A(m, k) B(k, n); a_kmajor: A stored [M][K] (else [K][M]); b_kmajor:
// B stored [N][K] (else [K][N]).
cudaError_t gemm_run(bool a_kmajor, bool b_kmajor, int M, int N, int K, const void* A, const void* B,
                     const void* bias, void* C, float* scratch, size_t scratch_bytes, unsigned int* status,
                     cudaStream_t st) {
  CUtensorMap am, bm;
  cudaError_t e;
  {
    const unsigned long long dims_k[5] = {(unsigned long long)K, (unsigned long long)M, 1, 1, 1};
    const unsigned long long dims_m[5] = {(unsigned long long)M, (unsigned long long)K, 1, 1, 1};
    const unsigned int box_k[5] = {64, 128, 1, 1, 1}, box_m[5] = {64, 64, 1, 1, 1};
    e = encode_tensor_map_sw128(&am, A, 5, a_kmajor ? dims_k : dims_m, a_kmajor ? box_k : box_m);
    if (e != cudaSuccess) return e;
  }
  Tiling tl = choose_tiling(M, N, K, !bias && scratch);
  if (tl.splits > 1 && scratch_bytes < (size_t)tl.splits * M * N * sizeof(float)) tl = choose_tiling(M, N, K, false);
  const int BN = tl.BN;
  {
    const unsigned long long dims_k[5] = {(unsigned long long)K, (unsigned long long)N, 1, 1, 1};
    const unsigned long long dims_n[5] = {(unsigned long long)N, (unsigned long long)K, 1, 1, 1};
    const unsigned int box_k[5] = {64, (unsigned)BN, 1, 1, 1}, box_n[5] = {64, 64, 1, 1, 1};
    e = encode_tensor_map_sw128(&bm, B, 5, b_kmajor ? dims_k : dims_n, b_kmajor ? box_k : box_n);
    if (e != cudaSuccess) return e;
  }
  // the output: C [M][N] bf16 in 32 x 32 boxes, or the split-K partials
  // [splits][M][N] fp32 in 16-column x 32-row boxes (one split per plane)
  CUtensorMap cm;
  if (tl.splits == 1) {
    const unsigned long long dims[5] = {(unsigned long long)N, (unsigned long long)M, 1, 1, 1};
    const unsigned int box[5] = {32, 32, 1, 1, 1};
    e = encode_tensor_map_swizzled(&cm, C, 2, 5, dims, box, 64);
  } else {
    const unsigned long long dims[5] = {(unsigned long long)N, (unsigned long long)M, (unsigned long long)tl.splits,
                                        1, 1};
    const unsigned int box[5] = {16, 32, 1, 1, 1};
    e = encode_tensor_map_swizzled(&cm, scratch, 4, 5, dims, box, 64);
  }
  if (e != cudaSuccess) return e;
  const int tiles = ((M + GM_TILE - 1) / GM_TILE) * ((N + BN - 1) / BN);
  GemmArgs g{};
  g.M = M; g.N = N; g.K = K;
  g.kps = tl.kps;
  g.splits = tl.splits;
  g.C = (__nv_bfloat16*)C;
  g.partial = scratch;
  g.bias = (const __nv_bfloat16*)bias;
  g.status = status;
  g.wait_limit_ns = wait_limit_ns();
  void (*k)(const CUtensorMap, const CUtensorMap, const CUtensorMap, GemmArgs);
  if (BN == 256)
    k = a_kmajor ? (b_kmajor ? gemm_umma_kernel<true, true, 256> : gemm_umma_kernel<true, false, 256>)
                 : (b_kmajor ? gemm_umma_kernel<false, true, 256> : gemm_umma_kernel<false, false, 256>);
  else
    k = a_kmajor ? (b_kmajor ? gemm_umma_kernel<true, true, 128> : gemm_umma_kernel<true, false, 128>)
                 : (b_kmajor ? gemm_umma_kernel<false, true, 128> : gemm_umma_kernel<false, false, 128>);
  const int smem = BN == 256 ? GmTile<256>::SMEM : GmTile<128>::SMEM;
  e = set_smem_attr((const void*)k, (size_t)smem);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (the shared-memory ring and the two
  // accumulators take the whole SM), never more CTAs than work units
  const int units = tiles * g.splits;
  const int ctas = units < device_sms() ? units : device_sms();
  k<<<ctas, GM_THREADS, smem, st>>>(am, bm, cm, g);
  note_launch();
  if (g.splits > 1) {
    gemm_reduce_kernel<<<2 * device_sms(), 256, 0, st>>>(scratch, (__nv_bfloat16*)C, (size_t)M * N, g.splits);
    note_launch();
  }
  return cudaGetLastError();
}

int proj_splits_bound(int M, int N, int K) { return choose_tiling(M, N, K, true).splits; }

bool proj_dims_ok(int BT, int I, int C) {
  // TMA: 16-byte row strides (I, C multiples of 8); boxes of 64 along I and C
  return BT >= 1 && I >= 64 && C >= 64 && I % 8 == 0 && C % 8 == 0;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return RNN_OK;
  fprintf(stderr, "librnn_gb300: CUDA error: %s\n", cudaGetErrorString(e));
  return RNN_ECUDA;
}

bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

}  // namespace rnn

using namespace rnn;

extern "C" {

size_t rnn_input_proj_workspace_size(int BT, int I, int C) {
  if (!proj_dims_ok(BT, I, C)) return 0;
  const int s = proj_splits_bound(C, I, BT);  // dW_x: M = C, N = I, K = B T
  const size_t dW_part = s > 1 ? (size_t)s * C * I * sizeof(float) : 0;
  const size_t db_part = colsum_scratch_bytes(BT, C);  // the dbias partials, after dW_x
  return 256 + (dW_part > db_part ? dW_part : db_part);
}

int rnn_input_proj_fwd(int BT, int I, int C, const void* x, const void* W, const void* bias, void* Wx,
                       void* workspace, size_t ws_bytes, void* stream) {
  if (!proj_dims_ok(BT, I, C) || !x || !W || !Wx || !workspace) return RNN_EINVAL;
  if (!al16(x) || !al16(W) || !al16(Wx) || !al16(workspace) || (bias && !al16(bias))) return RNN_EINVAL;
  if (ws_bytes < rnn_input_proj_workspace_size(BT, I, C)) return RNN_ENOSPC;
  cudaStream_t st = (cudaStream_t)stream;
  int rc = cuda_status(cudaMemsetAsync(workspace, 0, 256, st));
  if (rc) return rc;
  // Wx[m, c] = x[m, :] . W_x[c, :]: A = x [BT][I] (K-major), B = W_x [C][I] (K-major)
  return cuda_status(gemm_run(true, true, BT, C, I, x, W, bias, Wx, nullptr, 0, (unsigned int*)workspace, st));
}

int rnn_input_proj_bwd(int BT, int I, int C, const void* x, const void* W, const void* dWx, void* dx, void* dW,
                       void* dbias, void* workspace, size_t ws_bytes, void* stream) {
  if (!proj_dims_ok(BT, I, C) || !x || !W || !dWx || !workspace) return RNN_EINVAL;
  const void* ptrs[] = {x, W, dWx, dx, dW, dbias, workspace};
  for (const void* p : ptrs)
    if (p && !al16(p)) return RNN_EINVAL;
  if (ws_bytes < rnn_input_proj_workspace_size(BT, I, C)) return RNN_ENOSPC;
  cudaStream_t st = (cudaStream_t)stream;
  int rc = cuda_status(cudaMemsetAsync(workspace, 0, 256, st));
  if (rc) return rc;
  unsigned int* status = (unsigned int*)workspace;
  if (dx) {  // dx[m, i] = dWx[m, :] . W_x[:, i]: A = dWx [BT][C] (K-major), B = W_x [C][I] (MN-major)
    rc = cuda_status(gemm_run(true, false, BT, I, C, dWx, W, nullptr, dx, nullptr, 0, status, st));
    if (rc) return rc;
  }
  if (dW) {  // dW_x[c, i] = sum_m dWx[m, c] x[m, i]: A = dWx (MN-major), B = x [BT][I] (MN-major)
    float* scratch = (float*)((char*)workspace + 256);
    rc = cuda_status(gemm_run(false, false, C, I, BT, dWx, x, nullptr, dW, scratch, ws_bytes - 256, status, st));
    if (rc) return rc;
  }
  if (dbias) {
    float* scratch = (float*)((char*)workspace + 256);
    if (!colsum_bf16((const __nv_bfloat16*)dWx, (__nv_bfloat16*)dbias, BT, C, scratch, ws_bytes - 256, st)) {
      colsum_kernel<<<(C + 31) / 32, 1024, 0, st>>>((const __nv_bfloat16*)dWx, (__nv_bfloat16*)dbias, BT, C);
      note_launch();
    }
    rc = cuda_status(cudaGetLastError());
  }
  return rc;
}

}  // extern "C"
