// Column sums of a bf16 matrix [rows][cols] into bf16, in two deterministic
// passes over 16-byte loads. Pass 1: block (x, y) sums rows [y rpc, (y+1) rpc)
// of 256 columns (8 per thread, 8 row lanes, four rows in flight per lane)
// into fp32 partial[y][cols]. Pass 2 adds each column's partials in eight
// interleaved lanes, then the lanes in order. Both orders are fixed, so the
// result does not depend on timing.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.cuh"

namespace rnn {
namespace {  // each including translation unit has its own copy of the kernels

constexpr int COLSUM_MAX_CHUNKS = 64;
inline int colsum_chunks(int rows, int cols) {
  const int colblocks = (cols + 255) / 256;
  int c = (4 * device_sms() + colblocks - 1) / colblocks;  // about four blocks per SM
  if (c > COLSUM_MAX_CHUNKS) c = COLSUM_MAX_CHUNKS;
  if (c > (rows + 31) / 32) c = (rows + 31) / 32;  // at least 32 rows per chunk
  return c < 1 ? 1 : c;
}
// fp32 scratch the two passes need
inline size_t colsum_scratch_bytes(int rows, int cols) {
  return (size_t)colsum_chunks(rows, cols) * cols * sizeof(float);
}

__global__ void __launch_bounds__(256) colsum_partial_kernel(const __nv_bfloat16* X, float* partial, int rows,
                                                             int cols, int rpc) {
  __shared__ float red[8][256];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int c0 = blockIdx.x * 256 + tx * 8;
  const int r0 = blockIdx.y * rpc, r1 = min(rows, r0 + rpc);
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
  auto add = [&](const uint4& v) {
    const __nv_bfloat16* h = (const __nv_bfloat16*)&v;
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] += __bfloat162float(h[q]);
  };
  if (c0 < cols) {  // cols is a multiple of 8: the 8 columns are all inside
    const __nv_bfloat16* p = X + c0;
    int r = r0 + ty;
    for (; r + 24 < r1; r += 32) {
      const uint4 v0 = *(const uint4*)(p + (size_t)r * cols), v1 = *(const uint4*)(p + (size_t)(r + 8) * cols);
      const uint4 v2 = *(const uint4*)(p + (size_t)(r + 16) * cols), v3 = *(const uint4*)(p + (size_t)(r + 24) * cols);
      add(v0);
      add(v1);
      add(v2);
      add(v3);
    }
    for (; r < r1; r += 8) add(*(const uint4*)(p + (size_t)r * cols));
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) red[ty][tx * 8 + q] = acc[q];
  __syncthreads();
  if (ty == 0 && c0 < cols) {
    float t[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float v = 0.0f;
#pragma unroll
      for (int y = 0; y < 8; ++y) v += red[y][tx * 8 + q];
      t[q] = v;
    }
    float* out = partial + (size_t)blockIdx.y * cols + c0;
    *(float4*)out = make_float4(t[0], t[1], t[2], t[3]);
    *(float4*)(out + 4) = make_float4(t[4], t[5], t[6], t[7]);
  }
}

// 32 columns per block, 8 lanes each summing chunks k = lane, lane + 8, ...,
// then the 8 lane sums in lane order
__global__ void __launch_bounds__(256) colsum_final_kernel(const float* partial, __nv_bfloat16* out, int cols,
                                                           int chunks) {
  __shared__ float red[8][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + tx;
  float v = 0.0f;
  if (c < cols)
    for (int k = ty; k < chunks; k += 8) v += partial[(size_t)k * cols + c];
  red[ty][tx] = v;
  __syncthreads();
  if (ty == 0 && c < cols) {
    float t = 0.0f;
#pragma unroll
    for (int y = 0; y < 8; ++y) t += red[y][tx];
    out[c] = __float2bfloat16_rn(t);
  }
}

// Launches both passes on st and returns true, or returns false (launching
// nothing) when cols is not a multiple of 8, X is not 16-byte aligned or the
// scratch is too small.
inline bool colsum_bf16(const __nv_bfloat16* X, __nv_bfloat16* out, int rows, int cols, float* scratch,
                        size_t scratch_bytes, cudaStream_t st) {
  if (rows < 1 || cols % 8 != 0 || ((uintptr_t)X & 15) != 0 || !scratch ||
      scratch_bytes < colsum_scratch_bytes(rows, cols))
    return false;
  const int chunks = colsum_chunks(rows, cols);
  const int rpc = (rows + chunks - 1) / chunks;
  const int used = (rows + rpc - 1) / rpc;  // chunks that hold rows
  colsum_partial_kernel<<<dim3((cols + 255) / 256, used), 256, 0, st>>>(X, scratch, rows, cols, rpc);
  note_launch();
  colsum_final_kernel<<<(cols + 31) / 32, 256, 0, st>>>(scratch, out, cols, used);
  note_launch();
  return true;
}

}  // namespace
}  // namespace rnn
