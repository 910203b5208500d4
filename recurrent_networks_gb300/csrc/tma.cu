// TMA descriptor encoding and the per-cell dispatch of the cluster kernels.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "layout.h"

namespace rnn {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

cudaError_t encode_tensor_map_sw128(void* map, const void* base, int rank, const unsigned long long* dims,
                                    const unsigned int* box) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn || rank < 1 || rank > 5 || box[0] * 2 > 128) return cudaErrorNotSupported;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estr[5];
  unsigned long long stride = 2;  // bytes
  for (int d = 0; d < rank; ++d) {
    gdim[d] = dims[d];
    bdim[d] = box[d];
    estr[d] = 1;
    if (d > 0) gstride[d - 1] = stride;
    stride *= dims[d];
  }
  CUresult r = fn((CUtensorMap*)map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, (void*)base, gdim, gstride,
                  bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_tensor_map_sw128_strided(void* map, const void* base, int rank, const unsigned long long* dims,
                                            const unsigned long long* strides, const unsigned int* box) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn || rank < 2 || rank > 5 || box[0] * 2 > 128) return cudaErrorNotSupported;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estr[5];
  for (int d = 0; d < rank; ++d) {
    gdim[d] = dims[d];
    bdim[d] = box[d];
    estr[d] = 1;
    if (d > 0) gstride[d - 1] = strides[d - 1];
  }
  CUresult r = fn((CUtensorMap*)map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, (void*)base, gdim, gstride,
                  bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_tensor_map(void* map, const void* base, int elem_bytes, int rank,
                              const unsigned long long* dims, const unsigned int* box) {
  return encode_tensor_map_swizzled(map, base, elem_bytes, rank, dims, box, 0);
}

cudaError_t encode_tensor_map_swizzled(void* map, const void* base, int elem_bytes, int rank,
                                       const unsigned long long* dims, const unsigned int* box, int swizzle_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn || rank < 1 || rank > 5 || (elem_bytes != 2 && elem_bytes != 4)) return cudaErrorNotSupported;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estr[5];
  unsigned long long stride = (unsigned long long)elem_bytes;  // bytes
  for (int d = 0; d < rank; ++d) {
    gdim[d] = dims[d];
    bdim[d] = box[d];
    estr[d] = 1;
    if (d > 0) gstride[d - 1] = stride;
    stride *= dims[d];
  }
  const CUtensorMapDataType ty =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const CUtensorMapSwizzle sw = swizzle_bytes == 64    ? CU_TENSOR_MAP_SWIZZLE_64B
                                : swizzle_bytes == 32  ? CU_TENSOR_MAP_SWIZZLE_32B
                                : swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                       : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = fn((CUtensorMap*)map, ty, (cuuint32_t)rank, (void*)base, gdim,
                  gstride, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_tensor_map_bf16(void* map, const void* base, int rank, const unsigned long long* dims,
                                   const unsigned int* box) {
  return encode_tensor_map(map, base, 2, rank, dims, box);
}

template <int FN>
cudaError_t fused_fwd_launch(const FusedShape&, const FusedArgs&, cudaStream_t);
template <int FN>
cudaError_t fused_bwd_launch(const FusedShape&, const FusedArgs&, cudaStream_t);

cudaError_t fused_bwd_run(int fn, const FusedShape& sh, const FusedArgs& a, cudaStream_t st) {
  switch (fn) {
    case LSTM: return fused_bwd_launch<LSTM>(sh, a, st);
    case GRU: return fused_bwd_launch<GRU>(sh, a, st);
    case ELMAN: return fused_bwd_launch<ELMAN>(sh, a, st);
    case SLSTM: return fused_bwd_launch<SLSTM>(sh, a, st);
    case SLSTM_LS: return fused_bwd_launch<SLSTM_LS>(sh, a, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t fused_fwd_run(int fn, const FusedShape& sh, const FusedArgs& a, cudaStream_t st) {
  switch (fn) {
    case LSTM: return fused_fwd_launch<LSTM>(sh, a, st);
    case GRU: return fused_fwd_launch<GRU>(sh, a, st);
    case ELMAN: return fused_fwd_launch<ELMAN>(sh, a, st);
    case SLSTM: return fused_fwd_launch<SLSTM>(sh, a, st);
    case SLSTM_LS: return fused_fwd_launch<SLSTM_LS>(sh, a, st);
  }
  return cudaErrorInvalidValue;
}

template <int FN>
int fused_fwd_capacity(const FusedShape&);
template <int FN>
int fused_bwd_capacity(const FusedShape&);

int fused_capacity(int fn, bool bwd, const FusedShape& sh) {
  switch (fn) {
    case LSTM: return bwd ? fused_bwd_capacity<LSTM>(sh) : fused_fwd_capacity<LSTM>(sh);
    case GRU: return bwd ? fused_bwd_capacity<GRU>(sh) : fused_fwd_capacity<GRU>(sh);
    case ELMAN: return bwd ? fused_bwd_capacity<ELMAN>(sh) : fused_fwd_capacity<ELMAN>(sh);
    case SLSTM: return bwd ? fused_bwd_capacity<SLSTM>(sh) : fused_fwd_capacity<SLSTM>(sh);
    case SLSTM_LS: return bwd ? fused_bwd_capacity<SLSTM_LS>(sh) : fused_fwd_capacity<SLSTM_LS>(sh);
  }
  return 0;
}

template <int FN>
cudaError_t grid_fwd_launch(const FusedShape&, const FusedArgs&, cudaStream_t);
template <int FN>
cudaError_t grid_bwd_launch(const FusedShape&, const FusedArgs&, cudaStream_t, const UmmaMaps*);

cudaError_t grid_fwd_run(int fn, const FusedShape& sh, const FusedArgs& a, cudaStream_t st) {
  switch (fn) {
    case LSTM: return grid_fwd_launch<LSTM>(sh, a, st);
    case GRU: return grid_fwd_launch<GRU>(sh, a, st);
    case ELMAN: return grid_fwd_launch<ELMAN>(sh, a, st);
    case SLSTM: return grid_fwd_launch<SLSTM>(sh, a, st);
    case SLSTM_LS: return grid_fwd_launch<SLSTM_LS>(sh, a, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t grid_bwd_run(int fn, const FusedShape& sh, const FusedArgs& a, cudaStream_t st, const UmmaMaps* dmaps) {
  switch (fn) {
    case LSTM: return grid_bwd_launch<LSTM>(sh, a, st, dmaps);
    case GRU: return grid_bwd_launch<GRU>(sh, a, st, dmaps);
    case ELMAN: return grid_bwd_launch<ELMAN>(sh, a, st, dmaps);
    case SLSTM: return grid_bwd_launch<SLSTM>(sh, a, st, dmaps);
    case SLSTM_LS: return grid_bwd_launch<SLSTM_LS>(sh, a, st, dmaps);
  }
  return cudaErrorInvalidValue;
}

}  // namespace rnn
