// Instantiation of the forward persistent kernels (cluster and grid variants)
// for one cell type (one translation unit per cell keeps the build parallel).
#include "fused_fwd.cuh"

namespace rnn {
template cudaError_t fused_fwd_launch<ELMAN>(const FusedShape&, const FusedArgs&, cudaStream_t);
template cudaError_t grid_fwd_launch<ELMAN>(const FusedShape&, const FusedArgs&, cudaStream_t);
template int fused_fwd_capacity<ELMAN>(const FusedShape&);
}  // namespace rnn
