// Instantiation of the backward cluster kernels for one cell type.
#include "fused_bwd.cuh"

namespace rnn {
template cudaError_t fused_bwd_launch<GRU>(const FusedShape&, const FusedArgs&, cudaStream_t);
template int fused_bwd_capacity<GRU>(const FusedShape&);
}  // namespace rnn
