// Instantiation of the forward cluster kernels for one cell type (one
// translation unit per cell keeps the parallel build short).
#include "fused_fwd.cuh"

namespace rnn {
template cudaError_t fused_fwd_launch<ELMAN>(const FusedShape&, const FusedArgs&, cudaStream_t);
}  // namespace rnn
