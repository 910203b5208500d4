// Instantiation of the grid backward kernels for one cell type.
#include "grid_bwd.cuh"

namespace rnn {
template cudaError_t grid_bwd_launch<ELMAN>(const FusedShape&, const FusedArgs&, cudaStream_t, const UmmaMaps*);
}  // namespace rnn
