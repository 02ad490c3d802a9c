// Encode kernels for head_dim 256 (one translation unit per head_dim and
// direction, so the library builds in parallel).
#include "tq_kernels.cuh"

namespace tq {
template cudaError_t launch_encode<256>(const EncodeParams&, int, bool, cudaStream_t);
}  // namespace tq
