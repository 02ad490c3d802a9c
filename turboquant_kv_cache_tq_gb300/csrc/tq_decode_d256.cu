// Decode kernels for head_dim 256 (one translation unit per head_dim and
// direction, so the library builds in parallel).
#include "tq_kernels.cuh"

namespace tq {
template cudaError_t launch_decode<256>(const DecodeParams&, int, bool, bool, cudaStream_t);
template cudaError_t launch_unrotate<256>(const UnrotateParams&, bool, cudaStream_t);
}  // namespace tq
