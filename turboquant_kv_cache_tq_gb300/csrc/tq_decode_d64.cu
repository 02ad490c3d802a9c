// Decode kernels for head_dim 64 (one translation unit per head_dim and
// direction, so the library builds in parallel).
#include "tq_kernels.cuh"

namespace tq {
template cudaError_t launch_decode<64>(const DecodeParams&, int, bool, bool, cudaStream_t);
template cudaError_t launch_unrotate<64>(const UnrotateParams&, bool, cudaStream_t);
}  // namespace tq
