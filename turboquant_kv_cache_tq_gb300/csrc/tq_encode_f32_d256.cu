// Encode kernels for head_dim 256, fp32 inputs (one translation unit per
// head_dim, direction and input type, so the library builds in parallel).
#include "tq_kernels.cuh"

namespace tq {
template cudaError_t launch_encode_dt<256, true>(const EncodeParams&, int, cudaStream_t);
}  // namespace tq
