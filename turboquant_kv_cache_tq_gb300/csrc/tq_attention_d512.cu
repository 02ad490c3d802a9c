// Fused decode attention kernels for head_dim 512 (one translation unit per
// head_dim, so the library builds in parallel).
#include "tq_attention.cuh"

namespace tq {
template cudaError_t launch_attention<512>(const AttnParams&, int, int, bool, cudaStream_t);
}  // namespace tq
