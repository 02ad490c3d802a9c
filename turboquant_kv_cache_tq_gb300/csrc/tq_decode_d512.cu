// Decode kernels for head_dim 512, bf16 outputs, and the unrotate kernel (one
// translation unit per head_dim, direction and type, so the library builds in
// parallel).
#include "tq_kernels.cuh"

namespace tq {
template cudaError_t launch_decode_dt<512, false, false>(const DecodeParams&, int, cudaStream_t);
template cudaError_t launch_unrotate<512>(const UnrotateParams&, bool, cudaStream_t);
}  // namespace tq
