// Decode kernels for head_dim 512, rotated values, fp32 outputs (one
// translation unit per head_dim, direction and type, so the library builds in
// parallel).
#include "tq_kernels.cuh"

namespace tq {
template cudaError_t launch_decode_dt<512, true, true>(const DecodeParams&, int, cudaStream_t);
}  // namespace tq
