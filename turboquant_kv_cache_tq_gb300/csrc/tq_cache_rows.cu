// Batched packed-cache row assembly (tq_cache_assemble).
//
// Page "@mlx-bun/inference 0.0.0-stage -> 1.0.0", files
// package/src/model/batched-quant.ts (mergeQuantRows, extendQuantRows,
// extractQuantRow, filterQuantRows) and batched-mask.ts: continuous batching
// moves whole token rows of a quantized cache between batch rows, padding
// shorter rows on the left with zero bytes. Quantization packs along head_dim
// only, so a token is a whole row of each of the five packed buffers and all
// four operations are byte copies. They share one primitive: destination
// batch row r is assembled from one source (cache, batch row, token range),
// right-justified in a window of `width` tokens, with width - len zero tokens
// in front. One kernel launch assembles up to kRowsPerLaunch destination rows;
// the row descriptors travel in the kernel parameters, so nothing is
// allocated.
#include <cstdint>

#include "../../include/tq.h"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kRowsPerLaunch = 48;
constexpr int kChunkBytes = 8192;  // bytes of one buffer's window per block
constexpr int kCopyThreads = 256;

struct RowSrc {
  const uint8_t* p[5];  // the source's five buffers
  long long b, t_cap, t_start, len;
};

struct AssembleParams {
  RowSrc rows[kRowsPerLaunch];
  uint8_t* dst[5];
  long long X[5];       // bytes of one token row of each buffer
  long long chunks[5];  // blocks along the window of each buffer
  long long t_cap, width;
  int H;
  int row0;             // first destination batch row of this launch
};

// Window byte i of destination row r, head h, buffer k is zero for
// i < pad = (width - len) X and source byte i - pad otherwise.
__global__ void __launch_bounds__(kCopyThreads) assemble_kernel(const __grid_constant__ AssembleParams p) {
  const int r = blockIdx.z, h = blockIdx.y;
  int k = 0;
  long long c = blockIdx.x;
  while (k < 4 && c >= p.chunks[k]) {
    c -= p.chunks[k];
    ++k;
  }
  const long long X = p.X[k];
  const RowSrc& s = p.rows[r];
  const long long win = p.width * X;
  const long long pad = (p.width - s.len) * X;
  const long long lo = c * kChunkBytes;
  const long long hi = lo + kChunkBytes < win ? lo + kChunkBytes : win;
  uint8_t* dst = p.dst[k] + (static_cast<long long>(p.row0 + r) * p.H + h) * p.t_cap * X;
  // source byte j sits at src0 + pad + j for j in [0, len X); nothing is read
  // outside that range
  const uint8_t* src = s.len > 0 ? s.p[k] + ((s.b * p.H + h) * s.t_cap + s.t_start) * X : nullptr;
  const uintptr_t shifted = reinterpret_cast<uintptr_t>(src) - static_cast<uintptr_t>(pad);
  const bool vec = ((reinterpret_cast<uintptr_t>(dst) | shifted) & 15u) == 0;
  // 16-byte vectors up to the last whole vector of the chunk, words after it
  const long long hv = vec ? lo + ((hi - lo) & ~15LL) : lo;
  if (vec) {
    for (long long i = lo + 16LL * threadIdx.x; i < hv; i += 16LL * blockDim.x) {
      uint4 v;
      if (i >= pad) {
        v = *reinterpret_cast<const uint4*>(src + (i - pad));
      } else if (i + 16 <= pad) {
        v = make_uint4(0u, 0u, 0u, 0u);
      } else {  // straddles the pad: word by word (pad is a multiple of 4)
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const long long j = i + 4 * e;
          w[e] = j < pad ? 0u : *reinterpret_cast<const uint32_t*>(src + (j - pad));
        }
        v = make_uint4(w[0], w[1], w[2], w[3]);
      }
      *reinterpret_cast<uint4*>(dst + i) = v;
    }
  }
  for (long long i = hv + 4LL * threadIdx.x; i < hi; i += 4LL * blockDim.x) {
    *reinterpret_cast<uint32_t*>(dst + i) = i < pad ? 0u : *reinterpret_cast<const uint32_t*>(src + (i - pad));
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace tq

extern "C" tq_status tq_cache_assemble(const tq_row_source* rows, int64_t n_rows, int64_t H, int64_t D,
                                       int k_bits, int v_bits, void* k_codes, void* k_scales, void* k_zeros,
                                       void* v_codes, void* v_scales, int64_t t_cap, int64_t width,
                                       void* stream) {
  using namespace tq;
  if (n_rows < 0 || H < 1 || H > 65535 || t_cap < 0 || width < 0 || width > t_cap) return TQ_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256 && D != 512) return TQ_ERR_HEAD_DIM;
  if ((k_bits != 2 && k_bits != 4 && k_bits != 5 && k_bits != 8) ||
      (v_bits != 2 && v_bits != 3 && v_bits != 4 && v_bits != 5 && v_bits != 8))
    return TQ_ERR_BITS;
  if (n_rows == 0 || width == 0) return TQ_OK;
  if (!rows) return TQ_ERR_INVALID_ARG;
  void* dst[5] = {k_codes, k_scales, k_zeros, v_codes, v_scales};
  for (void* d : dst) {
    if (!d) return TQ_ERR_INVALID_ARG;
    if (!aligned16(d)) return TQ_ERR_ALIGNMENT;
  }
  const long long X[5] = {D * k_bits / 8, D / 16, D / 16, D * v_bits / 8, D / 16};
  if (n_rows > (1LL << 31) / H || t_cap > (1LL << 40) / 512) return TQ_ERR_INVALID_ARG;
  for (int64_t r = 0; r < n_rows; ++r) {
    const tq_row_source& s = rows[r];
    if (s.len < 0 || s.len > width || s.t_start < 0 || s.t_cap < 0 || s.b < 0 || s.B < 0) return TQ_ERR_INVALID_ARG;
    if (s.len == 0) continue;
    if (s.b >= s.B || s.t_start + s.len > s.t_cap || s.t_cap > (1LL << 40) / 512) return TQ_ERR_INVALID_ARG;
    const void* sp[5] = {s.k_codes, s.k_scales, s.k_zeros, s.v_codes, s.v_scales};
    for (const void* q : sp) {
      if (!q) return TQ_ERR_INVALID_ARG;
      if (!aligned16(q)) return TQ_ERR_ALIGNMENT;
    }
  }
  AssembleParams p{};
  long long blocks_x = 0;
  for (int k = 0; k < 5; ++k) {
    p.dst[k] = static_cast<uint8_t*>(dst[k]);
    p.X[k] = X[k];
    p.chunks[k] = (width * X[k] + kChunkBytes - 1) / kChunkBytes;
    blocks_x += p.chunks[k];
  }
  p.t_cap = t_cap;
  p.width = width;
  p.H = static_cast<int>(H);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int64_t r0 = 0; r0 < n_rows; r0 += kRowsPerLaunch) {
    const int n = static_cast<int>(n_rows - r0 < kRowsPerLaunch ? n_rows - r0 : kRowsPerLaunch);
    for (int i = 0; i < n; ++i) {
      const tq_row_source& s = rows[r0 + i];
      const void* sp[5] = {s.k_codes, s.k_scales, s.k_zeros, s.v_codes, s.v_scales};
      for (int k = 0; k < 5; ++k) p.rows[i].p[k] = static_cast<const uint8_t*>(sp[k]);
      p.rows[i].b = s.b;
      p.rows[i].t_cap = s.t_cap;
      p.rows[i].t_start = s.t_start;
      p.rows[i].len = s.len;
    }
    p.row0 = static_cast<int>(r0);
    assemble_kernel<<<dim3(static_cast<unsigned>(blocks_x), static_cast<unsigned>(H), static_cast<unsigned>(n)),
                      kCopyThreads, 0, st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return TQ_ERR_CUDA;
  }
  return TQ_OK;
}
