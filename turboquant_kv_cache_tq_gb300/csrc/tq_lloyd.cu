// Lloyd-Max table fit on the GPU (tq_lloyd_max_fit).
//
// Page "mlx-bun 0.0.9 -> 0.0.11", file package/src/mlx/turboquant-tables.ts:
// the value tables are an iterative Lloyd-Max fit on a unit-normal sample.
// One iteration: boundaries are the fp32 midpoints of adjacent centroids;
// every sample goes to cell count(boundaries < x) (the codec's searchsorted);
// every centroid becomes the mean of its cell (a cell with no samples keeps
// its centroid).
//
// One launch per iteration. Each block bins a fixed slice of the sample
// (loaded eight samples per thread at a time) by binary search over the
// boundaries (shared memory, padded with +Inf to a power of two) into
// per-warp shared histograms, then adds its per-cell
// counts and sums into global totals with integer atomics. Sums are int64
// fixed point in units of 2^-32: every sample of magnitude >= 2^-9 is exact
// there (smaller ones are rounded to the unit), so the totals are exact and do
// not depend on the order of the additions. The last block to finish (an
// atomic ticket after a fence; nobody waits) forms each mean as
// total / 2^32 / count in float64 rounded once to fp32, writes the centroids
// and their midpoints, and clears the totals and the ticket for the next
// launch.
#include <cstdint>

#include "../../include/tq.h"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kLloydThreads = 256;
constexpr int kLloydWarps = kLloydThreads / 32;
constexpr int kLloydBlocksPerSm = 2;
constexpr int kLloydBatch = 8;
constexpr double kFixedScale = 4294967296.0;  // 2^32

struct LloydParams {
  const float* x;
  long long n;
  int levels;             // a power of two, 2 .. 256
  float* centroids;       // [levels], read at the start, rewritten by the last block
  float* boundaries;      // [levels - 1]
  long long* total_sum;   // [levels], zero between launches
  unsigned long long* total_cnt;  // [levels], zero between launches
  unsigned* ticket;       // zero between launches
};

__device__ __forceinline__ void pdl_wait_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__global__ void __launch_bounds__(kLloydThreads) lloyd_iter_kernel(LloydParams p) {
  __shared__ float s_b[256];  // boundaries, +Inf past the last
  __shared__ long long s_sum[kLloydWarps][256];
  __shared__ unsigned s_cnt[kLloydWarps][256];
  __shared__ bool s_last;
  const int K = p.levels, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kLloydWarps * 256; i += blockDim.x) {
    (&s_sum[0][0])[i] = 0;
    (&s_cnt[0][0])[i] = 0;
  }
  pdl_wait_grid();  // the previous iteration's centroids are complete
  pdl_release();
  for (int k = threadIdx.x; k < 256; k += blockDim.x)
    s_b[k] = k < K - 1 ? __fmul_rn(__fadd_rn(p.centroids[k], p.centroids[k + 1]), 0.5f) : __int_as_float(0x7f800000);
  __syncthreads();
  const long long lo = static_cast<long long>(blockIdx.x) * p.n / gridDim.x;
  const long long hi = static_cast<long long>(blockIdx.x + 1) * p.n / gridDim.x;
  // A thread loads kLloydBatch samples before binning any of them, so their
  // reads overlap instead of each waiting out its own latency; the totals
  // are exact integers, so the order of the additions does not matter.
  for (long long base = lo + threadIdx.x; base < hi; base += kLloydBatch * static_cast<long long>(blockDim.x)) {
    float xs[kLloydBatch];
#pragma unroll
    for (int u = 0; u < kLloydBatch; ++u) {
      const long long i = base + static_cast<long long>(u) * blockDim.x;
      xs[u] = i < hi ? p.x[i] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kLloydBatch; ++u) {
      if (base + static_cast<long long>(u) * blockDim.x >= hi) break;
      const float x = xs[u];
      int cell = 0;  // count(boundaries < x): boundaries ascend, padding is +Inf
      for (int step = K >> 1; step > 0; step >>= 1)
        if (s_b[cell + step - 1] < x) cell += step;
      atomicAdd(reinterpret_cast<unsigned long long*>(&s_sum[warp][cell]),
                static_cast<unsigned long long>(__float2ll_rn(__fmul_rn(x, 4294967296.0f))));
      atomicAdd(&s_cnt[warp][cell], 1u);
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    long long s = 0;
    unsigned c = 0;
#pragma unroll
    for (int w = 0; w < kLloydWarps; ++w) {
      s += s_sum[w][k];
      c += s_cnt[w][k];
    }
    if (c != 0) {
      atomicAdd(reinterpret_cast<unsigned long long*>(p.total_sum + k), static_cast<unsigned long long>(s));
      atomicAdd(p.total_cnt + k, static_cast<unsigned long long>(c));
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(p.ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  // the last block: every other block's totals are visible (fence, ticket)
  __threadfence();
  float* s_c = &s_b[0];
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    const long long s = __ldcg(p.total_sum + k);
    const unsigned long long c = __ldcg(p.total_cnt + k);
    const float old = p.centroids[k];
    s_c[k] = c > 0 ? static_cast<float>(__ddiv_rn(static_cast<double>(s) / kFixedScale, static_cast<double>(c)))
                   : old;
    p.total_sum[k] = 0;
    p.total_cnt[k] = 0;
  }
  __syncthreads();
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    p.centroids[k] = s_c[k];
    if (k < K - 1) p.boundaries[k] = __fmul_rn(__fadd_rn(s_c[k], s_c[k + 1]), 0.5f);
  }
  if (threadIdx.x == 0) *p.ticket = 0u;
}

__global__ void lloyd_boundaries_kernel(const float* c, int K, float* b) {
  for (int k = threadIdx.x; k < K - 1; k += blockDim.x) b[k] = __fmul_rn(__fadd_rn(c[k], c[k + 1]), 0.5f);
}

int lloyd_grid() { return kLloydBlocksPerSm * sm_count(); }

bool aligned(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace tq

extern "C" int64_t tq_lloyd_max_fit_workspace_size(int levels) {
  if (levels < 2 || levels > 256 || (levels & (levels - 1)) != 0) return -static_cast<int64_t>(TQ_ERR_INVALID_ARG);
  return 16 + 16LL * levels;  // ticket, then int64 sums and counts per level
}

extern "C" tq_status tq_lloyd_max_fit(const float* x, int64_t n, int levels, int iters, const float* init,
                                      float* centroids, float* boundaries, void* workspace,
                                      int64_t workspace_bytes, void* stream) {
  using namespace tq;
  if (n < 0 || iters < 0 || levels < 2 || levels > 256 || (levels & (levels - 1)) != 0) return TQ_ERR_INVALID_ARG;
  if (n > (1LL << 31) - 1) return TQ_ERR_INVALID_ARG;
  if (!init || !centroids || !boundaries || !workspace || (n > 0 && !x)) return TQ_ERR_INVALID_ARG;
  if (!aligned(x, 4) || !aligned(init, 4) || !aligned(centroids, 4) || !aligned(boundaries, 4) ||
      !aligned(workspace, 16))
    return TQ_ERR_ALIGNMENT;
  const int grid = lloyd_grid();
  const long long need = 16 + 16LL * levels;
  if (workspace_bytes < need) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  LloydParams p{};
  p.x = x;
  p.n = n;
  p.levels = levels;
  p.centroids = centroids;
  p.boundaries = boundaries;
  p.ticket = reinterpret_cast<unsigned*>(ws);
  p.total_sum = reinterpret_cast<long long*>(ws + 16);
  p.total_cnt = reinterpret_cast<unsigned long long*>(ws + 16 + 8LL * levels);
  if (cudaMemcpyAsync(centroids, init, sizeof(float) * levels, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
      cudaMemsetAsync(ws, 0, need, s) != cudaSuccess)
    return TQ_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kLloydThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  for (int it = 0; it < iters; ++it)
    if (cudaLaunchKernelEx(&cfg, lloyd_iter_kernel, p) != cudaSuccess) return TQ_ERR_CUDA;
  if (iters == 0) lloyd_boundaries_kernel<<<1, 256, 0, s>>>(centroids, levels, boundaries);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
