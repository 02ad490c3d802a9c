// Lloyd-Max table fit on the GPU (tq_lloyd_max_fit).
//
// Page "mlx-bun 0.0.9 -> 0.0.11", file package/src/mlx/turboquant-tables.ts:
// the value tables are an iterative Lloyd-Max fit on a unit-normal sample.
// One iteration: boundaries are the fp32 midpoints of adjacent centroids;
// every sample goes to cell count(boundaries < x) (the codec's searchsorted);
// every centroid becomes the mean of its cell (a cell with no samples keeps
// its centroid).
//
// One cooperative launch runs every iteration; its blocks stay resident and
// meet at a grid barrier once per iteration. Each block bins a fixed slice of
// the sample (eight samples loaded per thread at a time) by binary search over
// the boundaries (shared memory, padded with +Inf to a power of two) into
// per-warp shared histograms, then adds its per-cell counts and sums into the
// iteration's global totals with integer atomics. Sums are int64 fixed point
// in units of 2^-32: every sample of magnitude >= 2^-9 is exact there
// (smaller ones are rounded to the unit), so the totals are exact and do not
// depend on the order of the additions. After the barrier every block forms
// the same means, total / 2^32 / count in float64 rounded once to fp32, as
// its next centroids. The totals rotate over three buffers: iteration i adds
// into buffer i mod 3, and block 0 clears buffer (i + 2) mod 3, which every
// block finished reading before the barrier of iteration i and which is next
// added into after the barrier of iteration i + 1. The barrier's wait is
// bounded: a block that gives up sets the error word, writes NaN centroids and
// boundaries and returns, and the others give up at their next barrier.
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

constexpr unsigned kLloydSpinLimit = 1u << 22;  // polls of ~64 ns: about a quarter of a second

struct LloydParams {
  const float* x;
  long long n;
  int levels;                // a power of two, 2 .. 256
  int iters;
  float* centroids;          // [levels]: the initial centroids on entry, the result on exit
  float* boundaries;         // [levels - 1]
  long long* sums;           // [3][levels], zero on entry
  unsigned long long* cnts;  // [3][levels], zero on entry
  unsigned* bar;             // arrivals, generation, error; zero on entry
  unsigned spin_limit;       // polls a block waits at a barrier before it gives up
  int absent_block;          // a block that leaves at its first barrier without arriving, or -1
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid barrier of a cooperative launch (all blocks resident). False when the
// wait gave up or another block reported an error. A block that gives up
// sets the error word bar[2] (read by tq_lloyd_max_fit_status). The absent
// block (failure-detection test hook) returns false without arriving, so
// every other block's wait runs out after spin_limit polls.
__device__ bool grid_barrier(unsigned* bar, unsigned spin_limit, int absent_block) {
  __shared__ int s_ok;
  __syncthreads();
  if (static_cast<int>(blockIdx.x) == absent_block) return false;
  if (threadIdx.x == 0) {
    const unsigned gen = ld_acquire(bar + 1);
    int ok = 1;
    __threadfence();
    if (atomicAdd(bar, 1u) == gridDim.x - 1) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicExch(bar + 1, gen + 1);
    } else {
      unsigned spins = 0;
      while (ld_acquire(bar + 1) == gen) {
        if (++spins > spin_limit) {
          atomicExch(bar + 2, 1u);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    if (ld_acquire(bar + 2) != 0) ok = 0;
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Per-warp cell sums in shared memory. SPLIT keeps each sum as three 32-bit
// words, the signed high word of the fixed-point values and the two 16-bit
// halves of their low words, added with native 32-bit shared atomics (a
// 64-bit shared atomic add cost 5 of the 12 us of an iteration at 16 levels:
// 12.1 -> 7.8 us with the split words); exact while a warp bins at most
// 65536 samples per iteration, so that the
// halves' sums stay below 2^32 (the high words wrap but their total, bounded by
// the sum of |x|, fits in int32). Larger slices take the int64 atomics.
template <bool SPLIT>
struct CellSums {
  unsigned w[SPLIT ? 3 : 2][kLloydWarps][256];
  __device__ void clear(int i) {
#pragma unroll
    for (int j = 0; j < (SPLIT ? 3 : 2); ++j) (&w[j][0][0])[i] = 0;
  }
  __device__ void add(int warp, int cell, unsigned long long v) {
    if constexpr (SPLIT) {
      atomicAdd(&w[0][warp][cell], static_cast<unsigned>(v >> 32));
      atomicAdd(&w[1][warp][cell], static_cast<unsigned>(v & 0xffffu));
      atomicAdd(&w[2][warp][cell], static_cast<unsigned>((v >> 16) & 0xffffu));
    } else {
      atomicAdd(reinterpret_cast<unsigned long long*>(&w[0][0][0]) + warp * 256 + cell, v);
    }
  }
  __device__ long long get(int warp, int cell) const {
    if constexpr (SPLIT) {
      return (static_cast<long long>(static_cast<int>(w[0][warp][cell])) << 32) +
             static_cast<long long>(w[1][warp][cell]) + (static_cast<long long>(w[2][warp][cell]) << 16);
    } else {
      return static_cast<long long>(reinterpret_cast<const unsigned long long*>(&w[0][0][0])[warp * 256 + cell]);
    }
  }
};

template <bool SPLIT>
__global__ void __launch_bounds__(kLloydThreads) lloyd_fit_kernel(LloydParams p) {
  __shared__ float s_c[256];  // current centroids, the same in every block
  __shared__ float s_b[256];  // boundaries, +Inf past the last
  __shared__ __align__(8) CellSums<SPLIT> s_sum;
  __shared__ unsigned s_cnt[kLloydWarps][256];
  const int K = p.levels, warp = threadIdx.x >> 5;
  for (int k = threadIdx.x; k < K; k += blockDim.x) s_c[k] = p.centroids[k];
  const long long lo = static_cast<long long>(blockIdx.x) * p.n / gridDim.x;
  const long long hi = static_cast<long long>(blockIdx.x + 1) * p.n / gridDim.x;
  for (int it = 0; it < p.iters; ++it) {
    long long* sums = p.sums + static_cast<long long>(it % 3) * K;
    unsigned long long* cnts = p.cnts + static_cast<long long>(it % 3) * K;
    for (int i = threadIdx.x; i < kLloydWarps * 256; i += blockDim.x) {
      s_sum.clear(i);
      (&s_cnt[0][0])[i] = 0;
    }
    __syncthreads();  // s_c complete (initial load or the previous means)
    for (int k = threadIdx.x; k < 256; k += blockDim.x)
      s_b[k] = k < K - 1 ? __fmul_rn(__fadd_rn(s_c[k], s_c[k + 1]), 0.5f) : __int_as_float(0x7f800000);
    __syncthreads();
    // A thread loads kLloydBatch samples before binning any of them, so their
    // reads overlap instead of each waiting out its own latency.
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
        s_sum.add(warp, cell, static_cast<unsigned long long>(__float2ll_rn(__fmul_rn(x, 4294967296.0f))));
        atomicAdd(&s_cnt[warp][cell], 1u);
      }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
      long long s = 0;
      unsigned c = 0;
#pragma unroll
      for (int w = 0; w < kLloydWarps; ++w) {
        s += s_sum.get(w, k);
        c += s_cnt[w][k];
      }
      if (c != 0) {
        atomicAdd(reinterpret_cast<unsigned long long*>(sums + k), static_cast<unsigned long long>(s));
        atomicAdd(cnts + k, static_cast<unsigned long long>(c));
      }
    }
    if (!grid_barrier(p.bar, p.spin_limit, p.absent_block)) {
      if (static_cast<int>(blockIdx.x) == p.absent_block) return;
      for (int k = threadIdx.x; k < K; k += blockDim.x) {
        p.centroids[k] = __int_as_float(0x7fc00000);
        if (k < K - 1) p.boundaries[k] = __int_as_float(0x7fc00000);
      }
      return;
    }
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
      const long long s = __ldcg(sums + k);
      const unsigned long long c = __ldcg(cnts + k);
      if (c > 0) s_c[k] = static_cast<float>(__ddiv_rn(static_cast<double>(s) / kFixedScale, static_cast<double>(c)));
    }
    if (blockIdx.x == 0) {
      long long* old_s = p.sums + static_cast<long long>((it + 2) % 3) * K;
      unsigned long long* old_c = p.cnts + static_cast<long long>((it + 2) % 3) * K;
      for (int k = threadIdx.x; k < K; k += blockDim.x) {
        old_s[k] = 0;
        old_c[k] = 0;
      }
    }
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
      p.centroids[k] = s_c[k];
      if (k < K - 1) p.boundaries[k] = __fmul_rn(__fadd_rn(s_c[k], s_c[k + 1]), 0.5f);
    }
  }
}

__global__ void lloyd_boundaries_kernel(const float* c, int K, float* b) {
  for (int k = threadIdx.x; k < K - 1; k += blockDim.x) b[k] = __fmul_rn(__fadd_rn(c[k], c[k + 1]), 0.5f);
}

// Blocks of the cooperative launch: kLloydBlocksPerSm per SM, at most what can
// be resident at once.
template <bool SPLIT>
int lloyd_grid() {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, lloyd_fit_kernel<SPLIT>, kLloydThreads, 0) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return (per_sm < kLloydBlocksPerSm ? per_sm : kLloydBlocksPerSm) * sm_count();
}

bool aligned(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace tq

extern "C" int64_t tq_lloyd_max_fit_workspace_size(int levels) {
  if (levels < 2 || levels > 256 || (levels & (levels - 1)) != 0) return -static_cast<int64_t>(TQ_ERR_INVALID_ARG);
  return 64 + 48LL * levels;  // barrier words, then three buffers of int64 sums and counts per level
}

extern "C" tq_status tq_lloyd_max_fit_bounded(const float* x, int64_t n, int levels, int iters,
                                              const float* init, float* centroids, float* boundaries,
                                              void* workspace, int64_t workspace_bytes, int64_t spin_limit,
                                              int absent_block, void* stream) {
  using namespace tq;
  if (spin_limit < 0 || spin_limit > 0xffffffffLL || absent_block < -1) return TQ_ERR_INVALID_ARG;
  if (n < 0 || iters < 0 || levels < 2 || levels > 256 || (levels & (levels - 1)) != 0) return TQ_ERR_INVALID_ARG;
  if (n > (1LL << 31) - 1) return TQ_ERR_INVALID_ARG;
  if (!init || !centroids || !boundaries || !workspace || (n > 0 && !x)) return TQ_ERR_INVALID_ARG;
  if (!aligned(x, 4) || !aligned(init, 4) || !aligned(centroids, 4) || !aligned(boundaries, 4) ||
      !aligned(workspace, 16))
    return TQ_ERR_ALIGNMENT;
  const long long need = 64 + 48LL * levels;
  if (workspace_bytes < need) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  LloydParams p{};
  p.x = x;
  p.n = n;
  p.levels = levels;
  p.iters = iters;
  p.centroids = centroids;
  p.boundaries = boundaries;
  p.bar = reinterpret_cast<unsigned*>(ws);
  p.spin_limit = spin_limit == 0 ? kLloydSpinLimit : static_cast<unsigned>(spin_limit);
  p.absent_block = absent_block;
  p.sums = reinterpret_cast<long long*>(ws + 64);
  p.cnts = reinterpret_cast<unsigned long long*>(ws + 64 + 24LL * levels);
  if (cudaMemcpyAsync(centroids, init, sizeof(float) * levels, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
      cudaMemsetAsync(ws, 0, need, s) != cudaSuccess)
    return TQ_ERR_CUDA;
  if (iters == 0) {
    lloyd_boundaries_kernel<<<1, 256, 0, s>>>(centroids, levels, boundaries);
  } else {
    void* args[] = {&p};
    // a warp bins at most ceil(n / grid) / warps + 32 samples per iteration
    const int grid = lloyd_grid<true>();
    const long long per_warp = ((n + grid - 1) / grid + kLloydWarps - 1) / kLloydWarps + 32;
    const bool split = per_warp <= 65536;
    const void* kernel = split ? reinterpret_cast<const void*>(lloyd_fit_kernel<true>)
                               : reinterpret_cast<const void*>(lloyd_fit_kernel<false>);
    if (cudaLaunchCooperativeKernel(kernel, dim3(split ? grid : lloyd_grid<false>()), dim3(kLloydThreads), args, 0,
                                    s) != cudaSuccess)
      return TQ_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

extern "C" tq_status tq_lloyd_max_fit(const float* x, int64_t n, int levels, int iters, const float* init,
                                      float* centroids, float* boundaries, void* workspace,
                                      int64_t workspace_bytes, void* stream) {
  return tq_lloyd_max_fit_bounded(x, n, levels, iters, init, centroids, boundaries, workspace, workspace_bytes, 0,
                                  -1, stream);
}

extern "C" tq_status tq_lloyd_max_fit_status(const void* workspace, void* stream) {
  if (!workspace) return TQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return TQ_ERR_ALIGNMENT;
  unsigned err = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      cudaMemcpy(&err, static_cast<const uint8_t*>(workspace) + 8, sizeof(err), cudaMemcpyDeviceToHost) !=
          cudaSuccess)
    return TQ_ERR_CUDA;
  return err != 0 ? TQ_ERR_TIMEOUT : TQ_OK;
}
