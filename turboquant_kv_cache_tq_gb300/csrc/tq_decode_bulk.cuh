// Decode with bulk asynchronous copies (the Blackwell tensor-memory-access
// path): the codec's decode (page "@mlx-bun/inference 0.0.0-stage -> 1.0.0",
// file package/src/kernels/turboquant/ops.ts: decodeKeys, decodeValues,
// decodeValuesRotated), with every global byte moved by the copy engine
// instead of per-lane loads and stores.
//
// Why: the per-lane decode kernel is bound by the L1 data pipe, where every
// 32-byte sector of a global load or store costs a cycle (a warp's 128-bit
// store of 512 bytes: 16 cycles), on top of the centroid lookups and the
// Hadamard shuffles. Here a warp's tile of packed inputs (codes, scales, zero
// points: contiguous rows) arrives in shared memory by cp.async.bulk several
// items ahead, completing on a per-stage mbarrier, and its decoded tile is
// written to shared memory with 128-bit stores (512 bytes: 4 cycles when
// conflict-free) and leaves by one cp.async.bulk store.
//
// Layout: a tile is Geo<D>::RPW consecutive rows = 32 groups, so lane L's
// group sits at byte 4 * bits * L of the tile's packed codes, at 2 L of its
// scales and zero points, and at 64 L (bf16) of its decoded output, whatever
// D. Each warp owns kStagesIn input stages (codes | scales | zero points) and
// kStagesOut output buffers; items are taken in the encode's orders
// (ItemOrder): interleaved (item gw + k n, a V item when (item ^ k) is odd)
// for long launches, all V items first in snake order for launches of at
// most kSnakeSteps steps per warp, whose end is set by the warps with one
// step more than the rest.
//
// Used when every tile's rows are contiguous and 16-byte aligned in all five
// packed buffers, the outputs are bf16 and every buffer is device memory
// (the host checks it: T a multiple of RPW, t_cap times each packed row size
// a multiple of 16, the pointers' memory type); other launches, for instance
// outputs written straight to pinned host memory, take the per-lane kernel.
//
// Waits on the mbarriers are bounded: a wait that gives up sets bit 0 of the
// library's device error word, waits (bounded) for the copies the warp still
// has in flight and stops the warp.
//
// Included by tq_kernels.cuh after the per-lane decode and the launch helpers.
#pragma once

// Ring sizes and the 8-bit-value occupancy bound. Measured alternatives on
// the long-context v8 / v3 decode (278 / 254 us as set): 2 input stages
// 279 / 255, 8 input stages 395 / 275 (fewer blocks fit), 1 output buffer
// 280 / 255, 4 output buffers 403 / 279, 3 blocks per SM at 8-bit values
// (80 registers; shared memory still fits only 2) 293 / 254.
#ifndef TQ_DECODE_BULK_STAGES_IN
#define TQ_DECODE_BULK_STAGES_IN 4
#endif
#ifndef TQ_DECODE_BULK_STAGES_OUT
#define TQ_DECODE_BULK_STAGES_OUT 2
#endif
#ifndef TQ_DECODE_BULK_V8_MIN_BLOCKS
#define TQ_DECODE_BULK_V8_MIN_BLOCKS 2
#endif

namespace tq {

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Completion of phase `parity` of the barrier, polled at most `limit` times.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, unsigned parity, unsigned limit) {
  for (unsigned i = 0; i < limit; ++i) {
    unsigned done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
// Global -> shared bulk copy completing on `bar` (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, unsigned bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// Shared -> global bulk copy in the issuing thread's current bulk group.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, unsigned bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// All but the N most recent bulk groups of this thread have read their source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's generic-proxy shared-memory accesses with later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

// The lane's B packed words from a staged tile (lane's words at 4 B lane).
// Bank-conflict free: 16 bytes per lane read by quarter-warps at distinct
// banks; 8 bytes by half-warps; odd word strides for 3 and 5 bits; the two
// 16-byte chunks of 8-bit codes read in an order that alternates every four
// lanes (lanes L and L + 4 would share banks), then put back in place.
template <int B>
__device__ __forceinline__ void lds_words(uint32_t tile, int lane, uint32_t (&w)[B]) {
  const uint32_t a = tile + 4u * B * lane;
  if constexpr (B == 8) {
    const uint32_t flip = (lane >> 2) & 1;
    const uint4 u = lds128(a + 16u * flip);
    const uint4 v = lds128(a + 16u * (flip ^ 1u));
    w[0] = flip ? v.x : u.x; w[1] = flip ? v.y : u.y; w[2] = flip ? v.z : u.z; w[3] = flip ? v.w : u.w;
    w[4] = flip ? u.x : v.x; w[5] = flip ? u.y : v.y; w[6] = flip ? u.z : v.z; w[7] = flip ? u.w : v.w;
  } else if constexpr (B == 4) {
    const uint4 u = lds128(a);
    w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
  } else if constexpr (B == 2) {
    const uint2 u = lds64(a);
    w[0] = u.x; w[1] = u.y;
  } else {
#pragma unroll
    for (int k = 0; k < B; ++k) w[k] = lds32(a + 4u * k);
  }
}

// The lane's 16 bf16 output words (64 bytes) into a staged output tile at
// byte 64 L. Quarter-warp lanes L and L + 2 hold the same banks for the same
// chunk, so lane L stores chunk (t + L / 2) mod 4 at step t (the chunks
// rotated into place by selects first).
__device__ __forceinline__ void sts_words16(uint32_t tile, int lane, const uint32_t (&o)[16]) {
  const uint32_t r = (lane >> 1) & 3;
  uint32_t c[16];
  // rotate the four 4-word chunks left by r: c[chunk t] = o[chunk (t + r) mod 4]
#pragma unroll
  for (int i = 0; i < 16; ++i) c[i] = (r & 1) ? o[(i + 4) & 15] : o[i];
  uint32_t d[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) d[i] = (r & 2) ? c[(i + 8) & 15] : c[i];
  const uint32_t a = tile + 64u * lane;
#pragma unroll
  for (int t = 0; t < 4; ++t) sts128(a + 16u * ((t + r) & 3), d[4 * t], d[4 * t + 1], d[4 * t + 2], d[4 * t + 3]);
}

template <int D, int VB, int KMODE>
struct BulkDecodeShape {
  static constexpr int kKB = KeySpec<KMODE>::B;
  static constexpr int kW = kKB > VB ? kKB : VB;
  static constexpr int kStagesIn = TQ_DECODE_BULK_STAGES_IN;    // a power of two
  static constexpr int kStagesOut = TQ_DECODE_BULK_STAGES_OUT;  // bulk groups a warp keeps in flight
  static constexpr int kCodeBytes = 128 * kW;  // 32 groups x 4 W bytes
  static constexpr int kScaleOff = kCodeBytes;
  static constexpr int kZeroOff = kCodeBytes + 64;
  static constexpr int kInBytes = kCodeBytes + 128;  // a multiple of 128
  static constexpr int kOutBytes = 32 * 32 * 2;      // 1024 bf16 outputs
  static constexpr int kWarpBytes = kStagesIn * kInBytes + kStagesOut * kOutBytes;
  static constexpr int kWarps = kThreads / 32;
  static constexpr int kBarOff = kWarps * kWarpBytes;
  static constexpr int kSmem = kBarOff + kWarps * kStagesIn * 8;
  static constexpr int kMinBlocks = VB == 8 ? TQ_DECODE_BULK_V8_MIN_BLOCKS : 3;
};

// Polls of a stage's mbarrier before a warp gives up (each poll may suspend
// the warp for a short hardware time slice; about a second in all).
constexpr unsigned kBulkWaitLimit = 1u << 20;

template <int D, int VB, int KMODE, bool ROT, bool SNAKE>
__global__ void __launch_bounds__(kThreads, (BulkDecodeShape<D, VB, KMODE>::kMinBlocks))
    decode_bulk_kernel(DecodeParams p) {
  using G = Geo<D>;
  using M = KeySpec<KMODE>;
  using SH = BulkDecodeShape<D, VB, KMODE>;
  constexpr int W = SH::kW;
  constexpr int S = SH::kStagesIn;
  __shared__ float s_cent[CentroidTable<VB>::kWords];
  __shared__ __align__(16) uint32_t s_sign[D / 2];
  extern __shared__ __align__(128) uint8_t s_dyn[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t in_sh = smem_u32(s_dyn) + warp * SH::kWarpBytes;
  const uint32_t out_sh = in_sh + S * SH::kInBytes;
  const uint32_t bar_sh = smem_u32(s_dyn) + SH::kBarOff + warp * S * 8;
  fill_centroids<VB>(s_cent);
  fill_sign_words<D>(s_sign);
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < S; ++i) mbar_init(bar_sh + 8 * i, 1);
    mbar_fence_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();

  const int l = lane % G::LPR;
  const int n_warps = gridDim.x * (blockDim.x >> 5);
  const int tiles = p.rows / G::RPW;  // every tile is full (checked on the host)
  const int items = 2 * tiles;
  const int gw = warp_index();
  // the encode's item orders: interleaved K and V items for long launches,
  // all V items first in snake order for short ones (see ItemOrder)
  const ItemOrder<SNAKE> ord{n_warps, gw, tiles};
  // Lane 0 issues the copies of step k into stage k mod S.
  auto issue = [&](int k) {
    const int it = ord.item(k);
    if (lane != 0 || it >= items) return;
    const int r0 = ord.tile(it) * G::RPW;
    const int bh = fast_div(r0, p.tdiv);
    const long long irow = static_cast<long long>(bh) * p.t_cap + (r0 - bh * p.T);
    const uint32_t st = in_sh + (k & (S - 1)) * SH::kInBytes;
    const uint32_t bar = bar_sh + 8 * (k & (S - 1));
    if (!TQ_CHECK(irow >= 0 && irow + G::RPW <= p.cache_rows && r0 + G::RPW <= p.rows, p.err)) {
      mbar_expect_tx(bar, 0);  // completes the stage's phase with no copy (the debug build's skip)
      return;
    }
    if (ord.is_v(it, k)) {
      mbar_expect_tx(bar, 128 * VB + 64);
      bulk_load(st, p.v_codes + irow * (D * VB / 8), 128 * VB, bar);
      bulk_load(st + SH::kScaleOff, p.v_scales + irow * (D / 32), 64, bar);
    } else {
      mbar_expect_tx(bar, 128 * M::B + 128);
      bulk_load(st, p.k_codes + irow * (D * M::B / 8), 128 * M::B, bar);
      bulk_load(st + SH::kScaleOff, p.k_scales + irow * (D / 32), 64, bar);
      bulk_load(st + SH::kZeroOff, p.k_zeros + irow * (D / 32), 64, bar);
    }
  };
  // the lane's sign words stay in registers (ROT: no signs)
  uint32_t S_l[16];
  if constexpr (!ROT) load_sign_words(s_sign, l, S_l);
  const float* cent = s_cent + (CentroidTable<VB>::kRep > 1 ? lane : 0);
  auto no_prefetch = [] {};

#pragma unroll
  for (int k = 0; k < S; ++k) issue(k);
  int k = 0;
  bool ok = true;
  for (;; ++k) {
    const int it = ord.item(k);
    if (it >= items) break;
    const bool is_v = ord.is_v(it, k);
    const uint32_t st = in_sh + (k & (S - 1)) * SH::kInBytes;
    if (!__all_sync(kFull, mbar_wait(bar_sh + 8 * (k & (S - 1)), (k / S) & 1, kBulkWaitLimit))) {
      ok = false;  // the same decision in every lane
      break;
    }
    PackedIn<W> in;
    if (is_v) {
      uint32_t t[VB];
      lds_words<VB>(st, lane, t);
#pragma unroll
      for (int j = 0; j < W; ++j) in.w[j] = j < VB ? t[j < VB ? j : 0] : 0u;
      in.sz = lds16(st + SH::kScaleOff + 2 * lane);
    } else {
      uint32_t t[M::B];
      lds_words<M::B>(st, lane, t);
#pragma unroll
      for (int j = 0; j < W; ++j) in.w[j] = j < M::B ? t[j < M::B ? j : 0] : 0u;
      in.sz = lds16(st + SH::kScaleOff + 2 * lane) | (lds16(st + SH::kZeroOff + 2 * lane) << 16);
    }
    __syncwarp();  // the whole warp has read stage k
    if (lane == 0) fence_proxy_async();
    issue(k + S);
    uint32_t o[16];
    if (!is_v) {
      float x[32];
      decode_key_item<KMODE>(in, x, no_prefetch);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * j], x[2 * j + 1]);
        o[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
    } else {
      decode_value_words<G::LPR, VB, false, ROT, true>(in, l, S_l, cent, p.rot_scale, p.neg_zero, o, no_prefetch);
    }
    // stage the decoded tile and send it out with one bulk store
    const uint32_t ob = out_sh + (k % SH::kStagesOut) * SH::kOutBytes;
    if (lane == 0) bulk_wait_read<SH::kStagesOut - 1>();  // the store that last read `ob` is done with it
    __syncwarp();
    sts_words16(ob, lane, o);
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) {
      const int r0 = ord.tile(it) * G::RPW;
      bulk_store(static_cast<__nv_bfloat16*>(is_v ? p.v_out : p.k_out) + static_cast<size_t>(r0) * D, ob,
                 SH::kOutBytes);
      bulk_commit();
    }
  }
  if (!ok) {
    if (lane == 0 && p.err != nullptr) atomicOr(p.err, 1u);
    // wait (bounded) for this warp's loads still in flight before leaving
    for (int j = k; j < k + S; ++j) {
      if (ord.item(j) >= items) break;
      if (!mbar_wait(bar_sh + 8 * (j & (S - 1)), (j / S) & 1, kBulkWaitLimit)) break;
    }
  }
  if (lane == 0) bulk_wait_all();
}

// Bulk-path eligibility: tiles never straddle a (b, h) boundary and every
// tile of every packed buffer starts on 16 bytes (the ABI already requires
// 16-byte aligned base pointers).
template <int D>
inline bool bulk_decode_ok(const DecodeParams& p, bool out_bf16) {
  if (!out_bf16 || !p.device_memory || p.T % Geo<D>::RPW != 0) return false;
  const long long row_bytes[] = {p.pdk, p.pdv, 2LL * p.ng};
  for (long long x : row_bytes)
    if ((p.t_cap * x) % 16 != 0) return false;
  return true;
}

template <int D, int VB, int KMODE, bool ROT>
cudaError_t launch_decode_bulk(const DecodeParams& p, cudaStream_t s) {
  using SH = BulkDecodeShape<D, VB, KMODE>;
  static const int resident =
      std::min(prepare_dyn_smem(decode_bulk_kernel<D, VB, KMODE, ROT, false>, SH::kSmem),
               prepare_dyn_smem(decode_bulk_kernel<D, VB, KMODE, ROT, true>, SH::kSmem));
  const long long items = 2LL * (p.rows / Geo<D>::RPW);
  const int grid = grid_for(items, resident);
  // short launches (at most kSnakeSteps steps per warp) take the snake order
  const bool snake = items <= static_cast<long long>(kSnakeSteps) * grid * SH::kWarps;
  const cudaError_t e = snake ? launch_pdl(decode_bulk_kernel<D, VB, KMODE, ROT, true>, grid, p, s, SH::kSmem)
                              : launch_pdl(decode_bulk_kernel<D, VB, KMODE, ROT, false>, grid, p, s, SH::kSmem);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace tq
