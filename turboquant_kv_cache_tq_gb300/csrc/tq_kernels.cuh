// Fused encode and decode kernels of the TurboQuant KV codec.
//
// Encode, per row (b, h, t) of K and V (page "@mlx-bun/inference 0.0.0-stage
// -> 1.0.0", file package/src/kernels/turboquant/ops.ts):
//   K: fp32 upcast, per-32-group min/max, scale = range / levels, zero point,
//      codes = clip(round(x / (scale + eps) - zero)), fp16 scale and zero
//      (encodeKeys), bit packing (packBits);
//   V: signs, normalised Hadamard transform (fwht, encode), per-32-group RMS
//      scale, Lloyd-Max index of x / (scale + eps) (encodeValues,
//      searchsorted), bit packing.
// Decode, per row: unpack; (code + zero) * scale for K (decodeKeys);
//   centroid * scale, Hadamard transform, signs for V (decodeValues).
//
// Division-free quantisation:
//   K: RN(x / se) is obtained exactly from the reciprocal by one remainder
//      correction (div_by_recip: q0 = RN(x y), q = RN(q0 + RN(x - q0 se) y),
//      y = RN(1/se); correctly rounded, see there), then RN(q - zp) and rint,
//      the page's operations in order, so K codes are exactly the page's. A
//      warp with a group whose codes need the clamp (or whose quotient could
//      overflow) takes IEEE division.
//   V: the index is count(boundaries < v) for the exact product
//      v = y * RN(1/se), which is within one ulp of RN(y / se) (|v| <=
//      sqrt(32), so within 5e-7); it can only differ from the divided value's
//      index when v is that close to a boundary.
//
// Work split: a work item is the K half or the V half of a tile of
// Geo<D>::RPW rows, and each step of a warp takes one item (ItemOrder), so
// registers cover one half at a time. Encode streams its inputs through a
// per-warp shared-memory ring (EncodeRing), several items ahead; decode loads
// the next item's packed words before the current item's math. Lanes of a
// partial last tile redo the last row (so shuffles stay converged) but store
// nothing.
//
// Launch: the kernels are launched with programmatic stream serialization.
// A block fills its shared tables, lets dependent launches begin
// (griddepcontrol.launch_dependents), then waits for the grids it depends on
// to complete (griddepcontrol.wait) before touching any input or output, so
// the prologue overlaps the previous kernel's tail and stream order holds.
#pragma once

#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

constexpr int kThreads = 256;
#ifndef TQ_ENCODE_MIN_BLOCKS
#define TQ_ENCODE_MIN_BLOCKS 3  // 24 resident warps per SM
#endif
#ifndef TQ_DECODE_MIN_BLOCKS
#define TQ_DECODE_MIN_BLOCKS 3  // 24 resident warps per SM
#endif
constexpr int kEncodeMinBlocks = TQ_ENCODE_MIN_BLOCKS;
constexpr int kDecodeMinBlocks = TQ_DECODE_MIN_BLOCKS;

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Encode input staging: each warp streams its items' inputs through a ring of
// shared-memory stages filled by asynchronous 16-byte copies (cp.async), so a
// warp keeps several items' loads in flight without holding them in
// registers. A lane copies, and later reads back, only its own group: the
// copies of one lane complete and become visible to that lane at
// cp.async.wait_group, so no cross-lane synchronisation is needed. Within a
// stage, lane L's 16-byte chunk j sits at chunk (j xor swz(L)), which keeps
// the 128-bit reads of every quarter-warp on distinct banks. Two stages (one
// item in flight while the warp works on another) measured faster than four
// at every size: long-context v8 encode 294 -> 284 us, v3 287 -> 279 us,
// head_dim 256 41.8 -> 40.5 us, the 8B-shaped layer 7.13 -> 7.05 us.
#ifndef TQ_ENCODE_STAGES
#define TQ_ENCODE_STAGES 2
#endif
template <bool F32, int STAGES = (F32 ? 2 : TQ_ENCODE_STAGES), int THREADS = kThreads>
struct EncodeRing {
  static constexpr int kLaneBytes = F32 ? 128 : 64;  // 32 inputs
  static constexpr int kChunks = kLaneBytes / 16;
  static constexpr int kStages = STAGES;  // a power of two
  static constexpr int kStageBytes = 32 * kLaneBytes;
  static constexpr int kBlockBytes = (THREADS / 32) * kStages * kStageBytes;
  static_assert((kStages & (kStages - 1)) == 0, "stages must be a power of two");
  __device__ static int swz(int lane) { return F32 ? (lane & 7) : ((lane >> 1) & 3); }
};

// Lloyd-Max cell lookups: the index of every value is one random 64-bit
// shared load into a cell table (CellGrid), and lanes of a half-warp loading
// different cells of the same bank pair serialize. With the 256- and
// 1024-cell tables of 5 and 8 bits those conflicts bound the kernel, so those
// shapes (bf16 inputs) keep the table once per half-warp lane (entry r for
// lane L at 16 r + L % 16: the 16 lanes of a half-warp never share a bank),
// restricted to the cells a finite-RMS group can reach: |v| <= sqrt(32), so
// cells OFF - R .. OFF + R with R = floor(5.6569 S) + 1 (23 and 93 KB), in one
// 512-thread block per SM beside a two-stage ring (which also holds each
// lane's sign words in registers). Narrower tables conflict less, but from
// head_dim 128 up the wide shape is faster at every width too (ablation runs:
// [32,8,8192,128] v3 encode 322 -> 301 us, hd256 v4 68 -> 58 us, hd512 v2
// 67 -> 59 us; v8 on the long-context cache 393 -> 299 us when the shape was
// introduced). Head_dim 64 (one cross-lane stage) keeps the shared single
// table in three 256-thread blocks per SM for widths below 5, unmeasured
// against the wide shape; fp32 inputs keep the single table.
#ifndef TQ_ENCODE_REP_THREADS
#define TQ_ENCODE_REP_THREADS 512
#endif
template <int VB>
struct RepCells {
  static constexpr int R = static_cast<int>(5.6569f * CellGrid<VB>::S) + 1;
  static constexpr int kLo = CellGrid<VB>::OFF - R;
  static constexpr int kCount = 2 * R + 1;
  static constexpr int kBytes = kCount * 16 * static_cast<int>(sizeof(CellEntry));
};

// Cells below and above the replicated range hold no boundary, so clamping a
// cell into the range leaves the count unchanged.
template <int VB>
constexpr bool rep_range_holds_all_boundaries() {
  for (int j = 0; j < (1 << VB) - 1; ++j) {
    const int c = grid_cell_host<VB>(lm_boundary<VB>(j));
    if (c <= RepCells<VB>::kLo || c >= RepCells<VB>::kLo + RepCells<VB>::kCount - 1) return false;
  }
  return RepCells<VB>::kLo >= 0 && RepCells<VB>::kLo + RepCells<VB>::kCount <= CellGrid<VB>::NC;
}
static_assert(rep_range_holds_all_boundaries<2>() && rep_range_holds_all_boundaries<3>() &&
                  rep_range_holds_all_boundaries<4>() && rep_range_holds_all_boundaries<5>() &&
                  rep_range_holds_all_boundaries<8>(),
              "a boundary lies outside the replicated cell range");

// The replicated table costs each block a 23 or 93 KB fill before its first
// item, which only pays off on launches of many rows; smaller launches (for
// instance decode-step appends) take the single-table shape.
// (The 8B-shaped layer, 32768 rows, encodes in 7.06 us with the single table
// and in 7.45 us with the replicated one.)
#ifndef TQ_ENCODE_REP_MIN_ROWS
#define TQ_ENCODE_REP_MIN_ROWS 65536
#endif
constexpr int kRepMinRows = TQ_ENCODE_REP_MIN_ROWS;
template <int D, int VB, bool F32, bool ALLOW_REP = true>
struct EncodeShape {
  static constexpr bool REP = ALLOW_REP && !F32 && (VB >= 5 || D >= 128);
  static constexpr bool WIDE = REP;
  static constexpr int kBlockThreads = WIDE ? TQ_ENCODE_REP_THREADS : kThreads;
  static constexpr int kMinBlocks = WIDE ? 1 : kEncodeMinBlocks;
  using Ring = EncodeRing<F32, F32 ? 2 : TQ_ENCODE_STAGES, kBlockThreads>;
  static constexpr int kRepBytes = REP ? RepCells<VB>::kBytes : 0;
  static constexpr int kSmem = Ring::kBlockBytes + kRepBytes;
};

// Lloyd-Max index of the pair y * inv from the lane's replica of the compact
// cell table: the same cell and comparison as lm_index2_scaled. No clamp is
// needed: for a finite RMS every element of the group has |y| <= sqrt(32) rms
// exactly, and the fp32 sum of squares, square root, eps and reciprocal move
// that bound by at most a dozen unit roundoffs (less still when eps
// dominates), so |y * inv| < sqrt(32) (1 + 2^-20) < 5.6569 and the cell
// rint(v S) lies within +-R of OFF (R = floor(5.6569 S) + 1). `rep_bias` is
// the shared-memory address of the lane's entry of the range's first cell
// minus (kMagicBits + kLo) * 128 (mod 2^32): the entry of a cell is then one
// multiply-add of the rounded value's bits away.
__device__ __forceinline__ CellEntry ld_cell_shared(uint32_t addr) {
  CellEntry e;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=f"(e.b), "=r"(e.base) : "r"(addr));
  return e;
}

template <int VB>
__device__ __forceinline__ uint32_t rep_bias_for(uint32_t rep_lane_sh) {
  return rep_lane_sh - (kMagicBits + static_cast<uint32_t>(RepCells<VB>::kLo)) * 128u;
}

template <int VB>
__device__ __forceinline__ void lm_index2_rep(float2 y, float inv, uint32_t rep_bias, uint32_t& i0, uint32_t& i1) {
  using G = CellGrid<VB>;
  const float2 s = fma2(y, f2(__fmul_rn(inv, G::S)), f2(grid_magic<VB>()));
  const CellEntry e0 = ld_cell_shared(__float_as_uint(s.x) * 128u + rep_bias);
  const CellEntry e1 = ld_cell_shared(__float_as_uint(s.y) * 128u + rep_bias);
  const float2 d = fma2(y, f2(-inv), make_float2(e0.b, e1.b));
  i0 = static_cast<uint32_t>(e0.base) + (__float_as_uint(d.x) >> 31);
  i1 = static_cast<uint32_t>(e1.base) + (__float_as_uint(d.y) >> 31);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Global warp index, numbered across blocks first (warp w of block b is
// w * gridDim.x + b), so that when the items do not divide evenly the warps
// with one item more are spread over all blocks, hence over all SMs.
__device__ __forceinline__ int warp_index() { return static_cast<int>((threadIdx.x >> 5) * gridDim.x + blockIdx.x); }

// Order of the 2 * tiles items of an encode launch over its n warps; step k
// of warp gw takes item(k). A V item costs about three times a K item.
//   Interleaved (SNAKE = false, long launches): item k * n + gw, a V item
//   when (item ^ k) is odd, of tile item / 2 (a bijection because n is
//   even). Every warp alternates kinds, so each SM mixes memory-heavy K items
//   with ALU-heavy V items throughout.
//   Snake (short launches of at most kSnakeSteps steps per warp, whose end is
//   set by the warps with one step more than the rest): all V tiles come
//   before all K tiles and the steps walk them in snake order (k * n + gw for
//   even k, k * n + n - 1 - gw for odd k), so the V items fill the first
//   steps and the warps with an extra step take K items in it.
// Measured: a [1, 8, 4096, 128] layer (2.25 steps per warp) encodes in 7.4
// instead of 7.8 us in snake order; on the [32, 8, 8192, 128] cache the
// interleaved order is 3% faster. The order is a template argument: as a
// runtime flag its selects cost the long launches another 2.5%.
constexpr int kSnakeSteps = 4;
template <bool SNAKE>
struct ItemOrder {
  int n, gw, tiles;
  __device__ int item(int k) const { return k * n + ((SNAKE && (k & 1)) ? n - 1 - gw : gw); }
  __device__ bool is_v(int it, int k) const { return SNAKE ? it < tiles : ((it ^ k) & 1) != 0; }
  __device__ int tile(int it) const { return SNAKE ? (it < tiles ? it : it - tiles) : (it >> 1); }
};

template <int KMODE>
struct KeySpec {
  static constexpr int B = (KMODE == kK2) ? 2 : (KMODE == kK4) ? 4 : (KMODE == kK5) ? 5 : 8;
  static constexpr bool SIGNED = (KMODE == kK8Signed);
  static constexpr int kMax = SIGNED ? (1 << (B - 1)) - 1 : (1 << B) - 1;
  static constexpr int kLo = SIGNED ? -kMax : 0;
  static constexpr int kHi = kMax;
};

// RN(a / b) from y = RN(1 / b) without a division: q0 = RN(a y), then one
// remainder correction q = RN(q0 + RN(a - b q0) y) (two fmas). Why q is the
// correctly rounded quotient (the argument is scale-free; Bi is b's 24-bit
// integer significand, "ulp" the spacing of a / b's fp32 grid):
// y = (1 + e) / b with |e| <= Bi 2^-48 < 2^-24, so q0 is within 1.5 ulp of
// a / b and the corrected value before its rounding, z, within 3 2^-24 ulp.
// q can only be wrong if a rounding midpoint m lies between z and a / b, so
// within d <= 3 2^-24 ulp of a / b. Then |a y - m| < 1 ulp (|m e| < 1 ulp,
// and only when M Bi >= 2^49 - 3 2^25, for m's 25-bit odd significand M, does
// it come within d of one ulp; no quotient lies that close to a midpoint in
// that corner, checked exhaustively on the host), so q0 = m +- ulp / 2 is
// within one ulp of a / b, the remainder a - b q0 is exact (Markstein) and
// z - a / b = -e (q0 - a / b), of magnitude below |e| (ulp / 2 + d). As
// a - m b is a nonzero multiple of ulp(b) ulp / 2, d >= ulp / (2 Bi), and
// |e| (Bi + 1) < 1 (Bi (Bi + 1) < 2^48): so |z - a / b| < d and z stays on
// a / b's side of m. Needs a / b and the remainder representable without
// overflow or underflow.
__device__ __forceinline__ float div_by_recip(float a, float b, float y) {
  const float q0 = __fmul_rn(a, y);
  return __fmaf_rn(__fmaf_rn(-q0, b, a), y, q0);
}

// Exact per-element quantisation (the page's operations, IEEE division).
template <int KMODE>
__device__ __forceinline__ uint32_t key_code_exact(float x, float se, float zp) {
  using M = KeySpec<KMODE>;
  float r = rintf(__fsub_rn(__fdiv_rn(x, se), zp));
  r = (r < static_cast<float>(M::kLo)) ? static_cast<float>(M::kLo) : r;
  r = (r > static_cast<float>(M::kHi)) ? static_cast<float>(M::kHi) : r;
  return static_cast<uint32_t>(static_cast<int>(r));
}

// Group min and max with the tie rule of a left-to-right scan (the first of
// equal values wins; only +0 / -0 can tell), used when the fast min or max
// is a zero.
__device__ __forceinline__ void scan_min_max(const float2 (&X)[16], float& mn, float& mx) {
  mn = X[0].x;
  mx = X[0].x;
#pragma unroll
  for (int i = 1; i < 32; ++i) {
    const float v = pair_elem(X, i);
    mn = (v < mn) ? v : mn;
    mx = (v > mx) ? v : mx;
  }
}

// One item's inputs: 16 words of bf16 pairs, or 32 fp32 values.
template <bool F32>
struct ItemIn {
  uint32_t w[F32 ? 32 : 16];
};

template <bool F32>
__device__ __forceinline__ void load_item(const void* base, size_t elem_off, ItemIn<F32>& in) {
  if constexpr (F32) {
    const uint4* q = reinterpret_cast<const uint4*>(static_cast<const float*>(base) + elem_off);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 u = __ldg(q + i);
      in.w[4 * i] = u.x; in.w[4 * i + 1] = u.y; in.w[4 * i + 2] = u.z; in.w[4 * i + 3] = u.w;
    }
  } else {
    load_words16(static_cast<const __nv_bfloat16*>(base) + elem_off, in.w);
  }
}

template <bool F32>
__device__ __forceinline__ void item_to_pairs(const ItemIn<F32>& in, float2 (&P)[16]) {
  if constexpr (F32) {
#pragma unroll
    for (int q = 0; q < 16; ++q) P[q] = make_float2(__uint_as_float(in.w[q]), __uint_as_float(in.w[q + 16]));
  } else {
    words_to_pairs(in.w, P);
  }
}

// ---------------------------------------------------------------------------
// K encode of the group held by this lane. `prefetch` runs once the inputs
// are in registers (it may overwrite `in`).
template <int KMODE, bool F32, typename Prefetch>
__device__ __forceinline__ void encode_key_item(ItemIn<F32>& in, float neg_zero, bool store, uint8_t* codes,
                                                uint16_t* scale_out, uint16_t* zero_out, Prefetch&& prefetch) {
  using M = KeySpec<KMODE>;
  float2 X[16];
  float mn, mx;
  // A NaN anywhere in the group makes both NaN (the page's min / max
  // reductions propagate it), so the NaN-propagating forms are used.
  if constexpr (F32) {
    mn = __uint_as_float(in.w[0]);
    mx = mn;
#pragma unroll
    for (int i = 1; i < 32; ++i) {
      mn = fmin_nan(mn, __uint_as_float(in.w[i]));
      mx = fmax_nan(mx, __uint_as_float(in.w[i]));
    }
  } else {
    // min / max on bf16 pairs (exact: the upcast preserves order)
    __nv_bfloat162 lo2 = *reinterpret_cast<const __nv_bfloat162*>(&in.w[0]);
    __nv_bfloat162 hi2 = lo2;
#pragma unroll
    for (int j = 1; j < 16; ++j) {
      const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&in.w[j]);
      lo2 = __hmin2_nan(lo2, v2);
      hi2 = __hmax2_nan(hi2, v2);
    }
    mn = fmin_nan(__low2float(lo2), __high2float(lo2));
    mx = fmax_nan(__low2float(hi2), __high2float(hi2));
  }
  item_to_pairs(in, X);
  prefetch();
  if (mn == 0.0f || mx == 0.0f) scan_min_max(X, mn, mx);

  // The group's quotients from the reciprocal with one remainder correction
  // (div_by_recip; code_bits below for the elements). scale = RN(range /
  // levels); a range below 2^-100 could make the remainder underflow, which
  // changes neither RN(scale + eps) (= eps) nor the fp16 scale (0). Inf and
  // NaN ranges keep IEEE semantics through the plain product.
  constexpr float kLevels = static_cast<float>(M::SIGNED ? 2 * M::kMax : M::kMax);
  constexpr float kInvLevels = 1.0f / kLevels;
  const float range = __fsub_rn(mx, mn);
  const float scale =
      range <= 3.402823466e38f ? div_by_recip(range, kLevels, kInvLevels) : __fmul_rn(range, kInvLevels);
  const float se = __fadd_rn(scale, kEps);
  const float inv = __frcp_rn(se);
  // zero point: RN(mn / se), or RN((mx + mn) / (2 se)) = RN((mx + mn) / se) / 2
  // for signed keys; a quotient that overflows, or a range that is not finite
  // (an Inf or NaN in the group: se = Inf gives inv = 0 and a NaN remainder,
  // where num / se is a signed zero or NaN), takes IEEE division. The
  // corrected quotient takes the sign of num (se > 0): for num = -0 the
  // correction's exact zero remainder would otherwise turn -0 into +0, and
  // the fp16 zero point keeps that sign.
  const float num = M::SIGNED ? __fadd_rn(mx, mn) : mn;
  const float zq0 = __fmul_rn(num, inv);
  float zq;
  if (fabsf(zq0) <= 3.402823466e38f && range <= 3.402823466e38f) {
    zq = copysignf(div_by_recip(num, se, inv), num);
    if constexpr (M::SIGNED) zq = __fmul_rn(zq, 0.5f);
  } else {
    zq = M::SIGNED ? __fdiv_rn(num, __fmul_rn(2.0f, se)) : __fdiv_rn(num, se);
  }
  const float zp = rintf(zq);
  const float2 nz = f2(neg_zero);
  // Code of a pair as the float bit pattern kMagicBits + rint(RN(RN(x/se) - zp)),
  // RN(x/se) by div_by_recip's correction in packed form, barring overflow
  // of x/se (the caller's range test rejects it) and underflow of the
  // remainder (only when |x/se| < 2^-70, too small to move rint(q - zp)).
  auto code_bits = [&](float2 x) {
    const float2 q0 = mul0(x, f2(inv), nz);  // rounded: it is the quotient's first guess
    const float2 q = fma2(fma2(q0, f2(-se), x), f2(inv), q0);
    return add2(add2(q, f2(-zp)), f2(kMagic));  // RN(q - zp), then rint
  };
  const int lo_bits = static_cast<int>(kMagicBits) + M::kLo;
  const int hi_bits = static_cast<int>(kMagicBits) + M::kHi;
  // The code is monotone in x, so when the group's min and max have codes
  // inside [kLo, kHi] every element does and no clamp is needed (an
  // overflowed quotient gives NaN or Inf, which fails this test).
  const float2 ext = code_bits(make_float2(mn, mx));
  const bool in_range = __float_as_int(ext.x) >= lo_bits && __float_as_int(ext.y) <= hi_bits;

  uint32_t w[M::B];
  if (__all_sync(kFull, in_range)) {
    pack_pairs<M::B, true>(w, [&](int q, uint32_t& lo, uint32_t& hi) {
      const float2 c = code_bits(X[q]);
      lo = __float_as_uint(c.x);
      hi = __float_as_uint(c.y);
    });
  } else {
    // rare: some group of the warp needs the clamp: the page's operations
    // with IEEE division, element by element
    pack_pairs<M::B, true>(w, [&](int q, uint32_t& lo, uint32_t& hi) {
      lo = kMagicBits + key_code_exact<KMODE>(X[q].x, se, zp);
      hi = kMagicBits + key_code_exact<KMODE>(X[q].y, se, zp);
    });
  }
  if (store) {
    store_words<M::B>(codes, w);
    *scale_out = __half_as_ushort(__float2half_rn(scale));
    *zero_out = __half_as_ushort(__float2half_rn(zp));
  }
}

// V encode of the group held by this lane (the whole row's lanes rotate together).
// REP: s_cells is the lane's replica of the compact cell table (bytes, see
// RepCells) and the rare masked path reads the full table from global memory.
// SIGNS_IN_REGS: s_sign is the lane's own 16 sign words (held in registers by
// the caller) instead of the block's shared table.
template <int LPR, int VB, bool F32, bool REP, bool SIGNS_IN_REGS, typename Prefetch>
__device__ __forceinline__ void encode_value_item(ItemIn<F32>& in, int l, const uint32_t* s_sign,
                                                  const void* s_cells, uint32_t rep_bias, float rot_scale,
                                                  float neg_zero, bool store, uint8_t* codes, uint16_t* scale_out,
                                                  Prefetch&& prefetch) {
  uint32_t S[16];
  if constexpr (SIGNS_IN_REGS) {
#pragma unroll
    for (int j = 0; j < 16; ++j) S[j] = s_sign[j];
  } else {
    load_sign_words(s_sign, l, S);
  }
  float2 Y[16];
  if constexpr (F32) {
#pragma unroll
    for (int i = 0; i < 32; ++i) in.w[i] ^= elem_sign(S, i);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) in.w[j] ^= S[j];
  }
  item_to_pairs(in, Y);
  prefetch();
  hadamard_row<LPR>(Y, l);
  const float2 c2 = f2(rot_scale);
#pragma unroll
  for (int q = 0; q < 16; ++q) Y[q] = mul2(Y[q], c2);
  const float rms = __fsqrt_rn(__fmul_rn(group_sum_sq(Y, f2(neg_zero)), 1.0f / kGroup));  // /32 is exact
  const float inv = __frcp_rn(__fadd_rn(rms, kEps));
  uint32_t w[VB];
  if (__all_sync(kFull, __float_as_uint(rms) < 0x7f800000u)) {
    // every group of the warp has a finite RMS: cells are in range unmasked
    pack_pairs<VB, false>(w, [&](int q, uint32_t& lo, uint32_t& hi) {
      if constexpr (REP) {
        lm_index2_rep<VB>(Y[q], inv, rep_bias, lo, hi);
      } else {
        lm_index2_scaled<VB, false>(Y[q], inv, static_cast<const CellEntry*>(s_cells), lo, hi);
      }
    });
  } else {
    const CellEntry* tab = REP ? cell_table<VB>() : static_cast<const CellEntry*>(s_cells);
    pack_pairs<VB, false>(w, [&](int q, uint32_t& lo, uint32_t& hi) {
      lm_index2_scaled<VB, true>(Y[q], inv, tab, lo, hi);
    });
  }
  if (store) {
    store_words<VB>(codes, w);
    *scale_out = __half_as_ushort(__float2half_rn(rms));
  }
}

template <int D, int VB, int KMODE, bool F32, bool ALLOW_REP, bool SNAKE>
__global__ void __launch_bounds__(EncodeShape<D, VB, F32, ALLOW_REP>::kBlockThreads,
                                  EncodeShape<D, VB, F32, ALLOW_REP>::kMinBlocks)
    encode_kernel(EncodeParams p) {
  using G = Geo<D>;
  using M = KeySpec<KMODE>;
  using SH = EncodeShape<D, VB, F32, ALLOW_REP>;
  constexpr int NC = SH::REP ? 1 : CellGrid<VB>::NC;
  constexpr int pdk = D * M::B / 8;
  constexpr int pdv = D * VB / 8;
  constexpr int NG = D / kGroup;
  __shared__ CellEntry s_cells[NC];
  __shared__ __align__(16) uint32_t s_sign[D / 2];
  extern __shared__ __align__(128) uint8_t s_ring[];
  {
    const CellEntry* tab = cell_table<VB>();
    if constexpr (SH::REP) {
      CellEntry* rep = reinterpret_cast<CellEntry*>(s_ring + SH::Ring::kBlockBytes);
      for (int i = threadIdx.x; i < RepCells<VB>::kCount * 16; i += blockDim.x) rep[i] = tab[RepCells<VB>::kLo + (i >> 4)];
    } else {
      for (int i = threadIdx.x; i < NC; i += blockDim.x) s_cells[i] = tab[i];
    }
    fill_sign_words<D>(s_sign);
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();

  const int lane = threadIdx.x & 31;
  const int sub = lane / G::LPR;
  const int l = lane % G::LPR;
  const int n_warps = gridDim.x * (blockDim.x >> 5);
  const int tiles = (p.rows + G::RPW - 1) / G::RPW;
  const int items = 2 * tiles;
  const int gw = warp_index();

  const ItemOrder<SNAKE> ord{n_warps, gw, tiles};
  using R = typename SH::Ring;
  const void* cells = static_cast<const void*>(s_cells);
  const uint32_t rep_bias =
      SH::REP ? rep_bias_for<VB>(static_cast<uint32_t>(__cvta_generic_to_shared(s_ring + R::kBlockBytes + 8 * (lane & 15))))
              : 0u;
  uint8_t* lane_ring = s_ring + (threadIdx.x >> 5) * (R::kStages * R::kStageBytes) + lane * R::kLaneBytes;
  const uint32_t lane_ring_sh = static_cast<uint32_t>(__cvta_generic_to_shared(lane_ring));
  const int swz = R::swz(lane);
  // Step k's inputs go to slot k mod kStages. Every issue commits one copy
  // group (empty past the end), so wait_group(kStages - 1) after issuing step
  // k + kStages - 1 means "step k landed". The first step's copies go out
  // alone and the next ones only once they have landed, so that at the start
  // of a launch the memory system serves every warp's first item before
  // anyone's second (8B-layer encode 8.2 -> 7.8 us).
  auto issue = [&](int k) {
    const int it = ord.item(k);
    if (it < items) {
      const int r0 = ord.tile(it) * G::RPW + sub;
      const int r = r0 < p.rows ? r0 : p.rows - 1;
      const char* src = static_cast<const char*>(ord.is_v(it, k) ? p.v : p.k) +
                        (static_cast<size_t>(r) * D + kGroup * l) * (F32 ? 4 : 2);
      const uint32_t dst = lane_ring_sh + (k & (R::kStages - 1)) * R::kStageBytes;
      if (TQ_CHECK(r >= 0 && r < p.rows, p.err)) {
#pragma unroll
        for (int j = 0; j < R::kChunks; ++j) cp_async16(dst + 16 * (j ^ swz), src + 16 * j);
      }
    }
    cp_async_commit();
  };
  // The wide (512-thread, replicated-table) shape keeps each lane's sign
  // words in registers for the whole launch: 16 fewer shared-memory
  // wavefronts per V item (long-context v8 encode 320 -> 310 us). The
  // 256-thread shapes would spill with them and measured slower.
  constexpr bool kRegSigns = SH::REP;
  uint32_t S_l[kRegSigns ? 16 : 1];
  if constexpr (kRegSigns) load_sign_words(s_sign, l, S_l);
  const uint32_t* signs = kRegSigns ? static_cast<const uint32_t*>(S_l) : static_cast<const uint32_t*>(s_sign);
  issue(0);
  cp_async_wait<0>();
#pragma unroll
  for (int j = 1; j < R::kStages - 1; ++j) issue(j);
  auto no_prefetch = [] {};
  for (int k = 0;; ++k) {
    const int it = ord.item(k);
    if (it >= items) break;
    issue(k + R::kStages - 1);
    cp_async_wait<R::kStages - 1>();
    ItemIn<F32> in;
    {
      const uint8_t* slot = lane_ring + (k & (R::kStages - 1)) * R::kStageBytes;
#pragma unroll
      for (int j = 0; j < R::kChunks; ++j) {
        const uint4 u = *reinterpret_cast<const uint4*>(slot + 16 * (j ^ swz));
        in.w[4 * j] = u.x; in.w[4 * j + 1] = u.y; in.w[4 * j + 2] = u.z; in.w[4 * j + 3] = u.w;
      }
    }
    const int r0 = ord.tile(it) * G::RPW + sub;
    const bool valid = r0 < p.rows;
    const int r = valid ? r0 : p.rows - 1;
    const int bh = fast_div(r, p.tdiv);
    const long long orow = static_cast<long long>(bh) * p.t_cap + p.t_off + (r - bh * p.T);
    const bool store = valid && TQ_CHECK(orow >= 0 && orow < p.cache_rows, p.err);
    if (!ord.is_v(it, k)) {
      encode_key_item<KMODE, F32>(in, p.neg_zero, store, p.k_codes + orow * pdk + 4 * M::B * l,
                                  p.k_scales + orow * NG + l, p.k_zeros + orow * NG + l, no_prefetch);
    } else {
      encode_value_item<G::LPR, VB, F32, SH::REP, kRegSigns>(in, l, signs, cells, rep_bias, p.rot_scale, p.neg_zero, store,
                                         p.v_codes + orow * pdv + 4 * VB * l, p.v_scales + orow * NG + l,
                                         no_prefetch);
    }
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// Decode. An item's inputs: the packed words of the group and its fp16 scale
// (and zero point for K).
template <int WORDS>
struct PackedIn {
  uint32_t w[WORDS];
  uint32_t sz;  // scale in the low half, zero point (K) in the high half
};

template <int KB, int VB>
__device__ __forceinline__ void load_packed_item(const DecodeParams& p, bool is_v, long long irow, int l,
                                                 PackedIn<(KB > VB ? KB : VB)>& in) {
  constexpr int W = KB > VB ? KB : VB;
  if (!TQ_CHECK(irow >= 0 && irow < p.cache_rows, p.err)) {
#pragma unroll
    for (int k = 0; k < W; ++k) in.w[k] = 0u;
    in.sz = 0u;
    return;
  }
  if (is_v) {
    uint32_t t[VB];
    load_words<VB>(p.v_codes + irow * p.pdv + 4 * VB * l, t);
#pragma unroll
    for (int k = 0; k < W; ++k) in.w[k] = (k < VB) ? t[k < VB ? k : 0] : 0u;
    in.sz = __ldg(p.v_scales + irow * p.ng + l);
  } else {
    uint32_t t[KB];
    load_words<KB>(p.k_codes + irow * p.pdk + 4 * KB * l, t);
#pragma unroll
    for (int k = 0; k < W; ++k) in.w[k] = (k < KB) ? t[k < KB ? k : 0] : 0u;
    in.sz = static_cast<uint32_t>(__ldg(p.k_scales + irow * p.ng + l)) |
            (static_cast<uint32_t>(__ldg(p.k_zeros + irow * p.ng + l)) << 16);
  }
}

// K decode of one group: x = (code + zero) * scale, zero and scale from fp16.
// Signed codes are first offset to [0, 255] by flipping their bytes' sign
// bits (code + 128). The zero point is an integer (or +-Inf, or NaN), so
// zero minus an integer bias below 2^24 is exact, and RN(code + zero), the
// page's sum, comes out of one rounding: for 8-bit codes a byte permute
// makes two fp16 values 1024 + byte and a mixed-precision add widens each
// and adds zero - 1024 - offset (FMA pipe); narrower codes become the floats
// 1.5 * 2^23 + offset + code (a shift and a mask) plus zero - 1.5 * 2^23 -
// offset. Then one rounding of the product with the scale.
// `prefetch` runs once the packed inputs are consumed (it may overwrite `in`).
template <int KMODE, int W, typename Prefetch>
__device__ __forceinline__ void decode_key_item(const PackedIn<W>& in, float (&x)[32], Prefetch&& prefetch) {
  using M = KeySpec<KMODE>;
  constexpr float kOffset = M::SIGNED ? 128.0f : 0.0f;
  const float s = __half2float(__ushort_as_half(static_cast<uint16_t>(in.sz & 0xffffu)));
  const float z = __half2float(__ushort_as_half(static_cast<uint16_t>(in.sz >> 16)));
  float cz[32];  // RN(code + zero)
  if constexpr (M::B == 8) {
    const float zh = __fsub_rn(z, 1024.0f + kOffset);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t wk = M::SIGNED ? (in.w[k] ^ 0x80808080u) : in.w[k];
      const uint32_t h01 = __byte_perm(wk, 0x64646464u, 0x4140u);
      const uint32_t h23 = __byte_perm(wk, 0x64646464u, 0x4342u);
      cz[4 * k] = add_f16_f32<false>(h01, zh);
      cz[4 * k + 1] = add_f16_f32<true>(h01, zh);
      cz[4 * k + 2] = add_f16_f32<false>(h23, zh);
      cz[4 * k + 3] = add_f16_f32<true>(h23, zh);
    }
    prefetch();
  } else {
    const float zb = __fsub_rn(z, kMagic + kOffset);
    uint32_t w[M::B];
#pragma unroll
    for (int k = 0; k < M::B; ++k) w[k] = in.w[k];
    uint32_t cb[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) cb[i] = unpack_code<M::B>(w, i) | kMagicBits;
    prefetch();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 f = add2(make_float2(__uint_as_float(cb[2 * i]), __uint_as_float(cb[2 * i + 1])), f2(zb));
      cz[2 * i] = f.x;
      cz[2 * i + 1] = f.y;
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 g = mul2(make_float2(cz[2 * i], cz[2 * i + 1]), f2(s));  // RN(RN(code + zero) * scale)
    x[2 * i] = g.x;
    x[2 * i + 1] = g.y;
  }
}

template <bool F32>
__device__ __forceinline__ void store_group(void* base, size_t off, const float (&x)[32]) {
  if constexpr (!F32) {
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * j], x[2 * j + 1]);
      w[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    uint4* q = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off);
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  } else {
    float4* q = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
  }
}

// Centroid tables in shared memory. 8-bit codes index 256 entries, which 32
// lanes would hit with bank conflicts, so that table is kept once per bank:
// entry c for lane L at word 32 c + L (s_cent is then offset by the lane).
// Smaller tables (<= 32 entries) map every entry to its own bank already.
template <int VB>
struct CentroidTable {
  static constexpr int kRep = VB == 8 ? 32 : 1;
  static constexpr int kWords = (1 << VB) * kRep;
};

template <int VB>
__device__ __forceinline__ void fill_centroids(float* s_cent) {
  constexpr int rep = CentroidTable<VB>::kRep;
  for (int i = threadIdx.x; i < CentroidTable<VB>::kWords; i += blockDim.x) s_cent[i] = centroid_table<VB>()[i / rep];
}

// Centroid of code i of the group, read at a byte offset formed straight from
// the packed words (shift and mask; codes straddling two words are unpacked
// first). `cent` is the table, already offset by the lane when replicated.
template <int VB>
__device__ __forceinline__ float centroid_at(const float* cent, const uint32_t (&w)[VB], int i) {
  constexpr int kShift = VB == 8 ? 7 : 2;  // bytes per code step: 128 when replicated, else 4
  constexpr uint32_t kMask = ((1u << VB) - 1u) << kShift;
  const int bit = i * VB, word = bit >> 5, off = bit & 31;
  uint32_t byte_off;
  if (off + VB > 32) {
    byte_off = unpack_code<VB>(w, i) << kShift;
  } else if (off >= kShift) {
    byte_off = (w[word] >> (off - kShift)) & kMask;
  } else {
    byte_off = (w[word] << (kShift - off)) & kMask;
  }
  return *reinterpret_cast<const float*>(reinterpret_cast<const char*>(cent) + byte_off);
}

// V decode of one group into its output words: 16 words of bf16 pairs or 32
// fp32 values, in element order. ROT: leave the values in the rotated domain
// (dequantScaled / decodeValuesRotated: centroid * scale only).
// SIGNS_IN_REGS: s_sign is the lane's own 16 sign words (held in registers by
// the caller) instead of the block's shared table.
template <int LPR, int VB, bool F32, bool ROT, bool SIGNS_IN_REGS, int W, typename Prefetch>
__device__ __forceinline__ void decode_value_words(const PackedIn<W>& in, int l, const uint32_t* s_sign,
                                                   const float* s_cent, float rot_scale, float neg_zero,
                                                   uint32_t (&o)[F32 ? 32 : 16], Prefetch&& prefetch) {
  const float s = __half2float(__ushort_as_half(static_cast<uint16_t>(in.sz & 0xffffu)));
  const float2 nz = f2(neg_zero);
  float2 Y[16];
  {
    uint32_t w[VB];
#pragma unroll
    for (int k = 0; k < VB; ++k) w[k] = in.w[k];
#pragma unroll
    for (int q = 0; q < 16; ++q) Y[q] = make_float2(centroid_at<VB>(s_cent, w, q), centroid_at<VB>(s_cent, w, q + 16));
  }
  prefetch();
#pragma unroll
  for (int q = 0; q < 16; ++q) Y[q] = mul0(Y[q], f2(s), nz);  // feeds the butterflies: must stay rounded
  uint32_t S[16];
  if constexpr (ROT) {
#pragma unroll
    for (int j = 0; j < 16; ++j) S[j] = 0u;  // no signs in the rotated domain
  } else {
    hadamard_row<LPR>(Y, l);
    const float2 c2 = f2(rot_scale);
#pragma unroll
    for (int q = 0; q < 16; ++q) Y[q] = mul2(Y[q], c2);
    if constexpr (SIGNS_IN_REGS) {
#pragma unroll
      for (int j = 0; j < 16; ++j) S[j] = s_sign[j];
    } else {
      load_sign_words(s_sign, l, S);
    }
  }
  if constexpr (!F32) {
    // round to bf16, then apply the signs on the packed words (exact)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const __nv_bfloat162 a = __floats2bfloat162_rn(Y[2 * j].x, Y[2 * j + 1].x);
      const __nv_bfloat162 b = __floats2bfloat162_rn(Y[2 * j].y, Y[2 * j + 1].y);
      o[j] = *reinterpret_cast<const uint32_t*>(&a) ^ S[j];
      o[j + 8] = *reinterpret_cast<const uint32_t*>(&b) ^ S[j + 8];
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(pair_elem(Y, i)) ^ elem_sign(S, i);
  }
}

// The same, stored to out + out_off (elements) when `store`.
template <int LPR, int VB, bool F32, bool ROT, bool SIGNS_IN_REGS, int W, typename Prefetch>
__device__ __forceinline__ void decode_value_item(const PackedIn<W>& in, int l, const uint32_t* s_sign,
                                                  const float* s_cent, float rot_scale, float neg_zero,
                                                  bool store, void* out, size_t out_off, Prefetch&& prefetch) {
  uint32_t o[F32 ? 32 : 16];
  decode_value_words<LPR, VB, F32, ROT, SIGNS_IN_REGS>(in, l, s_sign, s_cent, rot_scale, neg_zero, o, prefetch);
  if (!store) return;
  constexpr int kElem = F32 ? 4 : 2;
  uint4* q = reinterpret_cast<uint4*>(static_cast<char*>(out) + out_off * kElem);
#pragma unroll
  for (int i = 0; i < (F32 ? 8 : 4); ++i) q[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
}

// Decode staging, a template argument chosen per launch like the encode's
// item order:
//   SHORT (at most kSnakeSteps steps per warp): the packed inputs of the next
//   two items are in flight while an item computes, so the first steps of a
//   launch wait less on memory; the sign words come from shared memory.
//   Long launches: one item ahead, and (bf16 outputs) each lane keeps its 16
//   sign words in registers for the whole launch, which takes 16 wavefronts
//   of shared traffic off every V item (the V items are bound by
//   shared-memory and shuffle traffic).
// Measured: the [1, 8, 4096, 128] layer decodes in 7.11 instead of 7.37 us
// with two items ahead (7.60 us with the register signs); the
// [32, 8, 8192, 128] cache in 289.8 instead of 303.3 us with the register
// signs (308.2 us with two items ahead). Both at once spill.
template <int D, int VB, int KMODE, bool F32, bool ROT, bool SHORT>
__global__ void __launch_bounds__(kThreads, kDecodeMinBlocks) decode_kernel(DecodeParams p) {
  using G = Geo<D>;
  using M = KeySpec<KMODE>;
  constexpr int W = M::B > VB ? M::B : VB;
  constexpr int kAhead = SHORT ? 2 : 1;
  __shared__ float s_cent[CentroidTable<VB>::kWords];
  __shared__ __align__(16) uint32_t s_sign[D / 2];
  fill_centroids<VB>(s_cent);
  fill_sign_words<D>(s_sign);
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();

  const int lane = threadIdx.x & 31;
  const int sub = lane / G::LPR;
  const int l = lane % G::LPR;
  const int n_warps = gridDim.x * (blockDim.x >> 5);
  const int tiles = (p.rows + G::RPW - 1) / G::RPW;
  const int items = 2 * tiles;
  const int gw = warp_index();

  auto item_irow = [&](int it) {
    const int r0 = (it >> 1) * G::RPW + sub;
    const int r = r0 < p.rows ? r0 : p.rows - 1;
    const int bh = fast_div(r, p.tdiv);
    return static_cast<long long>(bh) * p.t_cap + (r - bh * p.T);
  };
  // The lane's sign words stay in registers for bf16 outputs of long
  // launches (fp32 outputs would spill with them).
  constexpr bool kRegSigns = !SHORT && !F32 && !ROT;
  uint32_t S_l[kRegSigns ? 16 : 1];
  if constexpr (kRegSigns) load_sign_words(s_sign, l, S_l);
  const uint32_t* signs = kRegSigns ? static_cast<const uint32_t*>(S_l) : static_cast<const uint32_t*>(s_sign);
  // Step k takes item gw + k * n_warps, a V item when (item ^ k) is odd.
  PackedIn<W> in, in2;
  int step = 0;
  if (gw < items) load_packed_item<M::B, VB>(p, (gw & 1) != 0, item_irow(gw), l, in);
  if constexpr (SHORT) {
    const int it1 = gw + n_warps;
    if (it1 < items) load_packed_item<M::B, VB>(p, ((it1 ^ 1) & 1) != 0, item_irow(it1), l, in2);
  }
  for (int it = gw; it < items; it += n_warps, ++step) {
    const bool is_v = ((it ^ step) & 1) != 0;
    const int r0 = (it >> 1) * G::RPW + sub;
    const bool valid = r0 < p.rows && TQ_CHECK(r0 >= 0, p.err);
    const int r = valid ? r0 : p.rows - 1;
    const size_t out_off = static_cast<size_t>(r) * D + kGroup * l;

    // the loads of step + kAhead are issued once this item's inputs are consumed
    const int nx = it + kAhead * n_warps;
    auto prefetch = [&]() {
      if constexpr (SHORT) {
        in = in2;
        if (nx < items) load_packed_item<M::B, VB>(p, ((nx ^ (step + 2)) & 1) != 0, item_irow(nx), l, in2);
      } else {
        if (nx < items) load_packed_item<M::B, VB>(p, ((nx ^ (step + 1)) & 1) != 0, item_irow(nx), l, in);
      }
    };
    if (!is_v) {
      float x[32];
      decode_key_item<KMODE>(in, x, prefetch);
      if (valid) store_group<F32>(p.k_out, out_off, x);
    } else {
      decode_value_item<G::LPR, VB, F32, ROT, kRegSigns>(in, l, signs,
                                                       s_cent + (CentroidTable<VB>::kRep > 1 ? lane : 0),
                                                       p.rot_scale, p.neg_zero, valid, p.v_out, out_off, prefetch);
    }
  }
}

// ---------------------------------------------------------------------------
template <typename K>
inline int resident_blocks(K kernel, int dyn_smem = 0, int threads = kThreads) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, dyn_smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  return per_sm * sm_count();
}

// Opt a kernel into dynamic shared memory above the default limit, with the
// largest shared-memory carveout; returns its resident blocks on the device.
template <typename K>
inline int prepare_dyn_smem(K kernel, int dyn_smem, int threads = kThreads) {
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem);
  cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  return resident_blocks(kernel, dyn_smem, threads);
}

inline int grid_for(long long items, int resident, int threads = kThreads) {
  const long long needed = (items + (threads / 32) - 1) / (threads / 32);
  return static_cast<int>(needed < resident ? needed : resident);
}

// Launch with programmatic stream serialization (see the file comment).
template <typename Params>
inline cudaError_t launch_pdl(void (*kernel)(Params), int grid, const Params& p, cudaStream_t s, int dyn_smem = 0,
                              int threads = kThreads) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = dyn_smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int D, int VB, int KMODE, bool F32, bool ALLOW_REP, bool SNAKE>
cudaError_t launch_encode_shape(const EncodeParams& p, cudaStream_t s, int grid) {
  using SH = EncodeShape<D, VB, F32, ALLOW_REP>;
  const cudaError_t e =
      launch_pdl(encode_kernel<D, VB, KMODE, F32, ALLOW_REP, SNAKE>, grid, p, s, SH::kSmem, SH::kBlockThreads);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Resident blocks of an encode kernel on this device (opting it into its
// dynamic shared memory first), computed once per instantiation.
template <int D, int VB, int KMODE, bool F32, bool ALLOW_REP, bool SNAKE>
int encode_resident() {
  using SH = EncodeShape<D, VB, F32, ALLOW_REP>;
  static const int resident =
      prepare_dyn_smem(encode_kernel<D, VB, KMODE, F32, ALLOW_REP, SNAKE>, SH::kSmem, SH::kBlockThreads);
  return resident;
}

template <int D, int VB, int KMODE, bool F32>
cudaError_t launch_encode_t(const EncodeParams& p, cudaStream_t s) {
  const long long items = 2LL * ((p.rows + Geo<D>::RPW - 1) / Geo<D>::RPW);
  if constexpr (EncodeShape<D, VB, F32, true>::REP) {
    if (p.rows >= kRepMinRows) {
      constexpr int threads = EncodeShape<D, VB, F32, true>::kBlockThreads;
      const int grid = grid_for(items, encode_resident<D, VB, KMODE, F32, true, false>(), threads);
      return launch_encode_shape<D, VB, KMODE, F32, true, false>(p, s, grid);
    }
  }
  constexpr int threads = EncodeShape<D, VB, F32, false>::kBlockThreads;
  const int resident = std::min(encode_resident<D, VB, KMODE, F32, false, false>(),
                                encode_resident<D, VB, KMODE, F32, false, true>());
  const int grid = grid_for(items, resident, threads);
  if (items <= static_cast<long long>(kSnakeSteps) * grid * (threads / 32))
    return launch_encode_shape<D, VB, KMODE, F32, false, true>(p, s, grid);
  return launch_encode_shape<D, VB, KMODE, F32, false, false>(p, s, grid);
}

}  // namespace tq

#include "tq_decode_bulk.cuh"

namespace tq {

template <int D, int VB, int KMODE, bool F32, bool ROT>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t s) {
  if constexpr (!F32) {
    if (bulk_decode_ok<D>(p, true)) return launch_decode_bulk<D, VB, KMODE, ROT>(p, s);
  }
  static const int resident = std::min(resident_blocks(decode_kernel<D, VB, KMODE, F32, ROT, false>),
                                       resident_blocks(decode_kernel<D, VB, KMODE, F32, ROT, true>));
  const long long items = 2LL * ((p.rows + Geo<D>::RPW - 1) / Geo<D>::RPW);
  const int grid = grid_for(items, resident);
  const bool short_launch = items <= static_cast<long long>(kSnakeSteps) * grid * (kThreads / 32);
  const cudaError_t e = short_launch ? launch_pdl(decode_kernel<D, VB, KMODE, F32, ROT, true>, grid, p, s)
                                     : launch_pdl(decode_kernel<D, VB, KMODE, F32, ROT, false>, grid, p, s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D, int VB, bool F32>
cudaError_t launch_encode_vb(const EncodeParams& p, cudaStream_t s) {
  switch (p.kmode) {
    case kK2: return launch_encode_t<D, VB, kK2, F32>(p, s);
    case kK4: return launch_encode_t<D, VB, kK4, F32>(p, s);
    case kK5: return launch_encode_t<D, VB, kK5, F32>(p, s);
    case kK8: return launch_encode_t<D, VB, kK8, F32>(p, s);
    default: return launch_encode_t<D, VB, kK8Signed, F32>(p, s);
  }
}

template <int D, int VB, bool F32, bool ROT>
cudaError_t launch_decode_vb(const DecodeParams& p, cudaStream_t s) {
  switch (p.kmode) {
    case kK2: return launch_decode_t<D, VB, kK2, F32, ROT>(p, s);
    case kK4: return launch_decode_t<D, VB, kK4, F32, ROT>(p, s);
    case kK5: return launch_decode_t<D, VB, kK5, F32, ROT>(p, s);
    case kK8: return launch_decode_t<D, VB, kK8, F32, ROT>(p, s);
    default: return launch_decode_t<D, VB, kK8Signed, F32, ROT>(p, s);
  }
}

template <int D, bool F32>
cudaError_t launch_encode_dt(const EncodeParams& p, int v_bits, cudaStream_t s) {
  switch (v_bits) {
    case 2: return launch_encode_vb<D, 2, F32>(p, s);
    case 3: return launch_encode_vb<D, 3, F32>(p, s);
    case 4: return launch_encode_vb<D, 4, F32>(p, s);
    case 5: return launch_encode_vb<D, 5, F32>(p, s);
    default: return launch_encode_vb<D, 8, F32>(p, s);
  }
}

template <int D, bool F32, bool ROT>
cudaError_t launch_decode_dt(const DecodeParams& p, int v_bits, cudaStream_t s) {
  switch (v_bits) {
    case 2: return launch_decode_vb<D, 2, F32, ROT>(p, s);
    case 3: return launch_decode_vb<D, 3, F32, ROT>(p, s);
    case 4: return launch_decode_vb<D, 4, F32, ROT>(p, s);
    case 5: return launch_decode_vb<D, 5, F32, ROT>(p, s);
    default: return launch_decode_vb<D, 8, F32, ROT>(p, s);
  }
}



// ---------------------------------------------------------------------------
// unrotateValues: the inverse rotation (Hadamard transform, then signs) of
// rows of D values in fp32 arithmetic, returned in the input's type. Same
// lane layout as the codecs: lane l of a row owns elements [32l, 32l+32).
template <int D, bool F32>
__global__ void __launch_bounds__(kThreads) unrotate_kernel(UnrotateParams p) {
  using G = Geo<D>;
  __shared__ __align__(16) uint32_t s_sign[D / 2];
  fill_sign_words<D>(s_sign);
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int sub = lane / G::LPR;
  const int l = lane % G::LPR;
  const int n_warps = gridDim.x * (blockDim.x >> 5);
  const int tiles = (p.rows + G::RPW - 1) / G::RPW;
  uint32_t S[16];
  load_sign_words(s_sign, l, S);
  for (int tile = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); tile < tiles; tile += n_warps) {
    const int r0 = tile * G::RPW + sub;
    const bool valid = r0 < p.rows && TQ_CHECK(r0 >= 0, p.err);
    const size_t off = static_cast<size_t>(valid ? r0 : p.rows - 1) * D + kGroup * l;
    ItemIn<F32> in;
    load_item<F32>(p.x, off, in);
    float2 Y[16];
    item_to_pairs(in, Y);
    hadamard_row<G::LPR>(Y, l);
#pragma unroll
    for (int q = 0; q < 16; ++q) Y[q] = mul2(Y[q], f2(p.rot_scale));
    if (!valid) continue;
    if constexpr (!F32) {
      uint32_t o[16];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(Y[2 * j].x, Y[2 * j + 1].x);
        const __nv_bfloat162 b = __floats2bfloat162_rn(Y[2 * j].y, Y[2 * j + 1].y);
        o[j] = *reinterpret_cast<const uint32_t*>(&a) ^ S[j];
        o[j + 8] = *reinterpret_cast<const uint32_t*>(&b) ^ S[j + 8];
      }
      uint4* q = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + off);
#pragma unroll
      for (int i = 0; i < 4; ++i) q[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    } else {
      float x[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(__float_as_uint(pair_elem(Y, i)) ^ elem_sign(S, i));
      store_group<true>(p.out, off, x);
    }
  }
}

template <int D>
cudaError_t launch_unrotate(const UnrotateParams& p, bool bf16, cudaStream_t s) {
  const long long tiles = (p.rows + Geo<D>::RPW - 1) / Geo<D>::RPW;
  if (bf16) {
    static const int resident = resident_blocks(unrotate_kernel<D, false>);
    return launch_pdl(unrotate_kernel<D, false>, grid_for(tiles, resident), p, s);
  }
  static const int resident = resident_blocks(unrotate_kernel<D, true>);
  return launch_pdl(unrotate_kernel<D, true>, grid_for(tiles, resident), p, s);
}

}  // namespace tq
