// Device building blocks of the TurboQuant codec kernels.
//
// Thread layout: every lane holds 8 consecutive head_dim elements of one row
// (one 16-byte load of bf16). A 32-element quantisation group is 4 adjacent
// lanes. A row uses D/8 lanes for D <= 256 (so a warp holds 4, 2 or 1 rows);
// for D = 512 a lane holds two 8-element chunks, at elements 8l and 256 + 8l.
//
// Rounding contract: every floating-point step is one IEEE binary32 operation
// with round-to-nearest-even (the __f*_rn intrinsics, rintf, IEEE sqrt and
// division; this translation unit is built with -fmad=false), taken in the
// order the codec page applies its ops (page "@mlx-bun/inference 0.0.0-stage
// -> 1.0.0", file package/src/kernels/turboquant/ops.ts). Reductions whose
// order is not fixed by the page use one fixed tree (see group_sum_sq and the
// Hadamard stage order), so the results are deterministic.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <limits>

#include "tq_tables.cuh"

namespace tq {

constexpr int kGroup = 32;     // BLOCK_SIZE on the ops.ts page
constexpr float kEps = 1e-8f;  // the page's eps as an fp32 scalar
constexpr unsigned kFull = 0xffffffffu;

template <int D>
struct Geo {
  static_assert(D == 64 || D == 128 || D == 256 || D == 512, "head_dim");
  static constexpr int CH = (D == 512) ? 2 : 1;       // 8-element chunks per lane
  static constexpr int LPR = (D >= 256) ? 32 : D / 8;  // lanes per row
  static constexpr int RPW = 32 / LPR;                 // rows per warp
};

// Byte offset, within a packed row of `bits`-bit codes, of the 8 codes of
// chunk c of lane l (elements c*256 + 8l ... +7).
template <int BITS>
__device__ __forceinline__ int chunk_byte(int c, int l) { return (c * 32 + l) * BITS; }

// Element offset of chunk c of lane l within a row.
__device__ __forceinline__ int chunk_elem(int c, int l) { return c * 256 + l * 8; }

// ---------------------------------------------------------------------------
// Loads and stores of 8 consecutive elements (16-byte aligned).
__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // bf16 -> fp32 is exact: the high half of the word
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ void store8(float* p, const float (&x)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&x)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------------------
// Rotation: y = H x / sqrt(D) (Sylvester order) for the row held by the LPR
// lanes of this row. Radix-2 stages in ascending stride: 1, 2, 4 inside a
// chunk, 8 .. 8*(LPR/2) across lanes (xor shuffles), then 256 across the two
// chunks of D = 512. Stage h maps (a, b) = (x[i], x[i+h]) to (a + b, a - b).
// The cross-lane update x' = fma(x, s, partner) with s = +1 (lower lane) or
// -1 (upper lane) is exactly one rounded add or subtract.
template <int D>
__device__ __forceinline__ void hadamard_unnormalised(float (&x)[Geo<D>::CH][8], int l) {
  constexpr int CH = Geo<D>::CH;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if ((i & h) == 0) {
          const float a = x[c][i], b = x[c][i + h];
          x[c][i] = __fadd_rn(a, b);
          x[c][i + h] = __fsub_rn(a, b);
        }
      }
    }
  }
#pragma unroll
  for (int m = 1; m < Geo<D>::LPR; m <<= 1) {
    const float s = (l & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float p = __shfl_xor_sync(kFull, x[c][i], m);
        x[c][i] = __fmaf_rn(x[c][i], s, p);
      }
    }
  }
  if constexpr (CH == 2) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float a = x[0][i], b = x[1][i];
      x[0][i] = __fadd_rn(a, b);
      x[1][i] = __fsub_rn(a, b);
    }
  }
}

// Multiply by -1 where the sign table says so (exact: flips the sign bit).
__device__ __forceinline__ void apply_signs(float (&x)[8], uint32_t neg_bits) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[i] = __uint_as_float(__float_as_uint(x[i]) ^ (((neg_bits >> i) & 1u) << 31));
  }
}

template <int D>
__device__ __forceinline__ uint32_t sign_byte(int idx) {
  if constexpr (D == 64) return kSignNeg64[idx];
  else if constexpr (D == 128) return kSignNeg128[idx];
  else if constexpr (D == 256) return kSignNeg256[idx];
  else return kSignNeg512[idx];
}

// ---------------------------------------------------------------------------
// Group reductions over the 4 lanes (32 elements) of a quantisation group.

// Min and max with the tie rule of a left-to-right scan (the first of equal
// values wins, which only matters for +0 / -0): in-lane in element order,
// then across lanes preferring the lower lane.
__device__ __forceinline__ void group_min_max(const float (&x)[8], int l, float& mn, float& mx) {
  mn = x[0];
  mx = x[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) {
    mn = (x[i] < mn) ? x[i] : mn;
    mx = (x[i] > mx) ? x[i] : mx;
  }
#pragma unroll
  for (int m = 1; m <= 2; m <<= 1) {
    const float omn = __shfl_xor_sync(kFull, mn, m);
    const float omx = __shfl_xor_sync(kFull, mx, m);
    const bool partner_lower = (l & m) != 0;
    mn = (omn < mn || (omn == mn && partner_lower)) ? omn : mn;
    mx = (omx > mx || (omx == mx && partner_lower)) ? omx : mx;
  }
}

// Sum of squares of the group's 32 elements as a pairwise tree: within a lane
// ((0,1),(2,3)),((4,5),(6,7)); then lanes (0,1),(2,3); then the two halves.
// Addition is commutative in IEEE arithmetic, so all 4 lanes get equal bits.
__device__ __forceinline__ float group_sum_sq(const float (&y)[8]) {
  float q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = __fmul_rn(y[i], y[i]);
  const float s01 = __fadd_rn(q[0], q[1]), s23 = __fadd_rn(q[2], q[3]);
  const float s45 = __fadd_rn(q[4], q[5]), s67 = __fadd_rn(q[6], q[7]);
  float s = __fadd_rn(__fadd_rn(s01, s23), __fadd_rn(s45, s67));
  s = __fadd_rn(s, __shfl_xor_sync(kFull, s, 1));
  s = __fadd_rn(s, __shfl_xor_sync(kFull, s, 2));
  return s;
}

// ---------------------------------------------------------------------------
// Lloyd-Max index = count(boundaries < u) (ops.ts, searchsorted).
//
// 2 and 3 bits: compare against the 3 or 7 boundaries as immediates.
// 4, 5, 8 bits: a cell table. cell(u) = clamp(floor((u - lo) * 2^k), 0, n-1)
// is monotone in u, so every boundary in a lower cell than u is below u and
// every boundary in a higher cell is at or above u; each cell holds at most
// one boundary (the grid step is below the table's smallest boundary gap),
// which is compared explicitly. The table is built at compile time with the
// same two fp32 operations (the product by 2^k is exact) and checked against
// the plain count by the tests on values at and next to every boundary.
struct CellEntry {
  float b;   // the boundary inside this cell, or +Inf
  int base;  // number of boundaries in lower cells
};

template <int BITS>
struct CellGrid;
template <>
struct CellGrid<4> {
  static constexpr float lo = -2.5f, scale = 4.0f;
  static constexpr int n = 20;
};
template <>
struct CellGrid<5> {
  static constexpr float lo = -3.25f, scale = 8.0f;
  static constexpr int n = 52;
};
template <>
struct CellGrid<8> {
  static constexpr float lo = -4.5f, scale = 64.0f;
  static constexpr int n = 576;
};

template <int N>
struct CellTable {
  CellEntry e[N];
};

template <int BITS>
__host__ __device__ constexpr float lm_boundary(int j) {
  if constexpr (BITS == 2) return LloydMax2::boundary(j);
  else if constexpr (BITS == 3) return LloydMax3::boundary(j);
  else if constexpr (BITS == 4) return LloydMax4::boundary(j);
  else if constexpr (BITS == 5) return LloydMax5::boundary(j);
  else return LloydMax8::boundary(j);
}

// Cell of u on the grid of a table, in the same two fp32 operations the
// device uses (the product by a power of two is exact).
template <int BITS>
constexpr int grid_cell(float u) {
  const float d = u - CellGrid<BITS>::lo;  // one fp32 rounding
  const float s = d * CellGrid<BITS>::scale;
  return static_cast<int>(s);
}

// True when every boundary lies inside the grid and no cell holds two.
template <int BITS>
constexpr bool cell_grid_fits() {
  int prev = -1;
  for (int j = 0; j < (1 << BITS) - 1; ++j) {
    const float b = lm_boundary<BITS>(j);
    if (b < CellGrid<BITS>::lo) return false;
    const int c = grid_cell<BITS>(b);
    if (c <= prev || c >= CellGrid<BITS>::n) return false;
    prev = c;
  }
  return true;
}
static_assert(cell_grid_fits<4>() && cell_grid_fits<5>() && cell_grid_fits<8>(),
              "a Lloyd-Max cell grid is too coarse for its table");

template <int BITS>
constexpr CellTable<CellGrid<BITS>::n> make_cell_table() {
  constexpr int n = CellGrid<BITS>::n;
  CellTable<n> t{};
  for (int c = 0; c < n; ++c) {
    t.e[c].b = std::numeric_limits<float>::infinity();
    t.e[c].base = 0;
  }
  for (int j = 0; j < (1 << BITS) - 1; ++j) t.e[grid_cell<BITS>(lm_boundary<BITS>(j))].b = lm_boundary<BITS>(j);
  int count = 0;
  for (int c = 0; c < n; ++c) {
    t.e[c].base = count;
    if (t.e[c].b != std::numeric_limits<float>::infinity()) ++count;
  }
  return t;
}

__device__ const CellTable<CellGrid<4>::n> kCells4 = make_cell_table<4>();
__device__ const CellTable<CellGrid<5>::n> kCells5 = make_cell_table<5>();
__device__ const CellTable<CellGrid<8>::n> kCells8 = make_cell_table<8>();

template <int BITS>
__device__ __forceinline__ const CellEntry* cell_table() {
  if constexpr (BITS == 4) return kCells4.e;
  else if constexpr (BITS == 5) return kCells5.e;
  else return kCells8.e;
}

template <int BITS>
__device__ __forceinline__ int lm_index_cells(float u, const CellEntry* tab) {
  using G = CellGrid<BITS>;
  float s = __fmul_rn(__fsub_rn(u, G::lo), G::scale);
  s = fminf(fmaxf(s, 0.0f), static_cast<float>(G::n - 1));  // NaN -> 0
  const CellEntry e = tab[static_cast<int>(s)];
  return e.base + (u > e.b ? 1 : 0);
}

template <int BITS>
__device__ __forceinline__ int lm_index_direct(float u) {
  int idx = 0;
#pragma unroll
  for (int j = 0; j < (1 << BITS) - 1; ++j) idx += (u > lm_boundary<BITS>(j)) ? 1 : 0;
  return idx;
}

template <int BITS>
__device__ __forceinline__ int lm_index(float u, const CellEntry* tab) {
  if constexpr (BITS <= 3) return lm_index_direct<BITS>(u);
  else return lm_index_cells<BITS>(u, tab);
}

template <int BITS>
__device__ __forceinline__ const float* centroid_table() {
  if constexpr (BITS == 2) return kCentroids2;
  else if constexpr (BITS == 3) return kCentroids3;
  else if constexpr (BITS == 4) return kCentroids4;
  else if constexpr (BITS == 5) return kCentroids5;
  else return kCentroids8;
}

// ---------------------------------------------------------------------------
// Bit packing (ops.ts, packBits / unpackBits): code i of a row occupies bits
// [i*b, i*b+b) of a little-endian bitstream, so the 8 codes of a chunk fill
// exactly b bytes starting at byte chunk*b.
template <int BITS>
__device__ __forceinline__ uint64_t pack8(const int (&q)[8]) {
  uint64_t acc = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) acc |= static_cast<uint64_t>(q[i] & ((1 << BITS) - 1)) << (i * BITS);
  return acc;
}

template <int BITS>
__device__ __forceinline__ void store_packed(uint8_t* p, uint64_t acc) {
  if constexpr (BITS == 8) {
    *reinterpret_cast<uint2*>(p) = make_uint2(static_cast<uint32_t>(acc), static_cast<uint32_t>(acc >> 32));
  } else if constexpr (BITS == 4) {
    *reinterpret_cast<uint32_t*>(p) = static_cast<uint32_t>(acc);
  } else if constexpr (BITS == 2) {
    *reinterpret_cast<uint16_t*>(p) = static_cast<uint16_t>(acc);
  } else {
#pragma unroll
    for (int i = 0; i < BITS; ++i) p[i] = static_cast<uint8_t>(acc >> (8 * i));
  }
}

template <int BITS>
__device__ __forceinline__ uint64_t load_packed(const uint8_t* p) {
  if constexpr (BITS == 8) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    return static_cast<uint64_t>(u.x) | (static_cast<uint64_t>(u.y) << 32);
  } else if constexpr (BITS == 4) {
    return __ldg(reinterpret_cast<const uint32_t*>(p));
  } else if constexpr (BITS == 2) {
    return __ldg(reinterpret_cast<const uint16_t*>(p));
  } else {
    uint64_t acc = 0;
#pragma unroll
    for (int i = 0; i < BITS; ++i) acc |= static_cast<uint64_t>(__ldg(p + i)) << (8 * i);
    return acc;
  }
}

template <int BITS>
__device__ __forceinline__ int unpack_code(uint64_t acc, int i) {
  return static_cast<int>((acc >> (i * BITS)) & ((1u << BITS) - 1));
}

}  // namespace tq
