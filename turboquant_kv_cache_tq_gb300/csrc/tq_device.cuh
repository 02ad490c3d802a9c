// Device building blocks of the TurboQuant codec kernels.
//
// Thread layout: lane l of a row owns quantisation group l, i.e. the 32
// consecutive head_dim elements [32l, 32l+32) of K and of V (one 64-byte
// load of bf16). A row uses D/32 lanes, so a warp holds 16, 8, 4 or 2 rows
// for D = 64, 128, 256, 512. Group reductions and the per-group scalars
// (scale, zero point, reciprocal) stay inside one lane.
//
// Pair layout: the 32 fp32 values of a group live in 16 float2 registers,
// pair p = (element p, element p + 16), so the packed Blackwell fp32x2
// instructions (add/mul/fma.rn.f32x2: two IEEE round-to-nearest operations
// per instruction) do the butterflies of strides 1..8, the squares and the
// scalings two elements at a time.
//
// Rounding contract: every floating-point step that feeds a stored result is
// one IEEE binary32 round-to-nearest-even operation in the order the codec
// page applies its ops (page "@mlx-bun/inference 0.0.0-stage -> 1.0.0", file
// package/src/kernels/turboquant/ops.ts); a - b is computed as fma(b, -1, a),
// which is the same single rounding. Reductions whose order the page leaves
// open use one fixed tree (group_sum_sq, the Hadamard stage order).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <limits>

#include "tq_internal.h"
#include "tq_tables.cuh"

namespace tq {

constexpr int kGroup = 32;     // BLOCK_SIZE on the ops.ts page
constexpr float kEps = 1e-8f;  // the page's eps as an fp32 scalar
constexpr unsigned kFull = 0xffffffffu;
// 1.5 * 2^23: for |t| < 2^22, RN(t + kMagic) = kMagic + rint(t) and the low
// 22 bits of its encoding hold rint(t) (two's complement around 0x4B400000).
constexpr float kMagic = 12582912.0f;

// RN(h + c) for the fp16 value h held in the low (HI = false) or high half of
// x: the mixed-precision add widens h exactly and rounds the sum once (an
// FMA-pipe instruction at full rate).
template <bool HI>
__device__ __forceinline__ float add_f16_f32(uint32_t x, float c) {
  float r;
  if constexpr (HI) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.f16 %0, hi, %2;\n\t}" : "=f"(r) : "r"(x), "f"(c));
  } else {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.f16 %0, lo, %2;\n\t}" : "=f"(r) : "r"(x), "f"(c));
  }
  return r;
}
constexpr uint32_t kMagicBits = 0x4B400000u;

template <int D>
struct Geo {
  static_assert(D == 64 || D == 128 || D == 256 || D == 512, "head_dim");
  static constexpr int LPR = D / kGroup;  // lanes per row = groups per row
  static constexpr int RPW = 32 / LPR;    // rows per warp
};

// Packed fp32x2 operations (PTX add/mul/fma.rn.f32x2), each component one IEEE
// round-to-nearest-even operation. The code generator may still fuse a packed
// multiply into a packed add that consumes it (measured on sm_103a even with
// explicit .rn modifiers), which would skip the product's rounding. So every
// product that feeds an add is formed as mul0(a, b, z) = fma(a, b, z) with z a
// runtime -0.0 from the kernel arguments: a*b + (-0) rounds to exactly
// RN(a*b) for every a, b (including signed zeros), and an fma result is never
// fused further.
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
// a - b as fma(b, -1, a): one rounding of the exact difference
__device__ __forceinline__ float2 sub2(float2 a, float2 b) { return fma2(b, f2(-1.0f), a); }
// RN(a * b) that cannot be fused into a consumer; nz must hold a runtime -0.0
__device__ __forceinline__ float2 mul0(float2 a, float2 b, float2 nz) { return fma2(a, b, nz); }

// A debug build's index check (TQ_CHECK): records a failure in the device
// error word and returns whether the access may go ahead.
__device__ __forceinline__ bool debug_check(bool ok, unsigned* err) {
  if (!ok && err != nullptr) atomicOr(err, kErrIndex);
  return ok;
}

// min / max that return NaN when either operand is NaN (PTX min.NaN / max.NaN).
__device__ __forceinline__ float fmin_nan(float a, float b) {
  float d;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ---------------------------------------------------------------------------
// Group loads. A group is 16 words of bf16 pairs (word j = elements 2j, 2j+1)
// or 32 fp32 values.
__device__ __forceinline__ void load_words16(const void* p, uint32_t (&w)[16]) {
  const uint4* q = static_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = __ldg(q + i);
    w[4 * i] = u.x; w[4 * i + 1] = u.y; w[4 * i + 2] = u.z; w[4 * i + 3] = u.w;
  }
}

__device__ __forceinline__ void load_floats32(const float* p, float (&x)[32]) {
  const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 u = __ldg(q + i);
    x[4 * i] = u.x; x[4 * i + 1] = u.y; x[4 * i + 2] = u.z; x[4 * i + 3] = u.w;
  }
}

// bf16 words -> pairs (element p, element p + 16)
__device__ __forceinline__ void words_to_pairs(const uint32_t (&w)[16], float2 (&P)[16]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    P[2 * j] = make_float2(bf16_lo(w[j]), bf16_lo(w[j + 8]));
    P[2 * j + 1] = make_float2(bf16_hi(w[j]), bf16_hi(w[j + 8]));
  }
}

__device__ __forceinline__ void floats_to_pairs(const float (&x)[32], float2 (&P)[16]) {
#pragma unroll
  for (int p = 0; p < 16; ++p) P[p] = make_float2(x[p], x[p + 16]);
}

// Element i of a pair array.
__device__ __forceinline__ float pair_elem(const float2 (&P)[16], int i) { return i < 16 ? P[i].x : P[i - 16].y; }

// Sign words: word j of a group has bit 15 set when element 2j has sign -1
// and bit 31 set when element 2j + 1 has; XOR into a bf16 pair word negates.
// A block keeps the D/2 words of its head_dim in shared memory.
template <int D>
__device__ __forceinline__ uint32_t sign_word(int l, int j) {
  const uint8_t* t;
  if constexpr (D == 64) t = kSignNeg64;
  else if constexpr (D == 128) t = kSignNeg128;
  else if constexpr (D == 256) t = kSignNeg256;
  else t = kSignNeg512;
  const int e = 32 * l + 2 * j;  // element index of the low half
  const uint32_t b = t[e >> 3];
  return (((b >> (e & 7)) & 1u) << 15) | (((b >> ((e & 7) + 1)) & 1u) << 31);
}

template <int D>
__device__ __forceinline__ void fill_sign_words(uint32_t* s_sign) {
  for (int i = threadIdx.x; i < D / 2; i += blockDim.x) s_sign[i] = sign_word<D>(i / 16, i % 16);
}

// The 16 sign words of group l.
__device__ __forceinline__ void load_sign_words(const uint32_t* s_sign, int l, uint32_t (&S)[16]) {
  const uint4* q = reinterpret_cast<const uint4*>(s_sign + 16 * l);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = q[i];
    S[4 * i] = u.x; S[4 * i + 1] = u.y; S[4 * i + 2] = u.z; S[4 * i + 3] = u.w;
  }
}

// Sign bit (bit 31) of element i of the group, from the sign words.
__device__ __forceinline__ uint32_t elem_sign(const uint32_t (&S)[16], int i) {
  return (i & 1) ? (S[i >> 1] & 0x80000000u) : ((S[i >> 1] << 16) & 0x80000000u);
}

// ---------------------------------------------------------------------------
// Rotation: H x (Sylvester order, unnormalised) on the D elements of a row
// held by its LPR lanes. Radix-2 stages in ascending stride: 1, 2, 4, 8 as
// packed ops across pairs, 16 inside each pair, then 32 .. D/2 across lanes
// (xor shuffles). Stage h maps (a, b) = (x[i], x[i+h]) to (a + b, a - b);
// across lanes the update is fma(x, s, partner), s = +1 in the lower lane
// and -1 in the upper one, i.e. exactly partner + x or partner - x.
template <int LPR>
__device__ __forceinline__ void hadamard_row(float2 (&P)[16], int l) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      if ((p & h) == 0) {
        const float2 a = P[p], b = P[p + h];
        P[p] = add2(a, b);
        P[p + h] = sub2(a, b);
      }
    }
  }
#pragma unroll
  for (int p = 0; p < 16; ++p) {
    const float a = P[p].x, b = P[p].y;
    P[p] = make_float2(__fadd_rn(a, b), __fsub_rn(a, b));
  }
#pragma unroll
  for (int m = 1; m < LPR; m <<= 1) {
    const float2 s = f2((l & m) ? -1.0f : 1.0f);
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      const float2 q = make_float2(__shfl_xor_sync(kFull, P[p].x, m), __shfl_xor_sync(kFull, P[p].y, m));
      P[p] = fma2(P[p], s, q);
    }
  }
}

// Sum of squares of a group as the pairwise tree over elements 0..31 in
// index order: (0,1),(2,3),... then pairs of those, up to (0..15)+(16..31).
__device__ __forceinline__ float group_sum_sq(const float2 (&P)[16], float2 nz) {
  float2 q[16];
#pragma unroll
  for (int p = 0; p < 16; ++p) q[p] = mul0(P[p], P[p], nz);
#pragma unroll
  for (int w = 1; w < 16; w <<= 1) {
#pragma unroll
    for (int p = 0; p < 16; p += 2 * w) q[p] = add2(q[p], q[p + w]);
  }
  return __fadd_rn(q[0].x, q[0].y);
}

// ---------------------------------------------------------------------------
// Lloyd-Max index = count(boundaries < u) (ops.ts, searchsorted), via a cell
// table. cell(u) = rint(u * S) + OFF with S a power of two, computed as the
// low bits of RN(u * S + (1.5 * 2^23 + OFF)) (u * S is exact, so this is one
// rounding on the device and in the compile-time builder alike). cell() is
// monotone, so a boundary in a lower cell than u is below u and one in a
// higher cell is not; each cell holds at most one boundary (the cell width
// 1/S is below the table's smallest boundary gap), compared explicitly: u > b
// exactly when RN(b - u) has its sign bit set. The grid covers |u| < 7.9; for
// finite inputs |u| <= sqrt(32) since u is a coordinate over its group's RMS.
struct __align__(8) CellEntry {  // one 64-bit shared-memory load
  float b;   // the boundary inside this cell, or +Inf
  int base;  // number of boundaries in lower cells
};

template <int BITS>
struct CellGrid;
template <> struct CellGrid<2> { static constexpr float S = 2.0f;  static constexpr int NC = 32, OFF = 16; };
template <> struct CellGrid<3> { static constexpr float S = 4.0f;  static constexpr int NC = 64, OFF = 32; };
template <> struct CellGrid<4> { static constexpr float S = 8.0f;  static constexpr int NC = 128, OFF = 64; };
template <> struct CellGrid<5> { static constexpr float S = 16.0f; static constexpr int NC = 256, OFF = 128; };
template <> struct CellGrid<8> { static constexpr float S = 64.0f; static constexpr int NC = 1024, OFF = 512; };

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

template <int BITS>
constexpr float grid_magic() {
  return kMagic + static_cast<float>(CellGrid<BITS>::OFF);
}

// The cell of u, with the device's arithmetic (one rounding of an exact
// product plus a constant); bounds are the caller's business.
template <int BITS>
constexpr int grid_cell_host(float u) {
  const float prod = u * CellGrid<BITS>::S;  // exact: S is a power of two
  const float s = prod + grid_magic<BITS>();  // one rounding
  return static_cast<int>(static_cast<long long>(s) - static_cast<long long>(kMagic));
}

template <int BITS>
constexpr bool cell_grid_fits() {
  int prev = -1;
  for (int j = 0; j < (1 << BITS) - 1; ++j) {
    const float b = lm_boundary<BITS>(j);
    if (b < -7.0f || b > 7.0f) return false;
    const int c = grid_cell_host<BITS>(b);
    if (c <= prev || c < 0 || c >= CellGrid<BITS>::NC) return false;
    prev = c;
  }
  return true;
}
static_assert(cell_grid_fits<2>() && cell_grid_fits<3>() && cell_grid_fits<4>() && cell_grid_fits<5>() &&
                  cell_grid_fits<8>(),
              "a Lloyd-Max cell grid is too coarse for its table");

template <int BITS>
constexpr CellTable<CellGrid<BITS>::NC> make_cell_table() {
  constexpr int n = CellGrid<BITS>::NC;
  CellTable<n> t{};
  for (int c = 0; c < n; ++c) {
    t.e[c].b = std::numeric_limits<float>::infinity();
    t.e[c].base = 0;
  }
  for (int j = 0; j < (1 << BITS) - 1; ++j) t.e[grid_cell_host<BITS>(lm_boundary<BITS>(j))].b = lm_boundary<BITS>(j);
  int count = 0;
  for (int c = 0; c < n; ++c) {
    t.e[c].base = count;
    if (t.e[c].b != std::numeric_limits<float>::infinity()) ++count;
  }
  return t;
}

__device__ const CellTable<CellGrid<2>::NC> kCells2 = make_cell_table<2>();
__device__ const CellTable<CellGrid<3>::NC> kCells3 = make_cell_table<3>();
__device__ const CellTable<CellGrid<4>::NC> kCells4 = make_cell_table<4>();
__device__ const CellTable<CellGrid<5>::NC> kCells5 = make_cell_table<5>();
__device__ const CellTable<CellGrid<8>::NC> kCells8 = make_cell_table<8>();

template <int BITS>
__device__ __forceinline__ const CellEntry* cell_table() {
  if constexpr (BITS == 2) return kCells2.e;
  else if constexpr (BITS == 3) return kCells3.e;
  else if constexpr (BITS == 4) return kCells4.e;
  else if constexpr (BITS == 5) return kCells5.e;
  else return kCells8.e;
}

// Indices of a pair of values (finite, |u| < 7.9) from the table in shared
// memory; u must not be an unfused product (see mul0).
template <int BITS>
__device__ __forceinline__ void lm_index2(float2 u, const CellEntry* tab, int& i0, int& i1) {
  using G = CellGrid<BITS>;
  const float2 s = fma2(u, f2(G::S), f2(grid_magic<BITS>()));
  const CellEntry e0 = tab[__float_as_uint(s.x) & (G::NC - 1)];
  const CellEntry e1 = tab[__float_as_uint(s.y) & (G::NC - 1)];
  const float2 d = sub2(make_float2(e0.b, e1.b), u);  // RN(b - u) < 0 exactly when u > b
  i0 = e0.base + static_cast<int>(__float_as_uint(d.x) >> 31);
  i1 = e1.base + static_cast<int>(__float_as_uint(d.y) >> 31);
}

// Indices of the pair y * inv without rounding the product first: the cell
// is RN(y * (inv * S) + magic) (inv * S is exact) and the comparison is the
// sign of RN(b - y * inv) (one fma), so both use the same exact value
// v = y * inv and the result is exactly count(boundaries < v).
// MASKED = false indexes the table by the float's bits minus the magic
// constant's, without a mask: the caller guarantees |v| * S < OFF, which
// holds whenever inv is the reciprocal of (a finite group RMS + eps) and y is
// an element of that group (|y| <= sqrt(32) * rms, so |v * S| <= 5.66 S).
// MASKED = true is safe for any input: NaN and Inf land in some cell, and a
// value v that is NaN (a group whose RMS is Inf or NaN: an Inf or NaN in the
// row) gets index 0, since searchsorted counts no boundary below NaN.
template <int BITS, bool MASKED>
__device__ __forceinline__ void lm_index2_scaled(float2 y, float inv, const CellEntry* tab, uint32_t& i0,
                                                 uint32_t& i1) {
  using G = CellGrid<BITS>;
  const float2 s = fma2(y, f2(__fmul_rn(inv, G::S)), f2(grid_magic<BITS>()));
  uint32_t c0 = __float_as_uint(s.x), c1 = __float_as_uint(s.y);
  if constexpr (MASKED) {
    c0 &= G::NC - 1;
    c1 &= G::NC - 1;
  } else {
    c0 -= kMagicBits;
    c1 -= kMagicBits;
  }
  const CellEntry e0 = tab[c0];
  const CellEntry e1 = tab[c1];
  const float2 d = fma2(y, f2(-inv), make_float2(e0.b, e1.b));
  i0 = static_cast<uint32_t>(e0.base) + (__float_as_uint(d.x) >> 31);
  i1 = static_cast<uint32_t>(e1.base) + (__float_as_uint(d.y) >> 31);
  if constexpr (MASKED) {
    // s is NaN exactly when v = y * inv is (|v| <= sqrt(32) otherwise)
    i0 = (s.x != s.x) ? 0u : i0;
    i1 = (s.y != s.y) ? 0u : i1;
  }
}

// Any fp32 value: clamp into the grid first (all boundaries lie inside it, so
// the count is unchanged; NaN clamps to the low end and counts nothing).
template <int BITS>
__device__ __forceinline__ int lm_index_any(float u, const CellEntry* tab) {
  const float c = fminf(fmaxf(u, -7.5f), 7.5f);
  int i0, i1;
  lm_index2<BITS>(make_float2(c, c), tab, i0, i1);
  return i0;
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
// [i*b, i*b+b) of a little-endian bitstream, so the 32 codes of group l fill
// exactly b 32-bit words starting at byte 4*b*l of the packed row.
// Put code i (its low B bits) into its place in the packed words. The words
// start at zero and every code owns its own bits, so the shifted code can be
// added (one shift-add instruction) instead of masked and or-ed in.
template <int B>
__device__ __forceinline__ void put_code(uint32_t (&w)[B], int i, uint32_t c) {
  const uint32_t v = c & ((1u << B) - 1u);
  const int bit = i * B, word = bit >> 5, off = bit & 31;
  w[word] += v << off;
  if (off + B > 32) w[word + 1] += v >> (32 - off);
}

// The same for a code already known to fit in B bits (no mask).
template <int B>
__device__ __forceinline__ void put_code_exact(uint32_t (&w)[B], int i, uint32_t v) {
  const int bit = i * B, word = bit >> 5, off = bit & 31;
  w[word] += v << off;
  if (off + B > 32) w[word + 1] += v >> (32 - off);
}

// Sum of (kMagicBits << offset) over the codes whose low part lies in word
// `word`, modulo 2^32.
template <int B>
__host__ __device__ constexpr uint32_t magic_correction(int word) {
  uint32_t c = 0;
  for (int i = 0; i < 32; ++i) {
    const int bit = i * B;
    if ((bit >> 5) == word) c += kMagicBits << (bit & 31);
  }
  return c;
}

// Low bytes of four words, in order, as one word.
__device__ __forceinline__ uint32_t gather_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Pack the 32 codes of a group, produced pair by pair: code_pair(q, lo, hi)
// yields the codes of elements q and q + 16 (the pair layout). Code i goes
// to bits [i*B, i*B+B) of w.
//   MAGIC = false: codes are plain values in [0, 2^B).
//   MAGIC = true: codes are float bit patterns kMagicBits + code (the output
//     of rounding by the magic constant), code in [0, 2^B), or in
//     [-127, 127] for B = 8. Narrow codes are accumulated shifted, pattern
//     and all, and the magic constant's share of each word is subtracted once
//     at the end (exact modulo 2^32); the part of a code that spills into the
//     next word is its true value shifted down.
// B = 8 takes the low byte of each code (two's complement when negative),
// four codes per word with byte permutes.
template <int B, bool MAGIC, typename CodePair>
__device__ __forceinline__ void pack_pairs(uint32_t (&w)[B], CodePair&& code_pair) {
  if constexpr (B == 8) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t lo[4], hi[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) code_pair(4 * j + r, lo[r], hi[r]);
      w[j] = gather_low_bytes(lo[0], lo[1], lo[2], lo[3]);
      w[j + 4] = gather_low_bytes(hi[0], hi[1], hi[2], hi[3]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < B; ++k) w[k] = 0;
    auto put = [&](int i, uint32_t c) {
      const int bit = i * B, word = bit >> 5, off = bit & 31;
      w[word] += c << off;
      if (off + B > 32) w[word + 1] += (MAGIC ? c - kMagicBits : c) >> (32 - off);
    };
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      uint32_t lo, hi;
      code_pair(q, lo, hi);
      put(q, lo);
      put(q + 16, hi);
    }
    if constexpr (MAGIC) {
#pragma unroll
      for (int k = 0; k < B; ++k) w[k] -= magic_correction<B>(k);
    }
  }
}

template <int B>
__device__ __forceinline__ uint32_t unpack_code(const uint32_t (&w)[B], int i) {
  const int bit = i * B, word = bit >> 5, off = bit & 31;
  uint32_t v = w[word] >> off;
  if (off + B > 32) v |= w[word + 1] << (32 - off);
  return v & ((1u << B) - 1u);
}

template <int B>
__device__ __forceinline__ void store_words(uint8_t* p, const uint32_t (&w)[B]) {
  if constexpr (B == 8) {
    reinterpret_cast<uint4*>(p)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(p)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  } else if constexpr (B == 4) {
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  } else if constexpr (B == 2) {
    *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
  } else {
#pragma unroll
    for (int k = 0; k < B; ++k) reinterpret_cast<uint32_t*>(p)[k] = w[k];
  }
}

template <int B>
__device__ __forceinline__ void load_words(const uint8_t* p, uint32_t (&w)[B]) {
  if constexpr (B == 8) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  } else if constexpr (B == 4) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  } else if constexpr (B == 2) {
    const uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
    w[0] = a.x; w[1] = a.y;
  } else {
#pragma unroll
    for (int k = 0; k < B; ++k) w[k] = __ldg(reinterpret_cast<const uint32_t*>(p) + k);
  }
}

// ---------------------------------------------------------------------------
// Row -> (b*h, t) by a multiply-shift: for 0 <= r < 2^31 and 1 <= T < 2^31,
// with s = ceil(log2 T) and m = ceil(2^(32+s) / T), floor(r * m / 2^(32+s))
// equals floor(r / T) (the error term r * (m*T - 2^(32+s)) / (T * 2^(32+s))
// stays below 1/(2T)).
__host__ inline FastDiv make_fast_div(int T) {
  int s = 0;
  while ((1LL << s) < T) ++s;
  const unsigned __int128 num = static_cast<unsigned __int128>(1) << (32 + s);
  const unsigned long long m = static_cast<unsigned long long>((num + T - 1) / T);
  return FastDiv{m, 32 + s};
}

__device__ __forceinline__ int fast_div(int r, FastDiv d) {
  return static_cast<int>((static_cast<unsigned long long>(r) * d.m) >> d.shift);
}

}  // namespace tq
