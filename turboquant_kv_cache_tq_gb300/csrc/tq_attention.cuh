// Fused decode attention over a packed TurboQuant KV cache.
//
// What it computes (page "@mlx-bun/inference 0.0.0-stage -> 1.0.0"): the
// deferV branch of tryDecodePackedKv in ops.ts decodes the keys with
// decodeKeys and the values with decodeValuesRotated, both returned as bf16;
// attention runs over those rows; unrotateValues then undoes the value
// rotation once on the attention output (attention is linear in V, the
// decodeValuesRotated comment). The key-validity mask of batched decode with
// left-padded rows comes from batched-mask.ts. Here the decoded rows never
// reach memory: each tile of the packed cache is decoded in registers
// straight into tensor-core operands.
//
//   o[q] = unrotate( sum_t softmax_t(scale * q . K[t]) V_rot[t] )
//   K[t]     = bf16(RN(RN(code + zero) * scale_k))    (decodeKeys, bf16 out)
//   V_rot[t] = bf16(RN(centroid[idx] * scale_v))      (decodeValuesRotated)
// over the valid keys t of query row q: left_pad[b] <= t <= T - Nq + n.
//
// Split kernel: the flattened (batch, kv head, 16-token tile) space is cut
// evenly over one wave of blocks of four warps (eight where the value table
// is 32 KB); a block's share is cut into per-head segments. A warp streams
// 16-token tiles of the five packed buffers through its own two-stage ring of
// shared memory (cp.async, 16-byte pieces) and, per tile:
//   scores  S^T = K Q^T on the tensor cores (mma.sync m16n8k16, bf16 in,
//           fp32 accumulate): M = the tile's 16 tokens, N = 8 query rows
//           (the Hq/Hkv heads of the group times Nq tokens) per row tile,
//           K = 16 head_dim elements. The head_dim order inside the
//           contraction is permuted so that the four lanes sharing a token
//           each own a quarter of the row (D/4 consecutive elements: one
//           quantisation group at D = 128), so a lane decodes its own
//           contiguous codes with its own group scale and zero point, and the
//           bf16 products are exact; the queries stay in registers;
//   softmax online in fp32 (exp2 of scores pre-scaled by log2 e), per query
//           row;
//   values  O^T += V^T P^T, M = 16 head_dim elements, N = 8 query rows,
//           K = 16 tokens. P comes straight from the score accumulators
//           (transposed 8x8 by movmatrix), split as P = P_hi + P_lo in bf16
//           (two MMAs), which keeps the weights exact to about 2^-18; the
//           values are exact in bf16.
// Above D = 128 two warps share each tile, one per half of head_dim (see
// AttnSplit). At the end of a segment the warps' partial (max, sum, O) are
// merged in shared memory and the block writes one partial record to the
// workspace.
//
// Combine kernel: merges each output row's records (in chunks over several
// blocks when a head has many, the last block to finish adding the chunks'
// results), divides by the softmax denominator and applies the inverse
// rotation in fp32 (the Hadamard butterflies of the codec, * 1/sqrt(D), then
// the signs: unrotateValues), storing fp32 or bf16.
#pragma once

#include "tq_kernels.cuh"

namespace tq {

#ifndef TQ_ATTN_STAGES
// ring stages of a four-warp block at <= 128 elements per warp (two measured
// faster than three: long-context v3 attention 119.4 -> 117.7 us)
#define TQ_ATTN_STAGES 2
#endif
#ifndef TQ_ATTN_MIN_TEAM_TILES
// fewest tiles per team of warps when heads are few and long (4: [4, 4, 8192,
// 256] v4 30.5 -> 28.1 us against 8 since the chunked combine; 2 the same as
// 4; 12 slower, 39.6 us)
#define TQ_ATTN_MIN_TEAM_TILES 4
#endif
constexpr long long kAttnMinTeamTiles = TQ_ATTN_MIN_TEAM_TILES;
constexpr int kAttnTile = 16;  // tokens per warp step
constexpr int kAttnRows = kAttnMaxRows;  // query rows per kv head (M of the score MMA)

__host__ __device__ constexpr int attn_round_up(int x, int m) { return (x + m - 1) / m * m; }

// Per-warp layout over D head_dim elements of a row whose scales and zero
// points (SNG groups: the whole row's) are staged whole.
template <int D, int KB, int VB, int SNG = D / kGroup>
struct AttnLayout {
  static constexpr int NG = D / kGroup;
  static constexpr int PDK = D * KB / 8;
  static constexpr int PDV = D * VB / 8;
  // one stage: the tile's rows of the five packed buffers, back to back
  static constexpr int KC = 0;                         // K codes  [16][PDK]
  static constexpr int KS = KC + kAttnTile * PDK;      // K scales [16][SNG] fp16
  static constexpr int KZ = KS + kAttnTile * SNG * 2;  // K zeros
  static constexpr int VC = KZ + kAttnTile * SNG * 2;  // V codes  [16][PDV]
  static constexpr int VS = VC + kAttnTile * PDV;      // V scales
  static constexpr int END = VS + kAttnTile * SNG * 2;
  static constexpr int STAGE = attn_round_up(END + 16, 128);  // + room for word over-reads
  // value lookup table (see ValueTable): pairs of centroids for widths up to
  // 4 bits, once per half-warp lane; single centroids once per lane above
  static constexpr int CENT = VB <= 4 ? (16 * 8) << (2 * VB) : (32 * 4) << VB;
  // per-lane element ranges
  static constexpr int EK = D / 4;  // keys: token g, elements [c EK, (c+1) EK)
  static constexpr int EV = D / 8;  // values: elements [g EV, (g+1) EV) of four tokens
  static constexpr int NWK = (EK * KB + 31) / 32;
  static constexpr int NWV = (EV * VB + 31) / 32;
  static constexpr bool KALIGN = (EK * KB / 8) % 4 == 0;  // byte offset of a lane's key codes
  static constexpr bool VALIGN = (EV * VB / 8) % 4 == 0;
  static constexpr int KGROUPS = EK > kGroup ? EK / kGroup : 1;  // groups a lane's key range spans
};

// Head_dim split: above D = 128 a warp holding a whole row's query operands
// and output accumulators needs 168 (D = 256) to 255 (D = 512) registers,
// which leaves 8 to 12 warps per SM, so SPL = 2 warps share each token tile,
// one per half of head_dim: each decodes its slice of the keys and values,
// their partial scores are added through shared memory (all add the same
// SPL terms in the same order, so all get the same scores and the same
// softmax), and each keeps the output accumulators of its slice. (Four
// 128-element slices at D = 512 measured slower: 37 -> 45 us on
// [2, 2, 16384, 512], the four-way exchange every tile.)
template <int D>
struct AttnSplit {
  static constexpr int SPL = D > 128 ? 2 : 1;
  static constexpr int DH = D / SPL;
};

// Warps per block (NW) and ring stages per warp (S). A block's warps share
// its value table; the 32 KB tables (4-bit pairs, 8-bit singles) would hold
// a four-warp block of head_dim <= 128 to two or three blocks per SM (8 or 12
// warps), so those blocks take eight warps with two stages each: two blocks,
// 16 warps per SM, the register limit at 128 registers a thread.
template <int D, int VB, int NT>
struct AttnShape {
  static constexpr int DH = AttnSplit<D>::DH;
  static constexpr int CENT = VB <= 4 ? (16 * 8) << (2 * VB) : (32 * 4) << VB;
  static constexpr bool WIDE = DH <= 128 && CENT >= 32768 && NT == 1;
  static constexpr int NW = WIDE ? 8 : 4;
  static constexpr int THREADS = 32 * NW;
  static constexpr int S = (WIDE || DH >= 256) ? 2 : TQ_ATTN_STAGES;
  // 128 registers a thread for one query-row tile (NT = 1) over 128-element
  // slices; wider slices or two tiles (NT = 2) need more and keep the
  // compiler's choice (0: no bound)
  static constexpr int MIN_BLOCKS = WIDE ? 2 : (NT == 1 && DH <= 128 ? 4 : 0);
};

// Block-level shared memory of the split kernel over the per-warp layout L:
// value table | score exchange (SPL > 1) | ring of stages, later the merge
// area of one record per warp group.
template <int D, int KB, int VB, int NT>
struct AttnSmem {
  using L = AttnLayout<AttnSplit<D>::DH, KB, VB, D / kGroup>;
  using Shape = AttnShape<D, VB, NT>;
  static_assert(Shape::CENT == L::CENT, "one table size");
  static constexpr int NW = Shape::NW;
  static constexpr int S = Shape::S;
  static constexpr int RING = NW * S * L::STAGE;
  static constexpr int SPL = AttnSplit<D>::SPL;
  static constexpr int REC = kAttnRows * (D + 2);  // floats of a partial record: m[16], l[16], O[16][D]
  static_assert(REC == kAttnRecordFloats(D), "record layout shared with the host");
  static constexpr int MERGE = (NW / SPL) * REC * 4;
  // two slots (tile parity) x warps x 32 lanes x NT x 4 partial scores
  static constexpr int XCHG = SPL > 1 ? 2 * NW * 32 * NT * 4 * 4 : 0;
  static constexpr int XOFF = L::CENT;
  static constexpr int WORK = XOFF + XCHG;
  static constexpr int SMEM = WORK + (RING > MERGE ? RING : MERGE);
};

// Copy ROWS rows of HB bytes (a multiple of 16) taken at a stride of FB bytes
// from global memory into ROWS x HB contiguous bytes of shared memory, with the
// warp's 16-byte asynchronous copies.
template <int ROWS, int HB, int FB>
__device__ __forceinline__ void copy_rows(uint32_t dst, const void* src, int lane) {
  static_assert(HB % 16 == 0 && FB % 16 == 0, "16-byte pieces");
  constexpr int PR = HB / 16;
  const char* s = static_cast<const char*>(src);
#pragma unroll
  for (int i = lane; i < ROWS * PR; i += 32) cp_async16(dst + 16 * i, s + (i / PR) * FB + 16 * (i % PR));
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// NW little-endian words from byte `off` of shared memory (any byte offset
// when !ALIGNED; reads up to 4 bytes past the last word).
template <int NW, bool ALIGNED>
__device__ __forceinline__ void lds_words(const uint8_t* base, int off, uint32_t (&w)[NW]) {
  if constexpr (ALIGNED) {
    const uint32_t* q = reinterpret_cast<const uint32_t*>(base + off);
#pragma unroll
    for (int k = 0; k < NW; ++k) w[k] = q[k];
  } else {
    const uint32_t* q = reinterpret_cast<const uint32_t*>(base + (off & ~3));
    const int sh = (off & 3) * 8;
    uint32_t r[NW + 1];
#pragma unroll
    for (int k = 0; k <= NW; ++k) r[k] = q[k];
#pragma unroll
    for (int k = 0; k < NW; ++k) w[k] = __funnelshift_r(r[k], r[k + 1], sh);
  }
}

// Code e (bits [e B, e B + B)) of a little-endian bitstream held in words.
template <int B, int NW>
__device__ __forceinline__ uint32_t code_at(const uint32_t (&w)[NW], int e) {
  const int bit = e * B, word = bit >> 5, off = bit & 31;
  uint32_t v = w[word] >> off;
  if (off + B > 32) v |= w[word + 1] << (32 - off);
  return v & ((1u << B) - 1u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Copy `bytes` (a multiple of 16, compile-time) from global to shared memory
// with the warp's 16-byte asynchronous copies.
template <int BYTES>
__device__ __forceinline__ void copy_region(uint32_t dst, const void* src, int lane) {
  static_assert(BYTES % 16 == 0, "16-byte pieces");
  const char* s = static_cast<const char*>(src);
#pragma unroll
  for (int i = lane; i < BYTES / 16; i += 32) cp_async16(dst + 16 * i, s + 16 * i);
}

// Centroid lookups of the value decode, free of shared-memory bank
// conflicts. Widths up to 4 bits use a pair table: entry j =
// (centroid[j & m], centroid[j >> VB]), so the 2 VB-bit field of two
// consecutive codes (the packing is a little-endian bitstream) fetches both
// centroids with one 64-bit load; the table is kept once per half-warp lane
// (entry j for lane L at float2 16 j + L % 16), so the 16 lanes of a
// half-warp always read 16 distinct bank pairs. Wider codes use the single
// table kept once per lane (entry j for lane L at word 32 j + L).
template <int VB>
struct ValueTable {
  static constexpr bool PAIRS = VB <= 4;
};

template <int VB>
__device__ __forceinline__ void fill_value_table(uint8_t* s) {
  constexpr int m = (1 << VB) - 1;
  if constexpr (ValueTable<VB>::PAIRS) {
    float2* t = reinterpret_cast<float2*>(s);
    for (int i = threadIdx.x; i < (16 << (2 * VB)); i += blockDim.x) {
      const int j = i >> 4;
      t[i] = make_float2(centroid_table<VB>()[j & m], centroid_table<VB>()[j >> VB]);
    }
  } else {
    float* t = reinterpret_cast<float*>(s);
    for (int i = threadIdx.x; i < (32 << VB); i += blockDim.x) t[i] = centroid_table<VB>()[i >> 5];
  }
}

// (field << SH) | lane_off for the W-bit field at bit `bit` (compile-time)
// of a little-endian bitstream held in words (one shift and one three-input
// logic op); lane_off's bits lie below SH or above the field's.
template <int W, int SH, int NW>
__device__ __forceinline__ uint32_t field_addr(const uint32_t (&w)[NW], int bit, uint32_t lane_off) {
  const int word = bit >> 5, off = bit & 31;
  constexpr uint32_t kMask = ((1u << W) - 1u) << SH;
  uint32_t x;
  if (off + W > 32) x = __funnelshift_r(w[word], w[word + 1], off) << SH;
  else if (off >= SH) x = w[word] >> (off - SH);
  else x = w[word] << (SH - off);
  return (x & kMask) | lane_off;
}

// The same address for a byte-aligned 8-bit field (byte k, compile-time): a
// byte permute and a multiply-add by the table's entry stride, a runtime
// value so the multiply stays on the FMA pipe (a shift and a mask would both
// take the ALU pipe, the busiest of this kernel).
template <int NW>
__device__ __forceinline__ uint32_t byte_field_addr(const uint32_t (&w)[NW], int k, uint32_t stride,
                                                    uint32_t lane_off) {
  return __byte_perm(w[k >> 2], 0u, 0x4440u | static_cast<uint32_t>(k & 3)) * stride + lane_off;
}

__device__ __forceinline__ float fast_exp2(float x) {
  // ex2.approx: relative error below 2^-22; results below 2^-126 flush to
  // zero, which only drops weights under 2^-126 of the row's largest one
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Transpose of an 8x8 bf16 matrix held as one register per lane (row
// lane / 4, columns 2 (lane % 4) and 2 (lane % 4) + 1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

template <int D, int VB, int KMODE, int NT>
__global__ void __launch_bounds__(AttnShape<D, VB, NT>::THREADS, AttnShape<D, VB, NT>::MIN_BLOCKS)
    attn_split_kernel(AttnParams p) {
  using M = KeySpec<KMODE>;
  constexpr int KB = M::B;
  using SM = AttnSmem<D, KB, VB, NT>;
  using L = typename SM::L;  // the per-warp layout over DH head_dim elements
  constexpr int SPL = SM::SPL;
  constexpr int DH = AttnSplit<D>::DH;
  constexpr int PDK_FULL = D * KB / 8, PDV_FULL = D * VB / 8, NG_FULL = D / kGroup;
  using VT = ValueTable<VB>;
  constexpr int S = SM::S;
  constexpr int NW = SM::NW;
  const float kNegInf = -__int_as_float(0x7f800000);
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* s_vtab = smem;
  float* s_xchg = reinterpret_cast<float*>(smem + SM::XOFF);
  uint8_t* s_work = smem + SM::WORK;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int Rq = p.G * p.Nq;
  const int team = warp / SPL;           // warps sharing a tile
  const int half = warp % SPL;           // the head_dim slice of this warp
  constexpr int kTeams = NW / SPL;

  fill_value_table<VB>(s_vtab);
  pdl_launch_dependents();
  pdl_wait();
  // the combine's tickets start at zero (it runs after this grid completes)
  if (p.chunks > 1 && blockIdx.x == 0 &&
      TQ_CHECK(static_cast<long long>(p.combine_tiles) * p.chunks * kCombinePartialFloats <= p.partial_floats, p.err))
    for (int i = threadIdx.x; i < p.combine_tiles; i += blockDim.x) p.counters[i] = 0u;

  // This block's share of the flattened (batch, kv head, tile) space, cut
  // into one segment per (batch, kv head) it touches; each segment ends in
  // one partial record at slot blockIdx.x + bh (unique: the heads of
  // consecutive blocks never go back).
  const long long seg_lo = static_cast<long long>(blockIdx.x) * p.total_tiles / gridDim.x;
  const long long seg_hi = static_cast<long long>(blockIdx.x + 1) * p.total_tiles / gridDim.x;
  for (long long s0 = seg_lo; s0 < seg_hi;) {
    const int bh = static_cast<int>(s0 / p.tiles_per_bh);
    const long long s1 = min(seg_hi, static_cast<long long>(bh + 1) * p.tiles_per_bh);
    const int tile_lo = static_cast<int>(s0 - static_cast<long long>(bh) * p.tiles_per_bh);
    const int tile_hi = static_cast<int>(s1 - static_cast<long long>(bh) * p.tiles_per_bh);
    s0 = s1;
    const int b = bh / p.Hkv, h = bh - b * p.Hkv;
    __syncthreads();  // the previous segment's merge area is free again

    // Query operands of the score MMAs, kept in registers: query row 8 n + g
    // (heads h G .. h G + G - 1, Nq tokens each: Rq contiguous rows of q),
    // head_dim elements c D/4 + 4 j .. + 3 for k-step j (the contraction's
    // permuted order: MMA k index kk of k-step j is element
    // (kk % 8 / 2) D/4 + 4 j + 2 (kk / 8) + kk % 2). Padding rows are zero.
    uint32_t qf[DH / 16][NT][2];
    {
      const uint16_t* qsrc = p.q + (static_cast<long long>(b) * p.Hq + static_cast<long long>(h) * p.G) * p.Nq * D +
                             half * DH;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int row = 8 * n + g;
#pragma unroll
        for (int j = 0; j < DH / 16; ++j) {
          uint2 u = make_uint2(0u, 0u);
          if (row < Rq) u = *reinterpret_cast<const uint2*>(qsrc + row * D + c * L::EK + 4 * j);
          qf[j][n][0] = u.x;
          qf[j][n][1] = u.y;
        }
      }
    }
    const int t_lo = p.left_pad != nullptr ? max(p.left_pad[b], 0) : 0;
    int t_beg = tile_lo * kAttnTile;
    const int t_end = min(tile_hi * kAttnTile, p.T);
    t_beg = max(t_beg, t_lo & ~(kAttnTile - 1));
    const int n_tiles = t_end > t_beg ? (t_end - t_beg + kAttnTile - 1) / kAttnTile : 0;
    // last key of the lane's query columns 8 n + 2 c + x; -1 for padding rows
    int hiq[NT][2];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int q = 8 * n + 2 * c + x;
        hiq[n][x] = q < Rq ? p.T - p.Nq + q % p.Nq : -1;
      }
    const int t_full = p.T - p.Nq;  // keys up to here are valid for every real row

    uint8_t* ring = s_work + warp * S * L::STAGE;
    const uint32_t ring_sh = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
    const long long tok0 = static_cast<long long>(bh) * p.t_cap + t_beg;
    const int my_tiles = n_tiles > team ? (n_tiles - team + kTeams - 1) / kTeams : 0;
    // Step k of this warp handles tile team + kTeams k in stage k mod S (its
    // slice of each row when SPL > 1); every step commits one copy group
    // (empty past the end).
    auto issue = [&](int k) {
      const long long tk = tok0 + static_cast<long long>(team + k * kTeams) * kAttnTile;
      if (k < my_tiles && TQ_CHECK(tk >= 0 && tk + kAttnTile <= static_cast<long long>(bh + 1) * p.t_cap, p.err)) {
        const long long t = tk;
        const uint32_t dst = ring_sh + (k % S) * L::STAGE;
        if constexpr (SPL == 1) {
          copy_region<kAttnTile * L::PDK>(dst + L::KC, p.k_codes + t * L::PDK, lane);
          copy_region<kAttnTile * L::NG * 2>(dst + L::KS, p.k_scales + t * L::NG, lane);
          copy_region<kAttnTile * L::NG * 2>(dst + L::KZ, p.k_zeros + t * L::NG, lane);
          copy_region<kAttnTile * L::PDV>(dst + L::VC, p.v_codes + t * L::PDV, lane);
          copy_region<kAttnTile * L::NG * 2>(dst + L::VS, p.v_scales + t * L::NG, lane);
        } else {
          copy_rows<kAttnTile, L::PDK, PDK_FULL>(dst + L::KC, p.k_codes + t * PDK_FULL + half * L::PDK, lane);
          copy_region<kAttnTile * NG_FULL * 2>(dst + L::KS, p.k_scales + t * NG_FULL, lane);
          copy_region<kAttnTile * NG_FULL * 2>(dst + L::KZ, p.k_zeros + t * NG_FULL, lane);
          copy_rows<kAttnTile, L::PDV, PDV_FULL>(dst + L::VC, p.v_codes + t * PDV_FULL + half * L::PDV, lane);
          copy_region<kAttnTile * NG_FULL * 2>(dst + L::VS, p.v_scales + t * NG_FULL, lane);
        }
      }
      cp_async_commit();
    };

    float acc[DH / 16][NT][4];
#pragma unroll
    for (int i = 0; i < DH / 16; ++i)
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][n][e] = 0.0f;
    float m_run[NT][2], l_run[NT][2];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        m_run[n][x] = kNegInf;
        l_run[n][x] = 0.0f;
      }
    const uint32_t vlane = VT::PAIRS ? 8u * (lane & 15) : 4u * lane;  // the lane's table replica
    const uint32_t vstride = p.vtab_stride;
    constexpr float kBias = kMagic + (M::SIGNED ? 128.0f : 0.0f);
    constexpr float kBias16 = 1024.0f + (M::SIGNED ? 128.0f : 0.0f);

#pragma unroll
    for (int k = 0; k < S - 1; ++k) issue(k);
    for (int k = 0; k < my_tiles; ++k) {
      __syncwarp();
      issue(k + S - 1);
      cp_async_wait<S - 1>();
      __syncwarp();
      const uint8_t* st = ring + (k % S) * L::STAGE;
      const int t0 = t_beg + (team + k * kTeams) * kAttnTile;
      // a tile inside [t_lo, T - Nq] needs no mask (warp-uniform)
      const bool full = t0 >= t_lo && t0 + kAttnTile - 1 <= t_full;

      // ---- keys: tokens g and g + 8, elements [c EK, (c+1) EK)
      uint32_t wk[2][L::NWK];
      float2 ks2[2][L::KGROUPS], kzb2[2][L::KGROUPS];
      float kzh[2][L::KGROUPS];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int tau = g + 8 * hf;
        lds_words<L::NWK, L::KALIGN>(st + L::KC + tau * L::PDK, c * (L::EK * KB / 8), wk[hf]);
        if constexpr (M::SIGNED) {
#pragma unroll
          for (int w = 0; w < L::NWK; ++w) wk[hf][w] ^= 0x80808080u;  // code + 128 in each byte
        }
#pragma unroll
        for (int lg = 0; lg < L::KGROUPS; ++lg) {
          const int grp = (c * L::EK) / kGroup + lg;
          const uint16_t* sc = reinterpret_cast<const uint16_t*>(st + L::KS);
          const uint16_t* zr = reinterpret_cast<const uint16_t*>(st + L::KZ);
          ks2[hf][lg] = f2(__half2float(__ushort_as_half(sc[tau * NG_FULL + half * L::NG + grp])));
          const float zp = __half2float(__ushort_as_half(zr[tau * NG_FULL + half * L::NG + grp]));
          kzb2[hf][lg] = f2(__fsub_rn(zp, kBias));
          kzh[hf][lg] = __fsub_rn(zp, kBias16);
        }
      }
      // scores S^T = K Q^T: M = the tile's 16 tokens, N = 8 query rows per tile
      // n, K = 16 head_dim elements per k-step; two accumulator chains
      float sacc[NT][2][4];
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[n][ch][e] = 0.0f;
#pragma unroll
      for (int j = 0; j < DH / 16; ++j) {
        const int lg = (4 * j) / kGroup;
        uint32_t af[2][2];  // [token g / g + 8][elements 0-1 / 2-3]
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          // RN(code + zero) for four codes (+ 128 for signed codes, whose
          // bytes are offset by flipping their sign bits). 8-bit codes: one
          // byte permute makes two fp16 values 1024 + byte, and one
          // mixed-precision add each widens one and adds zero - 1024 -
          // offset (exact: the zero point is an integer) in one rounding, on
          // the FMA pipe; narrower codes: the floats 1.5 * 2^23 + code plus
          // zero - 1.5 * 2^23 - offset. Then one rounding of the product
          // with the scale (decodeKeys), then bf16.
          float2 f01, f23;
          if constexpr (KB == 8) {
            const uint32_t w = wk[hf][j];
            const uint32_t h01 = __byte_perm(w, 0x64646464u, 0x4140);
            const uint32_t h23 = __byte_perm(w, 0x64646464u, 0x4342);
            f01 = make_float2(add_f16_f32<false>(h01, kzh[hf][lg]), add_f16_f32<true>(h01, kzh[hf][lg]));
            f23 = make_float2(add_f16_f32<false>(h23, kzh[hf][lg]), add_f16_f32<true>(h23, kzh[hf][lg]));
          } else {
            uint32_t u[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) u[e] = kMagicBits | code_at<KB>(wk[hf], 4 * j + e);
            f01 = add2(make_float2(__uint_as_float(u[0]), __uint_as_float(u[1])), kzb2[hf][lg]);
            f23 = add2(make_float2(__uint_as_float(u[2]), __uint_as_float(u[3])), kzb2[hf][lg]);
          }
          const float2 x01 = mul2(f01, ks2[hf][lg]);
          const float2 x23 = mul2(f23, ks2[hf][lg]);
          af[hf][0] = pack_bf16x2(x01.x, x01.y);
          af[hf][1] = pack_bf16x2(x23.x, x23.y);
        }
        const uint32_t a[4] = {af[0][0], af[1][0], af[0][1], af[1][1]};
#pragma unroll
        for (int n = 0; n < NT; ++n) mma_bf16_16816(sacc[n][j & 1], a, qf[j][n][0], qf[j][n][1]);
      }

      // ---- values: tokens 2c, 2c + 1, 2c + 8, 2c + 9, elements [g EV, (g+1) EV):
      // packed words and scales loaded here, ahead of the softmax, whose
      // shuffles and exponentials their shared-memory latency then overlaps
      uint32_t wv[4][L::NWV];
      float2 vs2[4];
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const int tau = 2 * c + (k4 & 1) + 8 * (k4 >> 1);
        lds_words<L::NWV, L::VALIGN>(st + L::VC + tau * L::PDV, g * (L::EV * VB / 8), wv[k4]);
        const uint16_t* sv = reinterpret_cast<const uint16_t*>(st + L::VS);
        float sc = __half2float(__ushort_as_half(sv[tau * NG_FULL + half * L::NG + (g * L::EV) / kGroup]));
        if (!full) {
          // tokens past T or inside the left pad contribute exactly zero
          const int t = t0 + tau;
          sc = (t >= t_lo && t < p.T) ? sc : 0.0f;
        }
        vs2[k4] = f2(sc);
      }
      // ---- the team's partial scores added (SPL > 1): each warp publishes
      // its slice's sums in slot k mod 2 and adds all SPL slices in order
      // (the same terms in the same order in every warp, so the same sums)
      float sfull[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) sfull[n][e] = __fadd_rn(sacc[n][0][e], sacc[n][1][e]);
      if constexpr (SPL > 1) {
        float* slot = s_xchg + (k & 1) * (NW * 32 * NT * 4);
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) slot[((warp * NT + n) * 4 + e) * 32 + lane] = sfull[n][e];
        named_barrier(1 + team, 32 * SPL);
        // the slices' sums added in slice order (own slice from registers)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float tot = 0.0f;
#pragma unroll
            for (int h = 0; h < SPL; ++h) {
              const float o = h == half ? sfull[n][e] : slot[(((team * SPL + h) * NT + n) * 4 + e) * 32 + lane];
              tot = h == 0 ? o : __fadd_rn(tot, o);
            }
            sfull[n][e] = tot;
          }
      }

      // ---- online softmax per query column 8 n + 2 c + x (tokens g, g + 8
      // in entries x and 2 + x); the column's values sit in the eight lanes
      // with the same c
      float pr[NT][4];
      float al[NT][2];
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        float xs[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float sv = sfull[n][e];
          if (full) {
            xs[e] = __fmul_rn(sv, p.scale_log2);
          } else {
            const int t = t0 + g + 8 * (e >> 1);
            const bool ok = t >= t_lo && t <= hiq[n][e & 1];
            xs[e] = ok ? __fmul_rn(sv, p.scale_log2) : kNegInf;
          }
        }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          float mt = fmaxf(xs[x], xs[2 + x]);
          mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 4));
          mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 8));
          mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 16));
          const float mn = fmaxf(m_run[n][x], mt);
          const float mu = mn == kNegInf ? 0.0f : mn;
          al[n][x] = fast_exp2(__fsub_rn(m_run[n][x], mu));
          m_run[n][x] = mn;
          pr[n][x] = fast_exp2(__fsub_rn(xs[x], mu));
          pr[n][2 + x] = fast_exp2(__fsub_rn(xs[2 + x], mu));
          l_run[n][x] = __fadd_rn(__fmul_rn(l_run[n][x], al[n][x]), __fadd_rn(pr[n][x], pr[n][2 + x]));
        }
      }
      // rescale O^T: its columns are this lane's query columns 2 c, 2 c + 1
      {
        bool change = false;
#pragma unroll
        for (int n = 0; n < NT; ++n) change = change || al[n][0] != 1.0f || al[n][1] != 1.0f;
        if (__any_sync(kFull, change)) {
#pragma unroll
          for (int i = 0; i < DH / 16; ++i)
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              acc[i][n][0] = __fmul_rn(acc[i][n][0], al[n][0]);
              acc[i][n][1] = __fmul_rn(acc[i][n][1], al[n][1]);
              acc[i][n][2] = __fmul_rn(acc[i][n][2], al[n][0]);
              acc[i][n][3] = __fmul_rn(acc[i][n][3], al[n][1]);
            }
        }
      }
      // P^T operands (k = token, n = query row): the weights of tokens g and
      // g + 8 for query columns 2 c, 2 c + 1, split into bf16 hi + lo, then
      // transposed 8x8 by 8x8
      uint32_t bhi[NT][2], blo[NT][2];
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const float p0 = pr[n][2 * hf], p1 = pr[n][2 * hf + 1];
          const uint32_t hi = pack_bf16x2(p0, p1);
          const uint32_t lo = pack_bf16x2(__fsub_rn(p0, bf16_lo(hi)), __fsub_rn(p1, bf16_hi(hi)));
          bhi[n][hf] = movmatrix_trans(hi);
          blo[n][hf] = movmatrix_trans(lo);
        }

#pragma unroll
      for (int i = 0; i < DH / 16; ++i) {
        // elements 2i, 2i + 1 of each token: RN(centroid * scale), to bf16
        float2 v[4];
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          float2 cc;
          if constexpr (VB == 4) {
            cc = *reinterpret_cast<const float2*>(s_vtab + byte_field_addr(wv[k4], i, vstride, vlane));
          } else if constexpr (VB == 8) {
            cc = make_float2(*reinterpret_cast<const float*>(s_vtab + byte_field_addr(wv[k4], 2 * i, vstride, vlane)),
                             *reinterpret_cast<const float*>(s_vtab + byte_field_addr(wv[k4], 2 * i + 1, vstride, vlane)));
          } else if constexpr (VT::PAIRS) {
            cc = *reinterpret_cast<const float2*>(s_vtab + field_addr<2 * VB, 7>(wv[k4], 2 * i * VB, vlane));
          } else {
            cc = make_float2(*reinterpret_cast<const float*>(s_vtab + field_addr<VB, 7>(wv[k4], 2 * i * VB, vlane)),
                             *reinterpret_cast<const float*>(s_vtab + field_addr<VB, 7>(wv[k4], (2 * i + 1) * VB, vlane)));
          }
          v[k4] = mul2(cc, vs2[k4]);
        }
        const uint32_t a[4] = {pack_bf16x2(v[0].x, v[1].x), pack_bf16x2(v[0].y, v[1].y),
                               pack_bf16x2(v[2].x, v[3].x), pack_bf16x2(v[2].y, v[3].y)};
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          mma_bf16_16816(acc[i][n], a, bhi[n][0], bhi[n][1]);
          mma_bf16_16816(acc[i][n], a, blo[n][0], blo[n][1]);
        }
      }
    }
    cp_async_wait<0>();
    // column sums over the eight lanes of a column
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        l_run[n][x] = __fadd_rn(l_run[n][x], __shfl_xor_sync(kFull, l_run[n][x], 4));
        l_run[n][x] = __fadd_rn(l_run[n][x], __shfl_xor_sync(kFull, l_run[n][x], 8));
        l_run[n][x] = __fadd_rn(l_run[n][x], __shfl_xor_sync(kFull, l_run[n][x], 16));
      }

    // ---- merge the teams in shared memory, one record per block (the
    // warps of a team share m and l and each holds its half of O)
    __syncthreads();  // every warp is done with its ring
    float* mine = reinterpret_cast<float*>(s_work) + team * SM::REC;
    if (g == 0 && half == 0) {
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          mine[8 * n + 2 * c + x] = m_run[n][x];
          mine[16 + 8 * n + 2 * c + x] = l_run[n][x];
        }
    }
    {
      float* O = mine + 32 + half * DH;
#pragma unroll
      for (int i = 0; i < DH / 16; ++i)
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const int q0 = 8 * n + 2 * c, d0 = g * L::EV + 2 * i;
          O[q0 * D + d0] = acc[i][n][0];
          O[(q0 + 1) * D + d0] = acc[i][n][1];
          O[q0 * D + d0 + 1] = acc[i][n][2];
          O[(q0 + 1) * D + d0 + 1] = acc[i][n][3];
        }
    }
    __syncthreads();
    const float* all = reinterpret_cast<const float*>(s_work);
    if (!TQ_CHECK(static_cast<long long>(blockIdx.x) + bh < p.ws_records, p.err)) continue;
    float* rec = p.ws + (static_cast<long long>(blockIdx.x) + bh) * SM::REC;
    for (int i = threadIdx.x; i < Rq * D; i += blockDim.x) {
      const int r = i / D;
      float mx = kNegInf;
#pragma unroll
      for (int w = 0; w < kTeams; ++w) mx = fmaxf(mx, all[w * SM::REC + r]);
      float sum = 0.0f;
#pragma unroll
      for (int w = 0; w < kTeams; ++w) {
        const float mw = all[w * SM::REC + r];
        if (mw != kNegInf) sum = __fadd_rn(sum, __fmul_rn(exp2f(__fsub_rn(mw, mx)), all[w * SM::REC + 32 + i]));
      }
      rec[32 + i] = sum;
    }
    for (int r = threadIdx.x; r < Rq; r += blockDim.x) {
      float mx = kNegInf;
#pragma unroll
      for (int w = 0; w < kTeams; ++w) mx = fmaxf(mx, all[w * SM::REC + r]);
      float l = 0.0f;
#pragma unroll
      for (int w = 0; w < kTeams; ++w) {
        const float mw = all[w * SM::REC + r];
        if (mw != kNegInf) l = __fadd_rn(l, __fmul_rn(exp2f(__fsub_rn(mw, mx)), all[w * SM::REC + 16 + r]));
      }
      rec[r] = mx;
      rec[16 + r] = l;
    }
  }  // segments
}

// Merge of the split records of each output row, normalisation, inverse
// rotation (unrotateValues: fp32 Hadamard butterflies, * 1/sqrt(D), signs)
// and the store. Rows are taken in tiles of the codec's lane layout (lane l
// of a row owns elements [32 l, 32 l + 32)), and each tile by p.chunks
// blocks, block c merging the c-th of p.chunks equal runs of each row's
// records (a head spread over many split blocks has many records). Partial
// results (m, l, O: running max, weight sum and weighted row, relative to
// exp2(m)) merge online: with M = max(m, m'), the sum is
// exp2(m - M) (l, O) + exp2(m' - M) (l', O'), a factor taken as 0 for a
// part whose m is -inf (it saw no valid key). Each warp merges records w,
// w + NW, ... of the block's run in one pass, two records in flight; warp 0
// merges the warps' results in warp order. With one chunk it finishes the
// row. Otherwise it writes its (m, l, O) to the partial area and takes a
// ticket (threadfence, then an atomic add on the tile's counter, which the
// split pass zeroed): the block drawing the last ticket merges every
// chunk's result in chunk order and finishes the row. No block waits on
// another.
struct OnlinePart {
  float m, den, x[32];
};

__device__ __forceinline__ void online_merge(OnlinePart& a, float m, float den, const float (&x)[32]) {
  const float kNegInf = -__int_as_float(0x7f800000);
  const float mn = fmaxf(a.m, m);
  const float fa = a.m == mn ? 1.0f : (a.m == kNegInf ? 0.0f : exp2f(__fsub_rn(a.m, mn)));
  const float fb = m == kNegInf ? 0.0f : exp2f(__fsub_rn(m, mn));
  a.den = __fadd_rn(__fmul_rn(a.den, fa), __fmul_rn(den, fb));
#pragma unroll
  for (int i = 0; i < 32; ++i) a.x[i] = __fadd_rn(__fmul_rn(a.x[i], fa), __fmul_rn(x[i], fb));
  a.m = mn;
}

template <int D, bool F32>
__global__ void __launch_bounds__(32 * kCombineWarps) attn_combine_kernel(AttnParams p) {
  using G = Geo<D>;
  constexpr int REC = kAttnRows * (D + 2);
  constexpr int NW = kCombineWarps;
  const float kNegInf = -__int_as_float(0x7f800000);
  __shared__ __align__(16) uint32_t s_sign[D / 2];
  __shared__ float s_part[NW][34][32];  // per warp: 32 weighted sums, the weight sum and the max, per lane
  __shared__ unsigned s_ticket;
  fill_sign_words<D>(s_sign);
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / G::LPR;
  const int l = lane % G::LPR;
  const int tile = blockIdx.x / p.chunks;
  const int chunk = blockIdx.x - tile * p.chunks;
  const int rows = p.B * p.Hq * p.Nq;
  const int row0 = tile * G::RPW + sub;
  const bool valid = row0 < rows;
  const int row = valid ? row0 : rows - 1;
  const int hq_n = p.Hq * p.Nq;
  const int b = row / hq_n;
  const int rem = row - b * hq_n;
  const int hq = rem / p.Nq, n = rem - (rem / p.Nq) * p.Nq;
  const int h = hq / p.G;
  const int r = (hq - h * p.G) * p.Nq + n;
  // the split blocks that covered this head's tiles wrote records at slots
  // (block + bh); block of tile x = floor(((x + 1) grid - 1) / total)
  const int bh = b * p.Hkv + h;
  int c0 = 0, n_rec = 0;
  if (p.tiles_per_bh > 0) {
    const long long x0 = static_cast<long long>(bh) * p.tiles_per_bh, x1 = x0 + p.tiles_per_bh - 1;
    c0 = static_cast<int>(((x0 + 1) * p.grid - 1) / p.total_tiles);
    n_rec = static_cast<int>(((x1 + 1) * p.grid - 1) / p.total_tiles) - c0 + 1;
  }
  if (!TQ_CHECK(static_cast<long long>(c0) + bh + n_rec <= p.ws_records, p.err)) n_rec = 0;
  const float* recs = p.ws + (static_cast<long long>(c0) + bh) * REC;
  // this block's run of the row's records, merged online by the warps
  const int lo = static_cast<int>(static_cast<long long>(chunk) * n_rec / p.chunks);
  const int hi = static_cast<int>(static_cast<long long>(chunk + 1) * n_rec / p.chunks);
  OnlinePart acc;
  acc.m = kNegInf;
  acc.den = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) acc.x[i] = 0.0f;
#pragma unroll 2
  for (int s = lo + warp; s < hi; s += NW) {
    const float* rec = recs + s * REC;
    const float4* o = reinterpret_cast<const float4*>(rec + 32 + r * D + kGroup * l);
    float u[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = o[i];
      u[4 * i] = v.x; u[4 * i + 1] = v.y; u[4 * i + 2] = v.z; u[4 * i + 3] = v.w;
    }
    online_merge(acc, rec[r], rec[16 + r], u);
  }
  if (warp != 0) {
#pragma unroll
    for (int i = 0; i < 32; ++i) s_part[warp][i][lane] = acc.x[i];
    s_part[warp][32][lane] = acc.den;
    s_part[warp][33][lane] = acc.m;
  }
  __syncthreads();
  if (warp != 0) return;
#pragma unroll 1
  for (int w = 1; w < NW; ++w) {
    float x[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = s_part[w][i][lane];
    online_merge(acc, s_part[w][33][lane], s_part[w][32][lane], x);
  }
  if (p.chunks > 1) {
    if (!TQ_CHECK(tile < p.combine_tiles &&
                      (static_cast<long long>(tile) + 1) * p.chunks * kCombinePartialFloats <= p.partial_floats,
                  p.err))
      return;
    // publish this chunk's (m, l, O) (float i of lane L at 32 i + L), take a ticket
    float* mine = p.partials + (static_cast<long long>(tile) * p.chunks + chunk) * kCombinePartialFloats;
#pragma unroll
    for (int i = 0; i < 32; ++i) mine[32 * i + lane] = acc.x[i];
    mine[32 * 32 + lane] = acc.den;
    mine[32 * 33 + lane] = acc.m;
    __threadfence();
    __syncwarp();
    if (lane == 0) s_ticket = atomicAdd(p.counters + tile, 1u);
    __syncwarp();
    if (s_ticket != static_cast<unsigned>(p.chunks - 1)) return;  // not the last chunk to finish
    __threadfence();
    const float* all = p.partials + static_cast<long long>(tile) * p.chunks * kCombinePartialFloats;
    acc.m = kNegInf;
    acc.den = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) acc.x[i] = 0.0f;
#pragma unroll 1
    for (int c = 0; c < p.chunks; ++c) {
      const float* part = all + static_cast<long long>(c) * kCombinePartialFloats;
      float x[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = __ldcg(part + 32 * i + lane);
      online_merge(acc, __ldcg(part + 32 * 33 + lane), __ldcg(part + 32 * 32 + lane), x);
    }
  }
  uint32_t Sg[16];
  load_sign_words(s_sign, l, Sg);
  // a row with no valid key is zero
  const float den = acc.den;
  const bool empty = den == 0.0f;
  float2 Y[16];
#pragma unroll
  for (int q = 0; q < 16; ++q)
    Y[q] = empty ? make_float2(0.0f, 0.0f) : make_float2(__fdiv_rn(acc.x[q], den), __fdiv_rn(acc.x[q + 16], den));
  hadamard_row<G::LPR>(Y, l);
#pragma unroll
  for (int q = 0; q < 16; ++q) Y[q] = mul2(Y[q], f2(p.rot_scale));
  if (!valid) return;
  float y[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(__float_as_uint(pair_elem(Y, i)) ^ elem_sign(Sg, i));
  store_group<F32>(p.out, static_cast<size_t>(row) * D + kGroup * l, y);
}

// Launch with programmatic stream serialization and a given block size.
template <typename Params>
inline cudaError_t launch_pdl_block(void (*kernel)(Params), int grid, int block, const Params& p, cudaStream_t s,
                                    int dyn_smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = dyn_smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Sets p.grid to the split grid it launches.
template <int D, int VB, int KMODE, int NT>
cudaError_t launch_attn_split_t(AttnParams& p, cudaStream_t s) {
  using L = AttnSmem<D, KeySpec<KMODE>::B, VB, NT>;
  static const cudaError_t attr = cudaFuncSetAttribute(attn_split_kernel<D, VB, KMODE, NT>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (attr != cudaSuccess) return attr;
  static const int per_sm = [] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_split_kernel<D, VB, KMODE, NT>, L::Shape::THREADS,
                                                      L::SMEM) != cudaSuccess || n < 1)
      n = 1;
    return n;
  }();
  // one wave of resident blocks (at most kAttnGridPerSm per SM, the bound
  // the workspace is sized for), never more blocks than tiles
  long long grid = static_cast<long long>(per_sm < kAttnGridPerSm ? per_sm : kAttnGridPerSm) * sm_count();
  // each team of warps gets at least kAttnMinTeamTiles tiles, so the per-block
  // start (value table, query operands) and the record merge stay small next
  // to its work when few heads hold many tiles
  const long long teams = L::NW / AttnSplit<D>::SPL;
  const long long by_work = (p.total_tiles + teams * kAttnMinTeamTiles - 1) / (teams * kAttnMinTeamTiles);
  if (grid > by_work) grid = by_work;
  if (grid > p.total_tiles) grid = p.total_tiles;
  if (grid < 1) grid = 1;
  p.grid = static_cast<int>(grid);
  // a head's records: at most grid / (B Hkv) + 2
  p.chunks = attn_combine_chunks(grid / (static_cast<long long>(p.B) * p.Hkv) + 2);
  return launch_pdl_block(attn_split_kernel<D, VB, KMODE, NT>, p.grid, L::Shape::THREADS, p, s, L::SMEM);
}

template <int D, int VB, int NT>
cudaError_t launch_attn_split_vb(AttnParams& p, int kmode, cudaStream_t s) {
  switch (kmode) {
    case kK2: return launch_attn_split_t<D, VB, kK2, NT>(p, s);
    case kK4: return launch_attn_split_t<D, VB, kK4, NT>(p, s);
    case kK5: return launch_attn_split_t<D, VB, kK5, NT>(p, s);
    case kK8: return launch_attn_split_t<D, VB, kK8, NT>(p, s);
    default: return launch_attn_split_t<D, VB, kK8Signed, NT>(p, s);
  }
}

template <int D, int NT>
cudaError_t launch_attn_split_nt(AttnParams& p, int v_bits, int kmode, cudaStream_t s) {
  switch (v_bits) {
    case 2: return launch_attn_split_vb<D, 2, NT>(p, kmode, s);
    case 3: return launch_attn_split_vb<D, 3, NT>(p, kmode, s);
    case 4: return launch_attn_split_vb<D, 4, NT>(p, kmode, s);
    case 5: return launch_attn_split_vb<D, 5, NT>(p, kmode, s);
    default: return launch_attn_split_vb<D, 8, NT>(p, kmode, s);
  }
}

template <int D>
cudaError_t launch_attention(const AttnParams& params, int v_bits, int kmode, bool out_bf16, cudaStream_t s) {
  AttnParams p = params;
  const int rq = p.G * p.Nq;
  cudaError_t e = rq <= 8 ? launch_attn_split_nt<D, 1>(p, v_bits, kmode, s) : launch_attn_split_nt<D, 2>(p, v_bits, kmode, s);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.Nq;
  const long long tiles = (rows + Geo<D>::RPW - 1) / Geo<D>::RPW;  // p.chunks blocks per row tile
  const int grid = static_cast<int>(tiles * p.chunks);
  if (out_bf16) {
    e = launch_pdl(attn_combine_kernel<D, false>, grid, p, s, 0, 32 * kCombineWarps);
  } else {
    e = launch_pdl(attn_combine_kernel<D, true>, grid, p, s, 0, 32 * kCombineWarps);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace tq
