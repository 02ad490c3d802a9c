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
// Split kernel: one block of four warps per (batch, kv head, chunk of
// tokens). A warp streams 16-token tiles of the five packed buffers through
// its own ring of shared-memory stages (cp.async, 16-byte pieces) and, per
// tile:
//   scores  S = Q K^T on the tensor cores (mma.sync m16n8k16, bf16 in, fp32
//           accumulate): M = 16 query rows (the Hq/Hkv heads of the group
//           times Nq tokens), N = 8 tokens, K = 16 head_dim elements. The
//           head_dim order inside the contraction is permuted so that the
//           four lanes sharing a token each own a quarter of the row
//           (D/4 consecutive elements: exactly one quantisation group at
//           D = 128), so a lane decodes its own contiguous codes with its own
//           group scale and zero point, and the bf16 products are exact;
//   softmax online in fp32 (exp2 of scores pre-scaled by log2 e), per row;
//   values  O^T += V^T P^T, M = 16 head_dim elements, N = 8 query rows,
//           K = 16 tokens. P comes straight from the score accumulators (the
//           accumulator layout of one MMA is the operand layout of the
//           other), split as P = P_hi + P_lo in bf16 (two MMAs), which keeps
//           the weights exact to about 2^-18; the values are exact in bf16.
// The four warps' partial (max, sum, O) are merged in shared memory and the
// block writes one partial record to the workspace.
//
// Combine kernel: per output row, merges the chunk partials, divides by the
// softmax denominator and applies the inverse rotation in fp32 (the Hadamard
// butterflies of the codec, * 1/sqrt(D), then the signs: unrotateValues),
// storing fp32 or bf16.
#pragma once

#include "tq_kernels.cuh"

namespace tq {

constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = 32 * kAttnWarps;
constexpr int kAttnTile = 16;  // tokens per warp step
constexpr int kAttnRows = kAttnMaxRows;  // query rows per kv head (M of the score MMA)

__host__ __device__ constexpr int attn_round_up(int x, int m) { return (x + m - 1) / m * m; }

template <int D, int KB, int VB>
struct AttnLayout {
  static constexpr int NG = D / kGroup;
  static constexpr int PDK = D * KB / 8;
  static constexpr int PDV = D * VB / 8;
  static constexpr int STAGES = D >= 256 ? 2 : 3;
  // one stage: the tile's rows of the five packed buffers, back to back
  static constexpr int KC = 0;                        // K codes  [16][PDK]
  static constexpr int KS = KC + kAttnTile * PDK;     // K scales [16][NG] fp16
  static constexpr int KZ = KS + kAttnTile * NG * 2;  // K zeros
  static constexpr int VC = KZ + kAttnTile * NG * 2;  // V codes  [16][PDV]
  static constexpr int VS = VC + kAttnTile * PDV;     // V scales
  static constexpr int END = VS + kAttnTile * NG * 2;
  static constexpr int STAGE = attn_round_up(END + 16, 128);  // + room for word over-reads
  static constexpr int CENT = attn_round_up(CentroidTable<VB>::kWords * 4, 128);
  static constexpr int QROW = D + 8;  // bf16 per staged query row (16-byte pad: ldmatrix rows on distinct banks)
  static constexpr int QBYTES = attn_round_up(kAttnRows * QROW * 2, 128);
  static constexpr int RING = kAttnWarps * STAGES * STAGE;
  static constexpr int REC = kAttnRows * (D + 2);  // floats of a partial record: m[16], l[16], O[16][D]
  static_assert(REC == kAttnRecordFloats(D), "record layout shared with the host");
  static constexpr int MERGE = kAttnWarps * REC * 4;
  static constexpr int SMEM = CENT + QBYTES + (RING > MERGE ? RING : MERGE);
  // per-lane element ranges
  static constexpr int EK = D / 4;  // keys: token g, elements [c EK, (c+1) EK)
  static constexpr int EV = D / 8;  // values: elements [g EV, (g+1) EV) of four tokens
  static constexpr int NWK = (EK * KB + 31) / 32;
  static constexpr int NWV = (EV * VB + 31) / 32;
  static constexpr bool KALIGN = (EK * KB / 8) % 4 == 0;  // byte offset of a lane's key codes
  static constexpr bool VALIGN = (EV * VB / 8) % 4 == 0;
  static constexpr int KGROUPS = EK > kGroup ? EK / kGroup : 1;  // groups a lane's key range spans
};

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
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&a)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr));
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

template <int D, int VB, int KMODE, int NT>
__global__ void __launch_bounds__(kAttnThreads) attn_split_kernel(AttnParams p) {
  using M = KeySpec<KMODE>;
  constexpr int KB = M::B;
  using L = AttnLayout<D, KB, VB>;
  constexpr int S = L::STAGES;
  const float kNegInf = -__int_as_float(0x7f800000);
  extern __shared__ __align__(128) uint8_t smem[];
  float* s_cent = reinterpret_cast<float*>(smem);
  uint16_t* s_q = reinterpret_cast<uint16_t*>(smem + L::CENT);
  uint8_t* s_work = smem + L::CENT + L::QBYTES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int bh = blockIdx.x / p.n_chunks;
  const int chunk = blockIdx.x - bh * p.n_chunks;
  const int b = bh / p.Hkv, h = bh - b * p.Hkv;
  const int Rq = p.G * p.Nq;

  fill_centroids<VB>(s_cent);
  pdl_launch_dependents();
  pdl_wait();

  // The group's query rows (heads h G .. h G + G - 1, Nq tokens each: Rq
  // contiguous rows of q) in bf16, head_dim permuted: MMA k index kk of
  // k-step j holds element (kk % 8 / 2) * D/4 + 4 j + 2 (kk / 8) + kk % 2.
  {
    const uint16_t* qsrc = p.q + (static_cast<long long>(b) * p.Hq + static_cast<long long>(h) * p.G) * p.Nq * D;
    for (int i = threadIdx.x; i < kAttnRows * D; i += blockDim.x) {
      const int r = i / D, d = i - r * D;
      const int cq = d / L::EK, rem = d - cq * L::EK;
      const int j = rem >> 2, w4 = rem & 3;
      const int kk = 2 * cq + (w4 & 1) + 8 * (w4 >> 1);
      s_q[r * L::QROW + 16 * j + kk] = r < Rq ? qsrc[r * D + d] : static_cast<uint16_t>(0);
    }
  }
  const int t_lo = p.left_pad != nullptr ? max(p.left_pad[b], 0) : 0;
  int t_beg = chunk * p.chunk;
  const int t_end = min(t_beg + p.chunk, p.T);
  t_beg = max(t_beg, t_lo & ~(kAttnTile - 1));
  const int n_tiles = t_end > t_beg ? (t_end - t_beg + kAttnTile - 1) / kAttnTile : 0;
  // last key of the lane's two score rows (g and g + 8); -1 for padding rows
  const int hi0 = g < Rq ? p.T - p.Nq + g % p.Nq : -1;
  const int hi1 = g + 8 < Rq ? p.T - p.Nq + (g + 8) % p.Nq : -1;
  __syncthreads();

  uint8_t* ring = s_work + warp * S * L::STAGE;
  const uint32_t ring_sh = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
  const uint32_t q_sh = static_cast<uint32_t>(__cvta_generic_to_shared(s_q)) +
                        2u * static_cast<uint32_t>((lane & 15) * L::QROW + (lane >> 4) * 8);
  const long long tok0 = static_cast<long long>(bh) * p.t_cap + t_beg;
  const int my_tiles = n_tiles > warp ? (n_tiles - warp + kAttnWarps - 1) / kAttnWarps : 0;
  // Step k of this warp handles tile warp + 4 k in stage k mod S; every step
  // commits one copy group (empty past the end).
  auto issue = [&](int k) {
    if (k < my_tiles) {
      const long long t = tok0 + static_cast<long long>(warp + k * kAttnWarps) * kAttnTile;
      const uint32_t dst = ring_sh + (k % S) * L::STAGE;
      copy_region<kAttnTile * L::PDK>(dst + L::KC, p.k_codes + t * L::PDK, lane);
      copy_region<kAttnTile * L::NG * 2>(dst + L::KS, p.k_scales + t * L::NG, lane);
      copy_region<kAttnTile * L::NG * 2>(dst + L::KZ, p.k_zeros + t * L::NG, lane);
      copy_region<kAttnTile * L::PDV>(dst + L::VC, p.v_codes + t * L::PDV, lane);
      copy_region<kAttnTile * L::NG * 2>(dst + L::VS, p.v_scales + t * L::NG, lane);
    }
    cp_async_commit();
  };

  float acc[D / 16][NT][4];
#pragma unroll
  for (int i = 0; i < D / 16; ++i)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][n][e] = 0.0f;
  float m_run[2] = {kNegInf, kNegInf}, l_run[2] = {0.0f, 0.0f};
  const float* cent = s_cent + (CentroidTable<VB>::kRep > 1 ? lane : 0);
  constexpr int kCentStride = CentroidTable<VB>::kRep;
  constexpr float kBias = kMagic + (M::SIGNED ? 128.0f : 0.0f);

#pragma unroll
  for (int k = 0; k < S - 1; ++k) issue(k);
  for (int k = 0; k < my_tiles; ++k) {
    __syncwarp();
    issue(k + S - 1);
    cp_async_wait<S - 1>();
    __syncwarp();
    const uint8_t* st = ring + (k % S) * L::STAGE;
    const int t0 = t_beg + (warp + k * kAttnWarps) * kAttnTile;

    // ---- keys: token g of each 8-token half, elements [c EK, (c+1) EK)
    uint32_t wk[2][L::NWK];
    float ks[2][L::KGROUPS], kzb[2][L::KGROUPS];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int tau = 8 * nt + g;
      lds_words<L::NWK, L::KALIGN>(st + L::KC + tau * L::PDK, c * (L::EK * KB / 8), wk[nt]);
      if constexpr (M::SIGNED) {
#pragma unroll
        for (int w = 0; w < L::NWK; ++w) wk[nt][w] ^= 0x80808080u;  // code + 128 in each byte
      }
#pragma unroll
      for (int lg = 0; lg < L::KGROUPS; ++lg) {
        const int grp = (c * L::EK) / kGroup + lg;
        const uint16_t* sc = reinterpret_cast<const uint16_t*>(st + L::KS);
        const uint16_t* zr = reinterpret_cast<const uint16_t*>(st + L::KZ);
        ks[nt][lg] = __half2float(__ushort_as_half(sc[tau * L::NG + grp]));
        kzb[nt][lg] = __fsub_rn(__half2float(__ushort_as_half(zr[tau * L::NG + grp])), kBias);
      }
    }
    float sacc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      uint32_t a[4];
      ldmatrix_x4(a, q_sh + 32u * j);
      const int lg = (4 * j) / kGroup;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          // magic + bias + code, then + (zero - magic - bias) = code + zero exactly
          const float f = __uint_as_float(kMagicBits | code_at<KB>(wk[nt], 4 * j + e));
          x[e] = __fmul_rn(__fadd_rn(f, kzb[nt][lg]), ks[nt][lg]);
        }
        mma_bf16_16816(sacc[nt], a, pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
      }
    }

    // ---- online softmax of rows g (sacc[.][0..1]) and g + 8 (sacc[.][2..3])
    float xs[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = t0 + 8 * nt + 2 * c + (e & 1);
        const bool ok = t >= t_lo && t <= (e < 2 ? hi0 : hi1);
        xs[nt][e] = ok ? __fmul_rn(sacc[nt][e], p.scale_log2) : kNegInf;
      }
    float mt0 = fmaxf(fmaxf(xs[0][0], xs[0][1]), fmaxf(xs[1][0], xs[1][1]));
    float mt1 = fmaxf(fmaxf(xs[0][2], xs[0][3]), fmaxf(xs[1][2], xs[1][3]));
    mt0 = fmaxf(mt0, __shfl_xor_sync(kFull, mt0, 1));
    mt0 = fmaxf(mt0, __shfl_xor_sync(kFull, mt0, 2));
    mt1 = fmaxf(mt1, __shfl_xor_sync(kFull, mt1, 1));
    mt1 = fmaxf(mt1, __shfl_xor_sync(kFull, mt1, 2));
    const float mn0 = fmaxf(m_run[0], mt0), mn1 = fmaxf(m_run[1], mt1);
    const float mu0 = mn0 == kNegInf ? 0.0f : mn0, mu1 = mn1 == kNegInf ? 0.0f : mn1;
    const float al0 = exp2f(__fsub_rn(m_run[0], mu0)), al1 = exp2f(__fsub_rn(m_run[1], mu1));
    m_run[0] = mn0;
    m_run[1] = mn1;
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) pr[nt][e] = exp2f(__fsub_rn(xs[nt][e], e < 2 ? mu0 : mu1));
    l_run[0] = __fadd_rn(__fmul_rn(l_run[0], al0),
                         __fadd_rn(__fadd_rn(pr[0][0], pr[0][1]), __fadd_rn(pr[1][0], pr[1][1])));
    l_run[1] = __fadd_rn(__fmul_rn(l_run[1], al1),
                         __fadd_rn(__fadd_rn(pr[0][2], pr[0][3]), __fadd_rn(pr[1][2], pr[1][3])));
    // rescale O^T: its columns are query rows 2c, 2c + 1 (+ 8 for the second tile)
    {
      const float r00 = __shfl_sync(kFull, al0, 8 * c), r01 = __shfl_sync(kFull, al0, 8 * c + 4);
      const float r10 = __shfl_sync(kFull, al1, 8 * c), r11 = __shfl_sync(kFull, al1, 8 * c + 4);
      const bool change = r00 != 1.0f || r01 != 1.0f || (NT == 2 && (r10 != 1.0f || r11 != 1.0f));
      if (__any_sync(kFull, change)) {
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
          acc[i][0][0] = __fmul_rn(acc[i][0][0], r00);
          acc[i][0][1] = __fmul_rn(acc[i][0][1], r01);
          acc[i][0][2] = __fmul_rn(acc[i][0][2], r00);
          acc[i][0][3] = __fmul_rn(acc[i][0][3], r01);
          if constexpr (NT == 2) {
            acc[i][1][0] = __fmul_rn(acc[i][1][0], r10);
            acc[i][1][1] = __fmul_rn(acc[i][1][1], r11);
            acc[i][1][2] = __fmul_rn(acc[i][1][2], r10);
            acc[i][1][3] = __fmul_rn(acc[i][1][3], r11);
          }
        }
      }
    }
    // P^T operands (k = token, n = query row) from the score accumulators,
    // split into bf16 hi + lo
    uint32_t bhi[NT][2], blo[NT][2];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float p0 = pr[nt][2 * n], p1 = pr[nt][2 * n + 1];
        const uint32_t hi = pack_bf16x2(p0, p1);
        bhi[n][nt] = hi;
        blo[n][nt] = pack_bf16x2(__fsub_rn(p0, bf16_lo(hi)), __fsub_rn(p1, bf16_hi(hi)));
      }

    // ---- values: tokens 2c, 2c + 1, 2c + 8, 2c + 9, elements [g EV, (g+1) EV)
    uint32_t wv[4][L::NWV];
    float vs[4];
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      const int tau = 2 * c + (k4 & 1) + 8 * (k4 >> 1);
      lds_words<L::NWV, L::VALIGN>(st + L::VC + tau * L::PDV, g * (L::EV * VB / 8), wv[k4]);
      const int t = t0 + tau;
      const uint16_t* sv = reinterpret_cast<const uint16_t*>(st + L::VS);
      // tokens past T or inside the left pad contribute exactly zero
      vs[k4] = (t >= t_lo && t < p.T) ? __half2float(__ushort_as_half(sv[tau * L::NG + (g * L::EV) / kGroup])) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      float v[4][2];
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          v[k4][e] = __fmul_rn(cent[kCentStride * code_at<VB>(wv[k4], 2 * i + e)], vs[k4]);
      const uint32_t a[4] = {pack_bf16x2(v[0][0], v[1][0]), pack_bf16x2(v[0][1], v[1][1]),
                             pack_bf16x2(v[2][0], v[3][0]), pack_bf16x2(v[2][1], v[3][1])};
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        mma_bf16_16816(acc[i][n], a, bhi[n][0], bhi[n][1]);
        mma_bf16_16816(acc[i][n], a, blo[n][0], blo[n][1]);
      }
    }
  }
  cp_async_wait<0>();
  // row sums over the four lanes of a row
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_run[r] = __fadd_rn(l_run[r], __shfl_xor_sync(kFull, l_run[r], 1));
    l_run[r] = __fadd_rn(l_run[r], __shfl_xor_sync(kFull, l_run[r], 2));
  }

  // ---- merge the four warps in shared memory, one record per block
  __syncthreads();  // every warp is done with its ring
  float* mine = reinterpret_cast<float*>(s_work) + warp * L::REC;
  if (c == 0) {
    mine[g] = m_run[0];
    mine[g + 8] = m_run[1];
    mine[16 + g] = l_run[0];
    mine[16 + g + 8] = l_run[1];
  }
  {
    float* O = mine + 32;
#pragma unroll
    for (int i = 0; i < D / 16; ++i)
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
  float* rec = p.ws + static_cast<long long>(blockIdx.x) * L::REC;
  for (int i = threadIdx.x; i < Rq * D; i += blockDim.x) {
    const int r = i / D;
    float mx = kNegInf;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) mx = fmaxf(mx, all[w * L::REC + r]);
    float sum = 0.0f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float mw = all[w * L::REC + r];
      if (mw != kNegInf) sum = __fadd_rn(sum, __fmul_rn(exp2f(__fsub_rn(mw, mx)), all[w * L::REC + 32 + i]));
    }
    rec[32 + i] = sum;
  }
  for (int r = threadIdx.x; r < Rq; r += blockDim.x) {
    float mx = kNegInf;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) mx = fmaxf(mx, all[w * L::REC + r]);
    float l = 0.0f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float mw = all[w * L::REC + r];
      if (mw != kNegInf) l = __fadd_rn(l, __fmul_rn(exp2f(__fsub_rn(mw, mx)), all[w * L::REC + 16 + r]));
    }
    rec[r] = mx;
    rec[16 + r] = l;
  }
}

// Merge of the chunk partials of one output row, normalisation, inverse
// rotation (unrotateValues: fp32 Hadamard butterflies, * 1/sqrt(D), signs)
// and the store, with the codec's lane layout: lane l of a row owns elements
// [32 l, 32 l + 32).
template <int D, bool F32>
__global__ void __launch_bounds__(kThreads) attn_combine_kernel(AttnParams p) {
  using G = Geo<D>;
  constexpr int REC = kAttnRows * (D + 2);
  const float kNegInf = -__int_as_float(0x7f800000);
  __shared__ __align__(16) uint32_t s_sign[D / 2];
  fill_sign_words<D>(s_sign);
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int sub = lane / G::LPR;
  const int l = lane % G::LPR;
  const int n_warps = gridDim.x * (blockDim.x >> 5);
  const int rows = p.B * p.Hq * p.Nq;
  const int tiles = (rows + G::RPW - 1) / G::RPW;
  uint32_t Sg[16];
  load_sign_words(s_sign, l, Sg);
  for (int tile = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); tile < tiles; tile += n_warps) {
    const int row0 = tile * G::RPW + sub;
    const bool valid = row0 < rows;
    const int row = valid ? row0 : rows - 1;
    const int hq_n = p.Hq * p.Nq;
    const int b = row / hq_n;
    const int rem = row - b * hq_n;
    const int hq = rem / p.Nq, n = rem - (rem / p.Nq) * p.Nq;
    const int h = hq / p.G;
    const int r = (hq - h * p.G) * p.Nq + n;
    const float* recs = p.ws + static_cast<long long>(b * p.Hkv + h) * p.n_chunks * REC;
    float mx = kNegInf;
    for (int s = 0; s < p.n_chunks; ++s) mx = fmaxf(mx, recs[s * REC + r]);
    float x[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = 0.0f;
    float den = 0.0f;
    for (int s = 0; s < p.n_chunks; ++s) {
      const float* rec = recs + s * REC;
      const float ms = rec[r];
      if (ms == kNegInf) continue;
      const float f = exp2f(__fsub_rn(ms, mx));
      den = __fadd_rn(den, __fmul_rn(f, rec[16 + r]));
      const float4* o = reinterpret_cast<const float4*>(rec + 32 + r * D + kGroup * l);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 u = o[i];
        x[4 * i] = __fadd_rn(x[4 * i], __fmul_rn(f, u.x));
        x[4 * i + 1] = __fadd_rn(x[4 * i + 1], __fmul_rn(f, u.y));
        x[4 * i + 2] = __fadd_rn(x[4 * i + 2], __fmul_rn(f, u.z));
        x[4 * i + 3] = __fadd_rn(x[4 * i + 3], __fmul_rn(f, u.w));
      }
    }
    // a row with no valid key is zero
    const bool empty = den == 0.0f;
    float2 Y[16];
#pragma unroll
    for (int q = 0; q < 16; ++q)
      Y[q] = empty ? make_float2(0.0f, 0.0f) : make_float2(__fdiv_rn(x[q], den), __fdiv_rn(x[q + 16], den));
    hadamard_row<G::LPR>(Y, l);
#pragma unroll
    for (int q = 0; q < 16; ++q) Y[q] = mul2(Y[q], f2(p.rot_scale));
    if (!valid) continue;
    float y[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(__float_as_uint(pair_elem(Y, i)) ^ elem_sign(Sg, i));
    store_group<F32>(p.out, static_cast<size_t>(row) * D + kGroup * l, y);
  }
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

template <int D, int VB, int KMODE, int NT>
cudaError_t launch_attn_split_t(const AttnParams& p, cudaStream_t s) {
  using L = AttnLayout<D, KeySpec<KMODE>::B, VB>;
  static const cudaError_t attr = cudaFuncSetAttribute(attn_split_kernel<D, VB, KMODE, NT>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (attr != cudaSuccess) return attr;
  const int grid = p.B * p.Hkv * p.n_chunks;
  return launch_pdl_block(attn_split_kernel<D, VB, KMODE, NT>, grid, kAttnThreads, p, s, L::SMEM);
}

template <int D, int VB, int NT>
cudaError_t launch_attn_split_vb(const AttnParams& p, int kmode, cudaStream_t s) {
  switch (kmode) {
    case kK2: return launch_attn_split_t<D, VB, kK2, NT>(p, s);
    case kK4: return launch_attn_split_t<D, VB, kK4, NT>(p, s);
    case kK5: return launch_attn_split_t<D, VB, kK5, NT>(p, s);
    case kK8: return launch_attn_split_t<D, VB, kK8, NT>(p, s);
    default: return launch_attn_split_t<D, VB, kK8Signed, NT>(p, s);
  }
}

template <int D, int NT>
cudaError_t launch_attn_split_nt(const AttnParams& p, int v_bits, int kmode, cudaStream_t s) {
  switch (v_bits) {
    case 2: return launch_attn_split_vb<D, 2, NT>(p, kmode, s);
    case 3: return launch_attn_split_vb<D, 3, NT>(p, kmode, s);
    case 4: return launch_attn_split_vb<D, 4, NT>(p, kmode, s);
    case 5: return launch_attn_split_vb<D, 5, NT>(p, kmode, s);
    default: return launch_attn_split_vb<D, 8, NT>(p, kmode, s);
  }
}

template <int D>
cudaError_t launch_attention(const AttnParams& p, int v_bits, int kmode, bool out_bf16, cudaStream_t s) {
  const int rq = p.G * p.Nq;
  cudaError_t e = rq <= 8 ? launch_attn_split_nt<D, 1>(p, v_bits, kmode, s) : launch_attn_split_nt<D, 2>(p, v_bits, kmode, s);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.Nq;
  const long long tiles = (rows + Geo<D>::RPW - 1) / Geo<D>::RPW;
  if (out_bf16) {
    static const int resident = resident_blocks(attn_combine_kernel<D, false>);
    e = launch_pdl(attn_combine_kernel<D, false>, grid_for(tiles, resident), p, s);
  } else {
    static const int resident = resident_blocks(attn_combine_kernel<D, true>);
    e = launch_pdl(attn_combine_kernel<D, true>, grid_for(tiles, resident), p, s);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace tq
