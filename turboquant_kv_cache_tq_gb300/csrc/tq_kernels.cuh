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
//   K: t = RN(x * RN(1/se) - zp) differs from the page's RN(RN(x / se) - zp)
//      by at most (|x/se| + |zp|) * 2^-22 (four unit roundoffs), so whenever t
//      is farther than that from a half-integer both round to the same code.
//      A lane whose group has any element inside that band recomputes the
//      group with IEEE division; K codes are therefore exactly the page's.
//   V: u = RN(y * RN(1/se)) is within 2 ulp of RN(y / se) (|u| <= sqrt(32),
//      so within 1.1e-6); an index can only differ from the divided value's
//      when u is that close to a boundary.
//
// One warp handles Geo<D>::RPW rows per step of a grid-stride loop over all
// B*H*T rows; the grid is sized to the resident capacity of the GPU. Lanes of
// a partial last step redo the last row (so shuffles stay converged) but
// store nothing.
#pragma once

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

constexpr int kThreads = 256;

template <int KB, bool SIGNED>
struct KeyLevels {
  static constexpr int kMax = SIGNED ? (1 << (KB - 1)) - 1 : (1 << KB) - 1;
  static constexpr int kLo = SIGNED ? -kMax : 0;
  static constexpr int kHi = kMax;
};

// Exact per-element quantisation (the page's operations, IEEE division).
template <int KB, bool SIGNED>
__device__ __forceinline__ uint32_t key_code_exact(float x, float se, float zp) {
  using L = KeyLevels<KB, SIGNED>;
  float r = rintf(__fsub_rn(__fdiv_rn(x, se), zp));
  r = (r < static_cast<float>(L::kLo)) ? static_cast<float>(L::kLo) : r;
  r = (r > static_cast<float>(L::kHi)) ? static_cast<float>(L::kHi) : r;
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

// K encode of one group held by this lane; X = pairs (element p, p + 16).
template <int KB, bool SIGNED>
__device__ __forceinline__ void encode_key_group(const float2 (&X)[16], float mn, float mx, bool store,
                                                 uint8_t* codes, uint16_t* scale_out, uint16_t* zero_out) {
  using L = KeyLevels<KB, SIGNED>;
  if (mn == 0.0f || mx == 0.0f) scan_min_max(X, mn, mx);
  const float range = __fsub_rn(mx, mn);
  float scale, zp;
  if constexpr (SIGNED) {
    scale = __fdiv_rn(range, static_cast<float>(2 * L::kMax));
    const float denom = __fmul_rn(2.0f, __fadd_rn(scale, kEps));
    zp = rintf(__fdiv_rn(__fadd_rn(mx, mn), denom));
  } else {
    scale = __fdiv_rn(range, static_cast<float>(L::kMax));
    zp = rintf(__fdiv_rn(mn, __fadd_rn(scale, kEps)));
  }
  const float se = __fadd_rn(scale, kEps);
  const float inv = __frcp_rn(se);
  // guard band: (max|x| * inv + |zp|) * 2.5e-7 >= the fast/exact gap bound
  const float amax = fmaxf(fabsf(mn), fabsf(mx));
  const float band = __fmul_rn(__fadd_rn(__fmul_rn(amax, inv), fabsf(zp)), 2.5e-7f);
  const float thr = __fsub_rn(0.5f, band);
  const int lo_bits = static_cast<int>(kMagicBits) + L::kLo;
  const int hi_bits = static_cast<int>(kMagicBits) + L::kHi;

  uint32_t w[KB];
#pragma unroll
  for (int k = 0; k < KB; ++k) w[k] = 0;
  bool ok = true;
#pragma unroll
  for (int p = 0; p < 16; ++p) {
    const float2 t = fma2(X[p], f2(inv), f2(-zp));
    const float2 s = add2(t, f2(kMagic));
    const float2 d = sub2(t, sub2(s, f2(kMagic)));
    ok = ok && (fabsf(d.x) < thr) && (fabsf(d.y) < thr);
    put_code<KB>(w, p, static_cast<uint32_t>(min(max(__float_as_int(s.x), lo_bits), hi_bits)));
    put_code<KB>(w, p + 16, static_cast<uint32_t>(min(max(__float_as_int(s.y), lo_bits), hi_bits)));
  }
  if (!ok) {
#pragma unroll
    for (int k = 0; k < KB; ++k) w[k] = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) put_code<KB>(w, i, key_code_exact<KB, SIGNED>(pair_elem(X, i), se, zp));
  }
  if (store) {
    store_words<KB>(codes, w);
    *scale_out = __half_as_ushort(__float2half_rn(scale));
    *zero_out = __half_as_ushort(__float2half_rn(zp));
  }
}

// ---------------------------------------------------------------------------
template <int D, int VB, bool BF16>
__global__ void __launch_bounds__(kThreads) encode_kernel(EncodeParams p) {
  using G = Geo<D>;
  constexpr int NC = CellGrid<VB>::NC;
  __shared__ CellEntry s_cells[NC];
  __shared__ __align__(16) uint32_t s_sign[D / 2];
  {
    const CellEntry* tab = cell_table<VB>();
    for (int i = threadIdx.x; i < NC; i += blockDim.x) s_cells[i] = tab[i];
    fill_sign_words<D>(s_sign);
  }
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int sub = lane / G::LPR;
  const int l = lane % G::LPR;

  const int pdk = D * ((p.kmode == kK2) ? 2 : (p.kmode == kK4) ? 4 : (p.kmode == kK5) ? 5 : 8) / 8;
  const int kbytes = pdk / G::LPR;  // packed key bytes of one group
  constexpr int pdv = D * VB / 8;
  constexpr int NG = D / kGroup;
  const int warps_per_block = blockDim.x >> 5;
  const int n_warps = gridDim.x * warps_per_block;
  const int tiles = (p.rows + G::RPW - 1) / G::RPW;

  for (int tile = blockIdx.x * warps_per_block + (threadIdx.x >> 5); tile < tiles; tile += n_warps) {
    const int r0 = tile * G::RPW + sub;
    const bool valid = r0 < p.rows;
    const int r = valid ? r0 : p.rows - 1;
    const int bh = fast_div(r, p.tdiv);
    const int t = r - bh * p.T;
    const long long orow = static_cast<long long>(bh) * p.t_cap + p.t_off + t;
    const size_t in_off = static_cast<size_t>(r) * D + kGroup * l;

    // loads of both K and V are issued up front
    uint32_t wk[16], wv[16];
    float xk[BF16 ? 1 : 32], xv[BF16 ? 1 : 32];
    if constexpr (BF16) {
      load_words16(static_cast<const __nv_bfloat16*>(p.k) + in_off, wk);
      load_words16(static_cast<const __nv_bfloat16*>(p.v) + in_off, wv);
    } else {
      load_floats32(static_cast<const float*>(p.k) + in_off, xk);
      load_floats32(static_cast<const float*>(p.v) + in_off, xv);
    }

    // ---- keys
    {
      float2 X[16];
      float mn, mx;
      if constexpr (BF16) {
        // min / max on bf16 pairs (exact: the upcast preserves order)
        __nv_bfloat162 lo2 = *reinterpret_cast<const __nv_bfloat162*>(&wk[0]);
        __nv_bfloat162 hi2 = lo2;
#pragma unroll
        for (int j = 1; j < 16; ++j) {
          const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&wk[j]);
          lo2 = __hmin2(lo2, v2);
          hi2 = __hmax2(hi2, v2);
        }
        mn = fminf(__low2float(lo2), __high2float(lo2));
        mx = fmaxf(__low2float(hi2), __high2float(hi2));
        words_to_pairs(wk, X);
      } else {
        mn = xk[0];
        mx = xk[0];
#pragma unroll
        for (int i = 1; i < 32; ++i) {
          mn = fminf(mn, xk[i]);
          mx = fmaxf(mx, xk[i]);
        }
        floats_to_pairs(xk, X);
      }
      uint8_t* codes = p.k_codes + orow * pdk + kbytes * l;
      uint16_t* sc = p.k_scales + orow * NG + l;
      uint16_t* zr = p.k_zeros + orow * NG + l;
      switch (p.kmode) {
        case kK2: encode_key_group<2, false>(X, mn, mx, valid, codes, sc, zr); break;
        case kK4: encode_key_group<4, false>(X, mn, mx, valid, codes, sc, zr); break;
        case kK5: encode_key_group<5, false>(X, mn, mx, valid, codes, sc, zr); break;
        case kK8: encode_key_group<8, false>(X, mn, mx, valid, codes, sc, zr); break;
        default: encode_key_group<8, true>(X, mn, mx, valid, codes, sc, zr); break;
      }
    }

    // ---- values
    {
      uint32_t S[16];
      load_sign_words(s_sign, l, S);
      float2 Y[16];
      if constexpr (BF16) {
#pragma unroll
        for (int j = 0; j < 16; ++j) wv[j] ^= S[j];
        words_to_pairs(wv, Y);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) xv[i] = __uint_as_float(__float_as_uint(xv[i]) ^ elem_sign(S, i));
        floats_to_pairs(xv, Y);
      }
      hadamard_row<G::LPR>(Y, l);
      const float2 c2 = f2(p.rot_scale);
#pragma unroll
      for (int q = 0; q < 16; ++q) Y[q] = mul2(Y[q], c2);
      const float2 nz = f2(p.neg_zero);
      const float rms = __fsqrt_rn(__fmul_rn(group_sum_sq(Y, nz), 1.0f / kGroup));  // /32 is exact
      const float inv = __frcp_rn(__fadd_rn(rms, kEps));
      uint32_t w[VB];
#pragma unroll
      for (int k2 = 0; k2 < VB; ++k2) w[k2] = 0;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        int i0, i1;
        lm_index2<VB>(mul0(Y[q], f2(inv), nz), s_cells, i0, i1);
        put_code<VB>(w, q, static_cast<uint32_t>(i0));
        put_code<VB>(w, q + 16, static_cast<uint32_t>(i1));
      }
      if (valid) {
        store_words<VB>(p.v_codes + orow * pdv + 4 * VB * l, w);
        p.v_scales[orow * NG + l] = __half_as_ushort(__float2half_rn(rms));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// K decode of one group: x = (code + zero) * scale, zero and scale from fp16.
// Codes become floats through the 1.5 * 2^23 encoding (exact for |q| < 2^22).
template <int KB, bool SIGNED>
__device__ __forceinline__ void decode_key_group(const uint8_t* codes, float z, float s, float (&x)[32]) {
  uint32_t w[KB];
  load_words<KB>(codes, w);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    int q0 = static_cast<int>(unpack_code<KB>(w, i));
    int q1 = static_cast<int>(unpack_code<KB>(w, i + 1));
    if constexpr (SIGNED) {
      q0 = static_cast<int>(static_cast<int8_t>(q0));
      q1 = static_cast<int>(static_cast<int8_t>(q1));
    }
    float2 f = make_float2(__int_as_float(static_cast<int>(kMagicBits) + q0),
                           __int_as_float(static_cast<int>(kMagicBits) + q1));
    f = sub2(f, f2(kMagic));                 // the code, exactly
    f = mul2(add2(f, f2(z)), f2(s));         // (code + zero) * scale
    x[i] = f.x;
    x[i + 1] = f.y;
  }
}

template <bool BF16>
__device__ __forceinline__ void store_group(void* base, size_t off, const float (&x)[32]) {
  if constexpr (BF16) {
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

template <int D, int VB, bool BF16>
__global__ void __launch_bounds__(kThreads) decode_kernel(DecodeParams p) {
  using G = Geo<D>;
  constexpr int NCENT = 1 << VB;
  __shared__ float s_cent[NCENT];
  __shared__ __align__(16) uint32_t s_sign[D / 2];
  for (int i = threadIdx.x; i < NCENT; i += blockDim.x) s_cent[i] = centroid_table<VB>()[i];
  fill_sign_words<D>(s_sign);
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int sub = lane / G::LPR;
  const int l = lane % G::LPR;

  const int pdk = D * ((p.kmode == kK2) ? 2 : (p.kmode == kK4) ? 4 : (p.kmode == kK5) ? 5 : 8) / 8;
  const int kbytes = pdk / G::LPR;
  constexpr int pdv = D * VB / 8;
  constexpr int NG = D / kGroup;
  const int warps_per_block = blockDim.x >> 5;
  const int n_warps = gridDim.x * warps_per_block;
  const int tiles = (p.rows + G::RPW - 1) / G::RPW;

  for (int tile = blockIdx.x * warps_per_block + (threadIdx.x >> 5); tile < tiles; tile += n_warps) {
    const int r0 = tile * G::RPW + sub;
    const bool valid = r0 < p.rows;
    const int r = valid ? r0 : p.rows - 1;
    const int bh = fast_div(r, p.tdiv);
    const int t = r - bh * p.T;
    const long long irow = static_cast<long long>(bh) * p.t_cap + t;
    const size_t out_off = static_cast<size_t>(r) * D + kGroup * l;

    // ---- keys
    {
      const uint8_t* codes = p.k_codes + irow * pdk + kbytes * l;
      const float z = __half2float(__ushort_as_half(__ldg(p.k_zeros + irow * NG + l)));
      const float s = __half2float(__ushort_as_half(__ldg(p.k_scales + irow * NG + l)));
      float x[32];
      switch (p.kmode) {
        case kK2: decode_key_group<2, false>(codes, z, s, x); break;
        case kK4: decode_key_group<4, false>(codes, z, s, x); break;
        case kK5: decode_key_group<5, false>(codes, z, s, x); break;
        case kK8: decode_key_group<8, false>(codes, z, s, x); break;
        default: decode_key_group<8, true>(codes, z, s, x); break;
      }
      if (valid) store_group<BF16>(p.k_out, out_off, x);
    }

    // ---- values
    {
      uint32_t w[VB];
      load_words<VB>(p.v_codes + irow * pdv + 4 * VB * l, w);
      const float s = __half2float(__ushort_as_half(__ldg(p.v_scales + irow * NG + l)));
      float2 Y[16];
      const float2 nz = f2(p.neg_zero);
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float2 c = make_float2(s_cent[unpack_code<VB>(w, q)], s_cent[unpack_code<VB>(w, q + 16)]);
        Y[q] = mul0(c, f2(s), nz);  // feeds the butterflies: must stay rounded
      }
      hadamard_row<G::LPR>(Y, l);
      const float2 c2 = f2(p.rot_scale);
#pragma unroll
      for (int q = 0; q < 16; ++q) Y[q] = mul2(Y[q], c2);
      uint32_t S[16];
      load_sign_words(s_sign, l, S);
      if (valid) {
        if constexpr (BF16) {
          // round to bf16, then apply the signs on the packed words (exact)
          uint32_t o[16];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const __nv_bfloat162 a = __floats2bfloat162_rn(Y[2 * j].x, Y[2 * j + 1].x);
            const __nv_bfloat162 b = __floats2bfloat162_rn(Y[2 * j].y, Y[2 * j + 1].y);
            o[j] = *reinterpret_cast<const uint32_t*>(&a) ^ S[j];
            o[j + 8] = *reinterpret_cast<const uint32_t*>(&b) ^ S[j + 8];
          }
          uint4* q = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.v_out) + out_off);
#pragma unroll
          for (int i = 0; i < 4; ++i) q[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        } else {
          float x[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(__float_as_uint(pair_elem(Y, i)) ^ elem_sign(S, i));
          store_group<false>(p.v_out, out_off, x);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
template <typename K>
inline int resident_blocks(K kernel) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  return per_sm * sm_count();
}

inline int grid_for(long long tiles, int resident) {
  const long long needed = (tiles + (kThreads / 32) - 1) / (kThreads / 32);
  return static_cast<int>(needed < resident ? needed : resident);
}

template <int D, int VB, bool BF16>
cudaError_t launch_encode_t(const EncodeParams& p, cudaStream_t s) {
  static const int resident = resident_blocks(encode_kernel<D, VB, BF16>);
  const long long tiles = (p.rows + Geo<D>::RPW - 1) / Geo<D>::RPW;
  encode_kernel<D, VB, BF16><<<grid_for(tiles, resident), kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <int D, int VB, bool BF16>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t s) {
  static const int resident = resident_blocks(decode_kernel<D, VB, BF16>);
  const long long tiles = (p.rows + Geo<D>::RPW - 1) / Geo<D>::RPW;
  decode_kernel<D, VB, BF16><<<grid_for(tiles, resident), kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_encode(const EncodeParams& p, int v_bits, bool in_bf16, cudaStream_t s) {
  if (in_bf16) {
    switch (v_bits) {
      case 2: return launch_encode_t<D, 2, true>(p, s);
      case 3: return launch_encode_t<D, 3, true>(p, s);
      case 4: return launch_encode_t<D, 4, true>(p, s);
      case 5: return launch_encode_t<D, 5, true>(p, s);
      default: return launch_encode_t<D, 8, true>(p, s);
    }
  }
  switch (v_bits) {
    case 2: return launch_encode_t<D, 2, false>(p, s);
    case 3: return launch_encode_t<D, 3, false>(p, s);
    case 4: return launch_encode_t<D, 4, false>(p, s);
    case 5: return launch_encode_t<D, 5, false>(p, s);
    default: return launch_encode_t<D, 8, false>(p, s);
  }
}

template <int D>
cudaError_t launch_decode(const DecodeParams& p, int v_bits, bool out_bf16, cudaStream_t s) {
  if (out_bf16) {
    switch (v_bits) {
      case 2: return launch_decode_t<D, 2, true>(p, s);
      case 3: return launch_decode_t<D, 3, true>(p, s);
      case 4: return launch_decode_t<D, 4, true>(p, s);
      case 5: return launch_decode_t<D, 5, true>(p, s);
      default: return launch_decode_t<D, 8, true>(p, s);
    }
  }
  switch (v_bits) {
    case 2: return launch_decode_t<D, 2, false>(p, s);
    case 3: return launch_decode_t<D, 3, false>(p, s);
    case 4: return launch_decode_t<D, 4, false>(p, s);
    case 5: return launch_decode_t<D, 5, false>(p, s);
    default: return launch_decode_t<D, 8, false>(p, s);
  }
}

}  // namespace tq
