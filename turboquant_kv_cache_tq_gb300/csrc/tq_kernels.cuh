// Fused encode and decode kernels of the TurboQuant KV codec.
//
// Encode, per row (b, h, t) of K and V (page "@mlx-bun/inference 0.0.0-stage
// -> 1.0.0", file package/src/kernels/turboquant/ops.ts):
//   K: fp32 upcast, per-32-group min/max, scale = range / levels, zero point,
//      codes = clip(round(x / (scale + eps) - zero)), fp16 scale and zero
//      (encodeKeys), bit packing (packBits);
//   V: signs, normalised Hadamard transform (fwht, encode), per-32-group
//      RMS scale, Lloyd-Max index of x / (scale + eps) (encodeValues,
//      searchsorted), bit packing.
// Decode, per row: unpack, (code + zero) * scale for K (decodeKeys);
//   centroid * scale, Hadamard transform, signs for V (decodeValues).
//
// One warp handles Geo<D>::RPW rows per step of a grid-stride loop; the grid
// is sized to the resident capacity of the GPU. Lanes of a partial last step
// recompute the last row (so shuffles stay converged) but store nothing.
#pragma once

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

constexpr int kThreads = 256;

// ---------------------------------------------------------------------------
// K encode for one chunk of 8 elements.
template <int KB, bool SIGNED>
__device__ __forceinline__ void encode_key_chunk(const float (&x)[8], int l, int c, bool store,
                                                 uint8_t* codes_row, uint16_t* scales_row,
                                                 uint16_t* zeros_row) {
  constexpr int kMax = SIGNED ? (1 << (KB - 1)) - 1 : (1 << KB) - 1;
  float mn, mx;
  group_min_max(x, l, mn, mx);
  const float range = __fsub_rn(mx, mn);
  float scale, zp, lo, hi;
  if constexpr (SIGNED) {
    scale = __fdiv_rn(range, static_cast<float>(2 * kMax));
    const float denom = __fmul_rn(2.0f, __fadd_rn(scale, kEps));
    zp = rintf(__fdiv_rn(__fadd_rn(mx, mn), denom));
    lo = static_cast<float>(-kMax);
    hi = static_cast<float>(kMax);
  } else {
    scale = __fdiv_rn(range, static_cast<float>(kMax));
    zp = rintf(__fdiv_rn(mn, __fadd_rn(scale, kEps)));
    lo = 0.0f;
    hi = static_cast<float>(kMax);
  }
  const float se = __fadd_rn(scale, kEps);
  int q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float r = rintf(__fsub_rn(__fdiv_rn(x[i], se), zp));
    r = (r < lo) ? lo : r;
    r = (r > hi) ? hi : r;
    q[i] = static_cast<int>(r);
  }
  if (store) {
    store_packed<KB>(codes_row + chunk_byte<KB>(c, l), pack8<KB>(q));
    if ((l & 3) == 0) {
      const int g = chunk_elem(c, l) / kGroup;
      scales_row[g] = __half_as_ushort(__float2half_rn(scale));
      zeros_row[g] = __half_as_ushort(__float2half_rn(zp));
    }
  }
}

template <int D, int KB, bool SIGNED>
__device__ __forceinline__ void encode_key_row(const float (&x)[Geo<D>::CH][8], int l, bool store,
                                               uint8_t* codes_row, uint16_t* scales_row,
                                               uint16_t* zeros_row) {
#pragma unroll
  for (int c = 0; c < Geo<D>::CH; ++c)
    encode_key_chunk<KB, SIGNED>(x[c], l, c, store, codes_row, scales_row, zeros_row);
}

// ---------------------------------------------------------------------------
template <int D, int VB, typename InT>
__global__ void __launch_bounds__(kThreads) encode_kernel(EncodeParams p) {
  using G = Geo<D>;
  constexpr int CH = G::CH;
  constexpr int kCells = (VB >= 4) ? CellGrid<(VB >= 4 ? VB : 4)>::n : 1;
  __shared__ CellEntry s_cells[kCells];
  if constexpr (VB >= 4) {
    const CellEntry* tab = cell_table<VB>();
    for (int i = threadIdx.x; i < kCells; i += blockDim.x) s_cells[i] = tab[i];
    __syncthreads();
  }

  const int lane = threadIdx.x & 31;
  const int sub = lane / G::LPR;
  const int l = lane % G::LPR;
  uint32_t neg[CH];
#pragma unroll
  for (int c = 0; c < CH; ++c) neg[c] = sign_byte<D>(c * 32 + l);

  const int pdk = (p.kmode == kK2) ? D / 4 : (p.kmode == kK4) ? D / 2 : (p.kmode == kK5) ? D * 5 / 8 : D;
  constexpr int pdv = D * VB / 8;
  constexpr int NG = D / kGroup;
  const int warps_per_block = blockDim.x >> 5;
  const int n_warps = gridDim.x * warps_per_block;
  const int tiles = (p.rows + G::RPW - 1) / G::RPW;
  const InT* kin = static_cast<const InT*>(p.k);
  const InT* vin = static_cast<const InT*>(p.v);

  for (int tile = blockIdx.x * warps_per_block + (threadIdx.x >> 5); tile < tiles; tile += n_warps) {
    const int r0 = tile * G::RPW + sub;
    const bool valid = r0 < p.rows;
    const int r = valid ? r0 : p.rows - 1;
    const int bh = r / p.T;
    const int t = r - bh * p.T;
    const long long orow = static_cast<long long>(bh) * p.t_cap + p.t_off + t;
    const size_t in_off = static_cast<size_t>(r) * D;

    // ---- keys
    {
      float x[CH][8];
#pragma unroll
      for (int c = 0; c < CH; ++c) load8(kin + in_off + chunk_elem(c, l), x[c]);
      uint8_t* codes_row = p.k_codes + orow * pdk;
      uint16_t* sc_row = p.k_scales + orow * NG;
      uint16_t* zr_row = p.k_zeros + orow * NG;
      switch (p.kmode) {
        case kK2: encode_key_row<D, 2, false>(x, l, valid, codes_row, sc_row, zr_row); break;
        case kK4: encode_key_row<D, 4, false>(x, l, valid, codes_row, sc_row, zr_row); break;
        case kK5: encode_key_row<D, 5, false>(x, l, valid, codes_row, sc_row, zr_row); break;
        case kK8: encode_key_row<D, 8, false>(x, l, valid, codes_row, sc_row, zr_row); break;
        default: encode_key_row<D, 8, true>(x, l, valid, codes_row, sc_row, zr_row); break;
      }
    }

    // ---- values
    {
      float y[CH][8];
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        load8(vin + in_off + chunk_elem(c, l), y[c]);
        apply_signs(y[c], neg[c]);
      }
      hadamard_unnormalised<D>(y, l);
      uint8_t* codes_row = p.v_codes + orow * pdv;
      uint16_t* sc_row = p.v_scales + orow * NG;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
#pragma unroll
        for (int i = 0; i < 8; ++i) y[c][i] = __fmul_rn(y[c][i], p.rot_scale);
        const float mean_sq = __fmul_rn(group_sum_sq(y[c]), 1.0f / kGroup);  // exact: a power of two
        const float rms = __fsqrt_rn(mean_sq);
        const float se = __fadd_rn(rms, kEps);
        int q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = lm_index<VB>(__fdiv_rn(y[c][i], se), s_cells);
        if (valid) {
          store_packed<VB>(codes_row + chunk_byte<VB>(c, l), pack8<VB>(q));
          if ((l & 3) == 0) sc_row[chunk_elem(c, l) / kGroup] = __half_as_ushort(__float2half_rn(rms));
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// K decode of one chunk: x = (code + zero) * scale, zero and scale from fp16.
template <int KB, bool SIGNED>
__device__ __forceinline__ void decode_key_chunk(const uint8_t* codes_row, const uint16_t* scales_row,
                                                 const uint16_t* zeros_row, int l, int c, float (&x)[8]) {
  const uint64_t acc = load_packed<KB>(codes_row + chunk_byte<KB>(c, l));
  const int g = chunk_elem(c, l) / kGroup;
  const float z = __half2float(__ushort_as_half(__ldg(zeros_row + g)));
  const float s = __half2float(__ushort_as_half(__ldg(scales_row + g)));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int q = unpack_code<KB>(acc, i);
    if constexpr (SIGNED) q = static_cast<int>(static_cast<int8_t>(static_cast<uint8_t>(q)));
    x[i] = __fmul_rn(__fadd_rn(static_cast<float>(q), z), s);
  }
}

template <int D, int KB, bool SIGNED>
__device__ __forceinline__ void decode_key_row(const uint8_t* codes_row, const uint16_t* scales_row,
                                               const uint16_t* zeros_row, int l,
                                               float (&x)[Geo<D>::CH][8]) {
#pragma unroll
  for (int c = 0; c < Geo<D>::CH; ++c) decode_key_chunk<KB, SIGNED>(codes_row, scales_row, zeros_row, l, c, x[c]);
}

template <int D, int VB, typename OutT>
__global__ void __launch_bounds__(kThreads) decode_kernel(DecodeParams p) {
  using G = Geo<D>;
  constexpr int CH = G::CH;
  constexpr int NC = 1 << VB;
  __shared__ float s_cent[NC];
  for (int i = threadIdx.x; i < NC; i += blockDim.x) s_cent[i] = centroid_table<VB>()[i];
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int sub = lane / G::LPR;
  const int l = lane % G::LPR;
  uint32_t neg[CH];
#pragma unroll
  for (int c = 0; c < CH; ++c) neg[c] = sign_byte<D>(c * 32 + l);

  const int pdk = (p.kmode == kK2) ? D / 4 : (p.kmode == kK4) ? D / 2 : (p.kmode == kK5) ? D * 5 / 8 : D;
  constexpr int pdv = D * VB / 8;
  constexpr int NG = D / kGroup;
  const int warps_per_block = blockDim.x >> 5;
  const int n_warps = gridDim.x * warps_per_block;
  const int tiles = (p.rows + G::RPW - 1) / G::RPW;
  OutT* kout = static_cast<OutT*>(p.k_out);
  OutT* vout = static_cast<OutT*>(p.v_out);

  for (int tile = blockIdx.x * warps_per_block + (threadIdx.x >> 5); tile < tiles; tile += n_warps) {
    const int r0 = tile * G::RPW + sub;
    const bool valid = r0 < p.rows;
    const int r = valid ? r0 : p.rows - 1;
    const int bh = r / p.T;
    const int t = r - bh * p.T;
    const long long irow = static_cast<long long>(bh) * p.t_cap + t;
    const size_t out_off = static_cast<size_t>(r) * D;

    // ---- keys
    {
      float x[CH][8];
      const uint8_t* codes_row = p.k_codes + irow * pdk;
      const uint16_t* sc_row = p.k_scales + irow * NG;
      const uint16_t* zr_row = p.k_zeros + irow * NG;
      switch (p.kmode) {
        case kK2: decode_key_row<D, 2, false>(codes_row, sc_row, zr_row, l, x); break;
        case kK4: decode_key_row<D, 4, false>(codes_row, sc_row, zr_row, l, x); break;
        case kK5: decode_key_row<D, 5, false>(codes_row, sc_row, zr_row, l, x); break;
        case kK8: decode_key_row<D, 8, false>(codes_row, sc_row, zr_row, l, x); break;
        default: decode_key_row<D, 8, true>(codes_row, sc_row, zr_row, l, x); break;
      }
      if (valid) {
#pragma unroll
        for (int c = 0; c < CH; ++c) store8(kout + out_off + chunk_elem(c, l), x[c]);
      }
    }

    // ---- values
    {
      float y[CH][8];
      const uint8_t* codes_row = p.v_codes + irow * pdv;
      const uint16_t* sc_row = p.v_scales + irow * NG;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const uint64_t acc = load_packed<VB>(codes_row + chunk_byte<VB>(c, l));
        const float s = __half2float(__ushort_as_half(__ldg(sc_row + chunk_elem(c, l) / kGroup)));
#pragma unroll
        for (int i = 0; i < 8; ++i) y[c][i] = __fmul_rn(s_cent[unpack_code<VB>(acc, i)], s);
      }
      hadamard_unnormalised<D>(y, l);
#pragma unroll
      for (int c = 0; c < CH; ++c) {
#pragma unroll
        for (int i = 0; i < 8; ++i) y[c][i] = __fmul_rn(y[c][i], p.rot_scale);
        apply_signs(y[c], neg[c]);
        if (valid) store8(vout + out_off + chunk_elem(c, l), y[c]);
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

template <int D, int VB, typename InT>
cudaError_t launch_encode_t(const EncodeParams& p, cudaStream_t s) {
  static const int resident = resident_blocks(encode_kernel<D, VB, InT>);
  const long long tiles = (p.rows + Geo<D>::RPW - 1) / Geo<D>::RPW;
  encode_kernel<D, VB, InT><<<grid_for(tiles, resident), kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <int D, int VB, typename OutT>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t s) {
  static const int resident = resident_blocks(decode_kernel<D, VB, OutT>);
  const long long tiles = (p.rows + Geo<D>::RPW - 1) / Geo<D>::RPW;
  decode_kernel<D, VB, OutT><<<grid_for(tiles, resident), kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_encode(const EncodeParams& p, int v_bits, bool in_bf16, cudaStream_t s) {
  if (in_bf16) {
    switch (v_bits) {
      case 2: return launch_encode_t<D, 2, __nv_bfloat16>(p, s);
      case 3: return launch_encode_t<D, 3, __nv_bfloat16>(p, s);
      case 4: return launch_encode_t<D, 4, __nv_bfloat16>(p, s);
      case 5: return launch_encode_t<D, 5, __nv_bfloat16>(p, s);
      default: return launch_encode_t<D, 8, __nv_bfloat16>(p, s);
    }
  }
  switch (v_bits) {
    case 2: return launch_encode_t<D, 2, float>(p, s);
    case 3: return launch_encode_t<D, 3, float>(p, s);
    case 4: return launch_encode_t<D, 4, float>(p, s);
    case 5: return launch_encode_t<D, 5, float>(p, s);
    default: return launch_encode_t<D, 8, float>(p, s);
  }
}

template <int D>
cudaError_t launch_decode(const DecodeParams& p, int v_bits, bool out_bf16, cudaStream_t s) {
  if (out_bf16) {
    switch (v_bits) {
      case 2: return launch_decode_t<D, 2, __nv_bfloat16>(p, s);
      case 3: return launch_decode_t<D, 3, __nv_bfloat16>(p, s);
      case 4: return launch_decode_t<D, 4, __nv_bfloat16>(p, s);
      case 5: return launch_decode_t<D, 5, __nv_bfloat16>(p, s);
      default: return launch_decode_t<D, 8, __nv_bfloat16>(p, s);
    }
  }
  switch (v_bits) {
    case 2: return launch_decode_t<D, 2, float>(p, s);
    case 3: return launch_decode_t<D, 3, float>(p, s);
    case 4: return launch_decode_t<D, 4, float>(p, s);
    case 5: return launch_decode_t<D, 5, float>(p, s);
    default: return launch_decode_t<D, 8, float>(p, s);
  }
}

}  // namespace tq
