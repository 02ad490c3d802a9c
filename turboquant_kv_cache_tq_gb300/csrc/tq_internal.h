// Internal launch interface between the C ABI (tq_abi.cu) and the per-head_dim
// kernel translation units (tq_kernels_d*.cu). Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace tq {

// Row -> (b*h, t) by a multiply-shift (see fast_div in tq_device.cuh).
struct FastDiv {
  unsigned long long m;
  int shift;
};

// Bits of the library's device error word (see device_error_word).
constexpr unsigned kErrTimeout = 1u;  // a bounded wait gave up
constexpr unsigned kErrIndex = 2u;    // a debug build's index check failed

// Device-side index checks of a debug build (-DTQ_DEBUG_CHECKS): TQ_CHECK(ok,
// err) is `ok`, and a false `ok` also sets kErrIndex in *err; the caller
// skips the access. In a normal build it is `true` and compiles to nothing.
#ifdef TQ_DEBUG_CHECKS
#define TQ_CHECK(ok, err) (::tq::debug_check((ok), (err)))
#else
#define TQ_CHECK(ok, err) true
#endif

// Key modes: (bits, signed) pairs the key path supports.
enum KeyMode : int { kK2 = 0, kK4 = 1, kK5 = 2, kK8 = 3, kK8Signed = 4 };

struct EncodeParams {
  const void* k;        // [rows, D] inputs (fp32 or bf16)
  const void* v;
  uint8_t* k_codes;     // [B*H, t_cap, pd(D, k_bits)]
  uint16_t* k_scales;   // [B*H, t_cap, D/32] fp16 bits
  uint16_t* k_zeros;
  uint8_t* v_codes;     // [B*H, t_cap, pd(D, v_bits)]
  uint16_t* v_scales;
  int rows;             // B*H*T
  int T;                // tokens per (b, h) in the input
  long long t_cap;      // cache capacity in tokens
  long long t_off;      // first cache token written
  int kmode;            // KeyMode
  float rot_scale;      // fp32(1/sqrt(D))
  FastDiv tdiv;         // division by T
  float neg_zero;       // -0.0f (a runtime value, see mul0)
  long long cache_rows; // B*H*t_cap (debug checks)
  unsigned* err;        // the library's device error word, or null
};

struct DecodeParams {
  const uint8_t* k_codes;
  const uint16_t* k_scales;
  const uint16_t* k_zeros;
  const uint8_t* v_codes;
  const uint16_t* v_scales;
  void* k_out;          // [rows, D] outputs (fp32 or bf16)
  void* v_out;
  int rows;             // B*H*T
  int T;                // tokens decoded per (b, h)
  long long t_cap;
  int kmode;
  float rot_scale;
  FastDiv tdiv;
  float neg_zero;       // -0.0f
  int pdk, pdv;         // bytes of a packed K / V row
  int ng;               // groups per row (D / 32)
  unsigned* err;        // the library's device error word, or null
  long long cache_rows; // B*H*t_cap (debug checks)
  int device_memory;    // every buffer is device memory (bulk copies allowed)
};

struct UnrotateParams {
  const void* x;        // [rows, D] rotated values (fp32 or bf16)
  void* out;            // [rows, D] same type
  int rows;
  float rot_scale;
  unsigned* err;        // the library's device error word, or null
};

// Fused decode attention: at most 16 query rows per kv head (Hq/Hkv heads
// times Nq tokens); one partial record per split block holds m[16], l[16]
// and O[16][D] as floats.
constexpr int kAttnMaxRows = 16;
constexpr long long kAttnRecordFloats(long long D) { return kAttnMaxRows * (D + 2); }
// Split blocks per SM at most; the workspace holds (this * SMs + B * Hkv)
// records.
constexpr int kAttnGridPerSm = 8;
// Combine: warps per block; a head's records are merged by up to
// kCombineMaxChunks blocks of kCombineChunkRecords records each (four per
// warp), whose partial results (32 lanes x 34 floats per row tile and
// block: 32 weighted sums, the weight sum, the running max) the last of them
// to finish merges.
constexpr int kCombineWarps = 8;
constexpr int kCombineMaxChunks = 8;
#ifndef TQ_COMBINE_CHUNK_RECORDS
// (8, 16, 64 measured: within a microsecond either way on the head_dim 256 and
// 512 attention steps, none better on both)
#define TQ_COMBINE_CHUNK_RECORDS 32
#endif
constexpr int kCombineChunkRecords = TQ_COMBINE_CHUNK_RECORDS;
constexpr int kCombinePartialFloats = 32 * 34;
// Chunks for heads of at most n records.
inline int attn_combine_chunks(long long n) {
  const long long c = (n + kCombineChunkRecords - 1) / kCombineChunkRecords;
  return static_cast<int>(c < 1 ? 1 : (c > kCombineMaxChunks ? kCombineMaxChunks : c));
}

struct AttnParams {
  const uint16_t* q;    // [B, Hq, Nq, D] bf16 queries
  const uint8_t* k_codes;
  const uint16_t* k_scales;
  const uint16_t* k_zeros;
  const uint8_t* v_codes;
  const uint16_t* v_scales;
  const int* left_pad;  // [B] or null
  float* ws;            // partial records, one per (split block, head segment)
  void* out;            // [B, Hq, Nq, D] fp32 or bf16
  int B, Hq, Hkv, G, Nq, T;
  long long t_cap;      // multiple of 16
  long long total_tiles;  // B * Hkv * tiles_per_bh
  int tiles_per_bh;     // ceil(T / 16)
  int grid;             // split blocks (set by the launcher)
  float scale_log2;     // softmax scale * log2(e)
  float rot_scale;      // fp32(1/sqrt(D))
  long long cache_rows; // B * Hkv * t_cap (debug checks)
  long long ws_records; // records the workspace holds (debug checks)
  unsigned* err;        // the library's device error word, or null
  float* partials;      // combine partial sums [combine_tiles][chunks][32 x 33] (chunks > 1)
  unsigned* counters;   // combine tickets per row tile, zeroed by the split pass (chunks > 1)
  int chunks;           // combine blocks per row tile (set by the launcher)
  int combine_tiles;    // row tiles of the output (B * Hq * Nq rows)
  long long partial_floats;  // floats the partial area holds (debug checks)
  unsigned vtab_stride; // 128: bytes between entries of the value lookup table
};

// Launchers per head_dim, one translation unit per input or output type (and
// rotated V for decode): tq_encode_d<D>.cu (bf16 inputs), tq_encode_f32_d<D>.cu,
// tq_decode_d<D>.cu (bf16 outputs), tq_decode_f32_d<D>.cu, tq_decode_rot_d<D>.cu,
// tq_decode_rot_f32_d<D>.cu; v_bits in {2,3,4,5,8}.
template <int D, bool F32>
cudaError_t launch_encode_dt(const EncodeParams& p, int v_bits, cudaStream_t s);
template <int D>
inline cudaError_t launch_encode(const EncodeParams& p, int v_bits, bool in_bf16, cudaStream_t s) {
  return in_bf16 ? launch_encode_dt<D, false>(p, v_bits, s) : launch_encode_dt<D, true>(p, v_bits, s);
}
template <int D, bool F32, bool ROT>
cudaError_t launch_decode_dt(const DecodeParams& p, int v_bits, cudaStream_t s);
template <int D>
inline cudaError_t launch_decode(const DecodeParams& p, int v_bits, bool out_bf16, bool rotated_v, cudaStream_t s) {
  if (rotated_v)
    return out_bf16 ? launch_decode_dt<D, false, true>(p, v_bits, s) : launch_decode_dt<D, true, true>(p, v_bits, s);
  return out_bf16 ? launch_decode_dt<D, false, false>(p, v_bits, s) : launch_decode_dt<D, true, false>(p, v_bits, s);
}
template <int D>
cudaError_t launch_unrotate(const UnrotateParams& p, bool bf16, cudaStream_t s);

template <int D>
cudaError_t launch_attention(const AttnParams& p, int v_bits, int kmode, bool out_bf16, cudaStream_t s);

cudaError_t launch_lloyd_max_index(const float* u, long long n, int v_bits, uint8_t* idx, cudaStream_t s);

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Device address of the library's device error word on the current device
// (looked up on first use per device), or null if the lookup failed.
unsigned* device_error_word();

}  // namespace tq
