// C ABI of the TurboQuant KV codec (declared in include/tq.h): argument
// checks on the host, then one fused kernel per call on the caller's stream.
// Page "@mlx-bun/inference 0.0.0-stage -> 1.0.0", file
// package/src/kernels/turboquant/ops.ts: packedDim throws on a non-byte-aligned
// size, fwht rejects unsupported head dims, the Lloyd-Max tables exist for
// 2/3/4/5/8 bits and signed keys exist only at 8 bits; each of those becomes a
// status code returned before any launch.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/tq.h"
#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

int sm_count() {
  static int cached[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

namespace {

// The library's device error word: kernels whose bounded waits give up set a
// bit here (bit 0: a decode stage never arrived); read and cleared by
// tq_device_status. Its device address is looked up once per device.
__device__ unsigned g_device_error;
std::mutex g_err_mutex;
unsigned* g_err_ptr[128] = {nullptr};

}  // namespace

unsigned* device_error_word() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(g_err_mutex);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_err_ptr[dev];
}

namespace {

__global__ void lloyd_max_index_kernel(const float* u, long long n, int v_bits, uint8_t* idx) {
  __shared__ CellEntry s_cells[CellGrid<8>::NC];
  const CellEntry* tab = v_bits == 2 ? cell_table<2>() : v_bits == 3 ? cell_table<3>() : v_bits == 4 ? cell_table<4>()
                       : v_bits == 5 ? cell_table<5>() : cell_table<8>();
  const int nc = v_bits == 2 ? CellGrid<2>::NC : v_bits == 3 ? CellGrid<3>::NC : v_bits == 4 ? CellGrid<4>::NC
               : v_bits == 5 ? CellGrid<5>::NC : CellGrid<8>::NC;
  for (int i = threadIdx.x; i < nc; i += blockDim.x) s_cells[i] = tab[i];
  __syncthreads();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n; i += stride) {
    const float x = u[i];
    int r;
    switch (v_bits) {
      case 2: r = lm_index_any<2>(x, s_cells); break;
      case 3: r = lm_index_any<3>(x, s_cells); break;
      case 4: r = lm_index_any<4>(x, s_cells); break;
      case 5: r = lm_index_any<5>(x, s_cells); break;
      default: r = lm_index_any<8>(x, s_cells); break;
    }
    idx[i] = static_cast<uint8_t>(r);
  }
}

bool head_dim_ok(int64_t d) { return d == 64 || d == 128 || d == 256 || d == 512; }
bool value_bits_ok(int b) { return b == 2 || b == 3 || b == 4 || b == 5 || b == 8; }

// Key mode of (bits, signed), or -1.
int key_mode(int bits, int is_signed) {
  if (is_signed) return bits == 8 ? kK8Signed : -1;
  switch (bits) {
    case 2: return kK2;
    case 4: return kK4;
    case 5: return kK5;
    case 8: return kK8;
    default: return -1;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Whether every pointer is device memory (as opposed to pinned host memory
// mapped into the device's address space, managed or unregistered memory).
// Bulk asynchronous copies are only used between device and shared memory.
bool all_device_memory(const void* const* ptrs, int n) {
  for (int i = 0; i < n; ++i) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, ptrs[i]) != cudaSuccess) {
      cudaGetLastError();  // leave no sticky error behind
      return false;
    }
    if (a.type != cudaMemoryTypeDevice) return false;
  }
  return true;
}

// Shared checks of encode and decode; fills rows.
tq_status check_common(int64_t B, int64_t H, int64_t T, int64_t D, int64_t t_cap, int64_t t_off,
                       int k_bits, int k_signed, int v_bits, int dtype, long long* rows) {
  if (B < 0 || H < 0 || T < 0 || t_cap < 0 || t_off < 0) return TQ_ERR_INVALID_ARG;
  if (!head_dim_ok(D)) return TQ_ERR_HEAD_DIM;
  if (key_mode(k_bits, k_signed) < 0 || !value_bits_ok(v_bits)) return TQ_ERR_BITS;
  if (dtype != TQ_F32 && dtype != TQ_BF16) return TQ_ERR_DTYPE;
  if (t_off > t_cap || T > t_cap - t_off) return TQ_ERR_INVALID_ARG;
  // Row indices and per-(b,h) token counts are 32-bit inside the kernels.
  const long long lim = 0x7fffffffLL;
  if (T > lim || t_cap > lim) return TQ_ERR_INVALID_ARG;
  if (B > lim || H > lim || (B > 0 && H > lim / B)) return TQ_ERR_INVALID_ARG;
  const long long bh = B * H;
  if (bh > 0 && T > lim / bh) return TQ_ERR_INVALID_ARG;
  if (bh > 0 && t_cap > (1LL << 62) / (bh * 512)) return TQ_ERR_INVALID_ARG;
  *rows = bh * T;
  // Item indices, including those a warp computes a few steps past the end
  // (its prefetches), stay in int with 2^24 to spare.
  if (*rows > lim - (1LL << 24)) return TQ_ERR_INVALID_ARG;
  return TQ_OK;
}

float rotation_scale(int64_t d) { return static_cast<float>(1.0 / std::sqrt(static_cast<double>(d))); }

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" int64_t tq_packed_dim(int64_t dim, int bits) {
  if (dim < 0 || bits < 1) return -static_cast<int64_t>(TQ_ERR_INVALID_ARG);
  if (dim > (INT64_MAX / 64)) return -static_cast<int64_t>(TQ_ERR_INVALID_ARG);
  if ((dim * bits) % 8 != 0) return -static_cast<int64_t>(TQ_ERR_ALIGNMENT);
  return dim * bits / 8;
}

extern "C" tq_status tq_encode_kv(const void* k, const void* v, tq_dtype in_dtype,
                                  int64_t B, int64_t H, int64_t T, int64_t D,
                                  int k_bits, int k_signed, int v_bits,
                                  void* k_codes, void* k_scales, void* k_zeros,
                                  void* v_codes, void* v_scales,
                                  int64_t t_cap, int64_t t_off, void* stream) {
  long long rows = 0;
  const tq_status st = check_common(B, H, T, D, t_cap, t_off, k_bits, k_signed, v_bits,
                                    static_cast<int>(in_dtype), &rows);
  if (st != TQ_OK) return st;
  if (rows == 0) return TQ_OK;
  const void* ptrs[] = {k, v, k_codes, k_scales, k_zeros, v_codes, v_scales};
  for (const void* p : ptrs) {
    if (!p) return TQ_ERR_INVALID_ARG;
    if (!aligned16(p)) return TQ_ERR_ALIGNMENT;
  }
  EncodeParams p{};
  p.k = k;
  p.v = v;
  p.k_codes = static_cast<uint8_t*>(k_codes);
  p.k_scales = static_cast<uint16_t*>(k_scales);
  p.k_zeros = static_cast<uint16_t*>(k_zeros);
  p.v_codes = static_cast<uint8_t*>(v_codes);
  p.v_scales = static_cast<uint16_t*>(v_scales);
  p.rows = static_cast<int>(rows);
  p.T = static_cast<int>(T);
  p.t_cap = t_cap;
  p.t_off = t_off;
  p.kmode = key_mode(k_bits, k_signed);
  p.rot_scale = rotation_scale(D);
  p.tdiv = make_fast_div(static_cast<int>(T));
  p.neg_zero = -0.0f;
  p.cache_rows = B * H * t_cap;
  p.err = device_error_word();
  const bool bf16 = in_dtype == TQ_BF16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (D) {
    case 64: e = launch_encode<64>(p, v_bits, bf16, s); break;
    case 128: e = launch_encode<128>(p, v_bits, bf16, s); break;
    case 256: e = launch_encode<256>(p, v_bits, bf16, s); break;
    default: e = launch_encode<512>(p, v_bits, bf16, s); break;
  }
  return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

namespace tq {
namespace {

tq_status decode_impl(const void* k_codes, const void* k_scales, const void* k_zeros, const void* v_codes,
                      const void* v_scales, int64_t B, int64_t H, int64_t T, int64_t D, int64_t t_cap, int k_bits,
                      int k_signed, int v_bits, void* k_out, void* v_out, tq_dtype out_dtype, bool rotated_v,
                      void* stream) {
  long long rows = 0;
  const tq_status st = check_common(B, H, T, D, t_cap, 0, k_bits, k_signed, v_bits,
                                    static_cast<int>(out_dtype), &rows);
  if (st != TQ_OK) return st;
  if (rows == 0) return TQ_OK;
  const void* ptrs[] = {k_codes, k_scales, k_zeros, v_codes, v_scales, k_out, v_out};
  for (const void* p : ptrs) {
    if (!p) return TQ_ERR_INVALID_ARG;
    if (!aligned16(p)) return TQ_ERR_ALIGNMENT;
  }
  DecodeParams p{};
  p.k_codes = static_cast<const uint8_t*>(k_codes);
  p.k_scales = static_cast<const uint16_t*>(k_scales);
  p.k_zeros = static_cast<const uint16_t*>(k_zeros);
  p.v_codes = static_cast<const uint8_t*>(v_codes);
  p.v_scales = static_cast<const uint16_t*>(v_scales);
  p.k_out = k_out;
  p.v_out = v_out;
  p.rows = static_cast<int>(rows);
  p.T = static_cast<int>(T);
  p.t_cap = t_cap;
  p.pdk = static_cast<int>(D * k_bits / 8);
  p.pdv = static_cast<int>(D * v_bits / 8);
  p.ng = static_cast<int>(D / 32);
  p.kmode = key_mode(k_bits, k_signed);
  p.rot_scale = rotation_scale(D);
  p.tdiv = make_fast_div(static_cast<int>(T));
  p.neg_zero = -0.0f;
  p.err = device_error_word();
  p.cache_rows = B * H * t_cap;
  p.device_memory = out_dtype == TQ_BF16 && all_device_memory(ptrs, 7) ? 1 : 0;
  const bool bf16 = out_dtype == TQ_BF16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (D) {
    case 64: e = launch_decode<64>(p, v_bits, bf16, rotated_v, s); break;
    case 128: e = launch_decode<128>(p, v_bits, bf16, rotated_v, s); break;
    case 256: e = launch_decode<256>(p, v_bits, bf16, rotated_v, s); break;
    default: e = launch_decode<512>(p, v_bits, bf16, rotated_v, s); break;
  }
  return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace
}  // namespace tq

extern "C" tq_status tq_decode_kv(const void* k_codes, const void* k_scales, const void* k_zeros,
                                  const void* v_codes, const void* v_scales,
                                  int64_t B, int64_t H, int64_t T, int64_t D, int64_t t_cap,
                                  int k_bits, int k_signed, int v_bits,
                                  void* k_out, void* v_out, tq_dtype out_dtype, void* stream) {
  return decode_impl(k_codes, k_scales, k_zeros, v_codes, v_scales, B, H, T, D, t_cap, k_bits, k_signed, v_bits,
                     k_out, v_out, out_dtype, false, stream);
}

extern "C" tq_status tq_decode_kv_rotated(const void* k_codes, const void* k_scales, const void* k_zeros,
                                          const void* v_codes, const void* v_scales,
                                          int64_t B, int64_t H, int64_t T, int64_t D, int64_t t_cap,
                                          int k_bits, int k_signed, int v_bits,
                                          void* k_out, void* v_out, tq_dtype out_dtype, void* stream) {
  return decode_impl(k_codes, k_scales, k_zeros, v_codes, v_scales, B, H, T, D, t_cap, k_bits, k_signed, v_bits,
                     k_out, v_out, out_dtype, true, stream);
}

extern "C" tq_status tq_unrotate(const void* x, tq_dtype dtype, int64_t n_rows, int64_t D, void* out, void* stream) {
  if (n_rows < 0) return TQ_ERR_INVALID_ARG;
  if (!head_dim_ok(D)) return TQ_ERR_HEAD_DIM;
  if (dtype != TQ_F32 && dtype != TQ_BF16) return TQ_ERR_DTYPE;
  if (n_rows > 0x7fffffffLL - (1LL << 24)) return TQ_ERR_INVALID_ARG;  // as in check_common
  if (n_rows == 0) return TQ_OK;
  if (!x || !out) return TQ_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out)) return TQ_ERR_ALIGNMENT;
  UnrotateParams p{};
  p.x = x;
  p.out = out;
  p.rows = static_cast<int>(n_rows);
  p.rot_scale = rotation_scale(D);
  p.err = device_error_word();
  const bool bf16 = dtype == TQ_BF16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (D) {
    case 64: e = launch_unrotate<64>(p, bf16, s); break;
    case 128: e = launch_unrotate<128>(p, bf16, s); break;
    case 256: e = launch_unrotate<256>(p, bf16, s); break;
    default: e = launch_unrotate<512>(p, bf16, s); break;
  }
  return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

extern "C" tq_status tq_lloyd_max_index(const float* u, int64_t n, int v_bits, uint8_t* idx, void* stream) {
  if (n < 0) return TQ_ERR_INVALID_ARG;
  if (!value_bits_ok(v_bits)) return TQ_ERR_BITS;
  if (n == 0) return TQ_OK;
  if (!u || !idx) return TQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(u) & 3u) != 0) return TQ_ERR_ALIGNMENT;
  const long long blocks_needed = (n + 255) / 256;
  const long long cap = static_cast<long long>(sm_count()) * 8;
  const int grid = static_cast<int>(blocks_needed < cap ? blocks_needed : cap);
  lloyd_max_index_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(u, n, v_bits, idx);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

namespace tq {
namespace {

// Partial records of the fused attention: one per split block and head it
// touches, at most kAttnGridPerSm blocks per SM plus one per (batch, kv head).
long long attn_records(long long bhkv) { return static_cast<long long>(kAttnGridPerSm) * sm_count() + bhkv; }

// Workspace of the fused attention: the records, then (when a head can have
// more records than one combine block takes) the combine's partial sums for
// up to 16 * bhkv output rows (kAttnMaxRows query rows per kv head) in row
// tiles of 1024 / D rows, then one ticket counter per row tile.
struct AttnWorkspace {
  long long records_bytes, partial_offset, counter_offset, bytes;
  long long tiles;  // row tiles the partial area and the counters cover
  int chunks;       // the most combine blocks per row tile any call of this size uses
};
AttnWorkspace attn_workspace(long long bhkv, long long D) {
  AttnWorkspace w{};
  w.records_bytes = attn_records(bhkv) * kAttnRecordFloats(D) * 4;
  // a head's records: at most grid / bhkv + 2 (the split grid is at most
  // kAttnGridPerSm blocks per SM)
  w.chunks = attn_combine_chunks(static_cast<long long>(kAttnGridPerSm) * sm_count() / bhkv + 2);
  w.tiles = (kAttnMaxRows * bhkv * D + 1023) / 1024;
  w.partial_offset = w.records_bytes;
  w.counter_offset = w.partial_offset + (w.chunks > 1 ? w.tiles * w.chunks * kCombinePartialFloats * 4 : 0);
  w.bytes = w.counter_offset + (w.chunks > 1 ? (w.tiles * 4 + 15) / 16 * 16 : 0);
  return w;
}

bool attn_head_dim_ok(int64_t d) { return d == 64 || d == 128 || d == 256 || d == 512; }

}  // namespace
}  // namespace tq

extern "C" int64_t tq_decode_attention_workspace_size(int64_t B, int64_t Hkv, int64_t T, int64_t D) {
  if (B < 0 || Hkv < 1 || T < 0 || T > 0x7fffffffLL || B > 0x7fffffffLL || Hkv > 0x7fffffffLL)
    return -static_cast<int64_t>(TQ_ERR_INVALID_ARG);
  if (!attn_head_dim_ok(D)) return -static_cast<int64_t>(TQ_ERR_HEAD_DIM);
  const long long bhkv = B * Hkv;
  if (bhkv > 0x7fffffffLL) return -static_cast<int64_t>(TQ_ERR_INVALID_ARG);
  return static_cast<int64_t>(attn_workspace(bhkv, D).bytes);
}

extern "C" tq_status tq_decode_attention(const void* q, int64_t B, int64_t Hq, int64_t Nq,
                                         const void* k_codes, const void* k_scales, const void* k_zeros,
                                         const void* v_codes, const void* v_scales,
                                         int64_t Hkv, int64_t T, int64_t D, int64_t t_cap,
                                         int k_bits, int k_signed, int v_bits,
                                         const int32_t* left_pad, float scale, void* out, tq_dtype out_dtype,
                                         void* workspace, int64_t workspace_bytes, void* stream) {
  const long long lim = 0x7fffffffLL;
  if (B < 0 || Hq < 1 || Hkv < 1 || Nq < 1 || T < 0 || t_cap < 0) return TQ_ERR_INVALID_ARG;
  if (!attn_head_dim_ok(D)) return TQ_ERR_HEAD_DIM;
  if (key_mode(k_bits, k_signed) < 0 || !value_bits_ok(v_bits)) return TQ_ERR_BITS;
  if (out_dtype != TQ_F32 && out_dtype != TQ_BF16) return TQ_ERR_DTYPE;
  if (Hq % Hkv != 0 || (Hq / Hkv) * Nq > kAttnMaxRows) return TQ_ERR_INVALID_ARG;
  if (T > t_cap || t_cap > lim || B > lim || Hq > lim) return TQ_ERR_INVALID_ARG;
  if (t_cap % 16 != 0) return TQ_ERR_ALIGNMENT;
  if (B > 0 && (Hq > lim / B || Hq * B > lim / Nq || Hkv * B > lim)) return TQ_ERR_INVALID_ARG;
  if (B == 0) return TQ_OK;
  const long long bhkv = B * Hkv;
  if (t_cap > (1LL << 62) / (bhkv * 512)) return TQ_ERR_INVALID_ARG;
  const long long tiles_per_bh = (T + 15) / 16;
  if (bhkv * tiles_per_bh > (1LL << 40)) return TQ_ERR_INVALID_ARG;
  const AttnWorkspace ws = attn_workspace(bhkv, D);
  const long long need = ws.bytes;
  const void* ptrs[] = {q, k_codes, k_scales, k_zeros, v_codes, v_scales, out, workspace};
  for (const void* p : ptrs) {
    if (!p) return TQ_ERR_INVALID_ARG;
    if (!aligned16(p)) return TQ_ERR_ALIGNMENT;
  }
  if ((reinterpret_cast<uintptr_t>(left_pad) & 3u) != 0) return TQ_ERR_ALIGNMENT;
  if (workspace_bytes < need) return TQ_ERR_INVALID_ARG;
  AttnParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.k_codes = static_cast<const uint8_t*>(k_codes);
  p.k_scales = static_cast<const uint16_t*>(k_scales);
  p.k_zeros = static_cast<const uint16_t*>(k_zeros);
  p.v_codes = static_cast<const uint8_t*>(v_codes);
  p.v_scales = static_cast<const uint16_t*>(v_scales);
  p.left_pad = left_pad;
  p.ws = static_cast<float*>(workspace);
  p.out = out;
  p.B = static_cast<int>(B);
  p.Hq = static_cast<int>(Hq);
  p.Hkv = static_cast<int>(Hkv);
  p.G = static_cast<int>(Hq / Hkv);
  p.Nq = static_cast<int>(Nq);
  p.T = static_cast<int>(T);
  p.t_cap = t_cap;
  p.tiles_per_bh = static_cast<int>(tiles_per_bh);
  p.total_tiles = bhkv * tiles_per_bh;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.rot_scale = rotation_scale(D);
  p.cache_rows = bhkv * t_cap;
  p.ws_records = ws.records_bytes / (kAttnRecordFloats(D) * 4);
  p.err = device_error_word();
  p.partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.partial_offset);
  p.counters = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + ws.counter_offset);
  p.chunks = 1;  // the launcher sets it from the split grid (at most ws.chunks)
  p.combine_tiles = static_cast<int>((B * Hq * Nq * D + 1023) / 1024);
  p.vtab_stride = 128;
  p.partial_floats = (ws.counter_offset - ws.partial_offset) / 4;
  const int kmode = key_mode(k_bits, k_signed);
  const bool bf16 = out_dtype == TQ_BF16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (D) {
    case 64: e = launch_attention<64>(p, v_bits, kmode, bf16, s); break;
    case 128: e = launch_attention<128>(p, v_bits, kmode, bf16, s); break;
    case 256: e = launch_attention<256>(p, v_bits, kmode, bf16, s); break;
    default: e = launch_attention<512>(p, v_bits, kmode, bf16, s); break;
  }
  return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

extern "C" tq_status tq_device_status(void* stream) {
  unsigned* err = device_error_word();
  if (err == nullptr) return TQ_ERR_CUDA;
  unsigned v = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return TQ_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return TQ_ERR_CUDA;
    return (v & kErrIndex) ? TQ_ERR_DEVICE_CHECK : TQ_ERR_TIMEOUT;
  }
  return TQ_OK;
}

extern "C" int tq_debug_checks(void) {
#ifdef TQ_DEBUG_CHECKS
  return 1;
#else
  return 0;
#endif
}

extern "C" const char* tq_status_string(int status) {
  switch (status) {
    case TQ_OK: return "TQ_OK";
    case TQ_ERR_INVALID_ARG: return "TQ_ERR_INVALID_ARG: null pointer, negative or inconsistent size";
    case TQ_ERR_HEAD_DIM: return "TQ_ERR_HEAD_DIM: head_dim must be 64, 128, 256 or 512";
    case TQ_ERR_BITS: return "TQ_ERR_BITS: v_bits in {2,3,4,5,8}, k_bits in {2,4,5,8}, signed keys need 8 bits";
    case TQ_ERR_ALIGNMENT: return "TQ_ERR_ALIGNMENT: size not byte-aligned or buffer not 16-byte aligned";
    case TQ_ERR_DTYPE: return "TQ_ERR_DTYPE: dtype must be TQ_F32 or TQ_BF16";
    case TQ_ERR_CUDA: return "TQ_ERR_CUDA: the CUDA runtime reported an error";
    case TQ_ERR_TIMEOUT: return "TQ_ERR_TIMEOUT: a bounded device-side wait gave up";
    case TQ_ERR_DEVICE_CHECK: return "TQ_ERR_DEVICE_CHECK: a debug build's device-side index check failed";
    default: return "unknown tq_status";
  }
}
