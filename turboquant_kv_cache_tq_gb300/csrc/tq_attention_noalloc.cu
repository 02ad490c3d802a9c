// tq_decode_attention_noalloc: the fused decode attention for callers that
// cannot allocate device memory.
//
// Some callers of this library may not call cudaMalloc at all: a plugin
// inside a serving runtime that reserves the whole device memory budget at
// start-up and owns every allocation afterwards, or code on a latency-bound
// path where an allocation (which can synchronize the device) is not
// acceptable. tq_decode_attention needs scratch memory for its per-chunk
// partial results, which such a caller cannot provide. This entry point takes
// that scratch from a fixed array compiled into the library instead, so the
// caller passes only its inputs and outputs.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes: every
// GPU that loads the library holds it until the process exits. Host code
// cannot use the variable's name as a device address (on the host it names a
// stand-in object), so the device address is looked up with
// cudaGetSymbolAddress, once per device, with that device current, the first
// time this entry point runs on it, and cached.
//
// All calls share the array and it keeps whatever the last call left there.
// Nothing in it has to start at zero: the split pass writes every partial
// record it owns in full before the combine pass reads it. Two calls whose
// work overlaps on the GPU (different streams without ordering between them)
// write the same array and race; order such calls on one stream or with
// events.
#include <cstdint>
#include <mutex>

#include "../../include/tq.h"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr long long kNoAllocScratchBytes = TQ_ATTENTION_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch size");

static __device__ __align__(256) unsigned char g_attention_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up on
// the first call per device). Returns null when the lookup fails.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attention_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // leave no sticky error behind for the caller
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace tq

extern "C" tq_status tq_decode_attention_noalloc(const void* q, int64_t B, int64_t Hq, int64_t Nq,
                                                 const void* k_codes, const void* k_scales, const void* k_zeros,
                                                 const void* v_codes, const void* v_scales,
                                                 int64_t Hkv, int64_t T, int64_t D, int64_t t_cap,
                                                 int k_bits, int k_signed, int v_bits,
                                                 const int32_t* left_pad, float scale, void* out,
                                                 tq_dtype out_dtype, void* stream) {
  // An empty batch launches nothing and needs no scratch: the workspace call's
  // own checks and result.
  if (B == 0)
    return tq_decode_attention(q, B, Hq, Nq, k_codes, k_scales, k_zeros, v_codes, v_scales, Hkv, T, D, t_cap,
                               k_bits, k_signed, v_bits, left_pad, scale, out, out_dtype, nullptr, 0, stream);
  const int64_t need = tq_decode_attention_workspace_size(B, Hkv, T, D);
  if (need < 0) return static_cast<tq_status>(-need);
  if (need > tq::kNoAllocScratchBytes) return TQ_ERR_INVALID_ARG;  // beyond the fixed scratch
  void* scratch = tq::scratch_address();
  if (scratch == nullptr) return TQ_ERR_CUDA;
  return tq_decode_attention(q, B, Hq, Nq, k_codes, k_scales, k_zeros, v_codes, v_scales, Hkv, T, D, t_cap,
                             k_bits, k_signed, v_bits, left_pad, scale, out, out_dtype, scratch,
                             tq::kNoAllocScratchBytes, stream);
}
