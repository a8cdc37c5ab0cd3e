// Split-KV decode that allocates nothing: the split partials live in a fixed,
// file-scope device array instead of caller-provided scratch.
//
// Who needs this: callers that may not allocate GPU memory at the point where they
// run decode -- for example a serving loop with a fixed memory budget that forbids
// allocation after warm-up, code running under another framework's allocator that
// hands out only the tensors it owns, or a plain C caller with no allocator of its
// own.  cudaMalloc would also synchronise the device in the middle of a latency-
// critical decode step.  Such callers pass only the inputs and the output; the
// scratch comes from here.
//
// The array is part of the loaded module, so every GPU that loads this library
// holds kScratchBytes of device memory until the process exits.
#include <mutex>

#include "sl8_internal.h"

namespace sl8 {
namespace {

constexpr size_t kScratchBytes = SL8_NOALLOC_SCRATCH_BYTES;
constexpr size_t kScratchFloats = kScratchBytes / sizeof(float);

// The scratch itself.  In host code this name is only a stand-in for the symbol,
// not a device address: the address is looked up per device below.
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device
// (with that device current).  Returns nullptr if the lookup fails.
float* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    float* ptr = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace sl8

using namespace sl8;

extern "C" int sl8_attn_int8_decode_noalloc(const void* q, int q_dtype, const int8_t* k_cache, const float* k_scale,
                                            const int8_t* v_cache, const float* v_scale, const int32_t* seqlens,
                                            int32_t B, int32_t Hq, int32_t Hkv, int32_t Lmax, int32_t d, void* out,
                                            int out_dtype, void* stream) {
  if (!q || !k_cache || !k_scale || !v_cache || !v_scale || !seqlens || !out) return SL8_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) &
      15u)
    return SL8_ERR_INVALID_ARG;
  if (q_dtype != SL8_F16 && q_dtype != SL8_BF16 && q_dtype != SL8_F32) return SL8_ERR_INVALID_ARG;
  if (out_dtype != SL8_F16 && out_dtype != SL8_BF16 && out_dtype != SL8_F32) return SL8_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Lmax < 0 || Hq % Hkv != 0) return SL8_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return SL8_ERR_UNSUPPORTED;
  if (Hq / Hkv > 8 || B > 65535 || Hkv > 65535) return SL8_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * Hkv * Lmax >= (int64_t(1) << 31)) return SL8_ERR_UNSUPPORTED;
  if (B == 0 || Lmax == 0) return SL8_OK;

  // Partials per split: [B][Hq][d] fp32 O and [B][Hq] fp32 lse.  Use the automatic split
  // count, lowered to what the fixed scratch holds; refuse if one split does not fit.
  const size_t per_split = static_cast<size_t>(B) * Hq * (static_cast<size_t>(d) + 1);
  if (per_split > kScratchFloats) return SL8_ERR_WORKSPACE;
  int32_t S = sl8_attn_decode_num_splits(B, Hkv, Lmax, d, 0);
  const size_t fit = kScratchFloats / per_split;
  if (static_cast<size_t>(S) > fit) S = static_cast<int32_t>(fit);

  float* scratch = scratch_on_current_device();
  if (!scratch) return SL8_ERR_CUDA;
  // Nothing here needs to start at zero: the split kernel writes the lse of every split and
  // the O of every non-empty split before the combine reads them, and the combine reads no
  // other slot.
  float* o_partial = scratch;
  float* lse_partial = scratch + static_cast<size_t>(B) * Hq * S * d;

  DecodeArgs a{};
  a.q = q;
  a.q_dtype = static_cast<sl8_dtype>(q_dtype);
  a.k_cache = k_cache;
  a.k_scale = k_scale;
  a.v_cache = v_cache;
  a.v_scale = v_scale;
  a.seqlens = seqlens;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Lmax = Lmax;
  a.d = d;
  a.num_splits = sl8_attn_decode_num_splits(B, Hkv, Lmax, d, S);  // <= S: fits the array
  a.split_size = sl8_attn_decode_split_size(B, Hkv, Lmax, d, S);
  a.kv_groups = 1;
  a.o_partial = o_partial;
  a.lse_partial = lse_partial;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_decode_split(a, s) != cudaSuccess) return SL8_ERR_CUDA;
  if (launch_decode_combine(o_partial, lse_partial, seqlens, B, Hq, d, a.num_splits, a.split_size, out,
                            static_cast<sl8_dtype>(out_dtype), nullptr, s) != cudaSuccess)
    return SL8_ERR_CUDA;
  return SL8_OK;
}
