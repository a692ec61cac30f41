// fa_decode_noalloc.cu -- fa_decode_fwd_noalloc: the single-token decode with
// its split-KV partials kept in one fixed, file-scope device array instead of
// memory allocated on every call.
//
// Who needs it: callers that must not allocate device memory while they run
// attention.  Examples: a serving loop whose memory is reserved once at start-up
// under a hard budget, code that runs while an allocator lock is held (a
// cudaMallocAsync from there can deadlock or re-enter the caller's allocator),
// and embedded runtimes that forbid allocation after initialisation.  This entry
// point touches only the caller's tensors and the array below.
//
// Limits and sharing:
// - The array holds kNoAllocScratchFloats fp32 values (4 MiB).  Every GPU that
//   loads the library keeps it for the life of the process.  A request whose
//   partials do not fit is rejected with FA_ERR_TOO_LARGE before any work is
//   enqueued.
// - All calls on a device share the one array.  Calls whose kernels overlap on
//   the GPU (e.g. issued on two streams without ordering between them) race on
//   it and give wrong results; calls ordered on one stream are safe.
// - Nothing in the array has to start at zero: every call overwrites every
//   partial it later reads, so the contents left by the previous call are never
//   used.
// - Set-up: the first call on each device looks up the array's device address
//   with cudaGetSymbolAddress while that device is current (the host-side name
//   of the array is only a stand-in, never a device address).  Make that first
//   call before any stream capture on the device.
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr size_t kNoAllocScratchFloats = size_t(1) << 20;  // 4 MiB of fp32 partials
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

// Device address of g_noalloc_scratch on the current device, looked up once per
// device.  Returns nullptr and sets *err on failure.
float* scratch_for_current_device(cudaError_t* err) {
  static std::mutex mu;
  static float* addr[kMaxDevices] = {nullptr};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *err = e;
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      *err = (e != cudaSuccess) ? e : cudaErrorInvalidSymbol;
      return nullptr;
    }
    addr[dev] = static_cast<float*>(p);
  }
  return addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int fa_decode_fwd_noalloc(const void* q, const void* kcache, const void* vcache,
                                     const int32_t* valid_len_dev, void* o, int B, int Hq,
                                     int Hkv, int cap, int D, float scale,
                                     cudaStream_t stream) {
  // Same argument rules as fa_decode_fwd.
  if (B < 0 || Hq < 0 || Hkv < 0 || cap < 0) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_INVALID_ARG;
  if (!isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (B == 0 || Hq == 0) return FA_OK;
  if (Hkv == 0 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (B > 65535 || Hq > 65535 || (int64_t)Hkv * ((Hq / Hkv + 15) / 16) > 65535)
    return FA_ERR_INVALID_ARG;
  if (!q || !o || !aligned16(q) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (cap > 0 && (!kcache || !vcache || !valid_len_dev || !aligned16(kcache) ||
                  !aligned16(vcache) || (reinterpret_cast<uintptr_t>(valid_len_dev) & 3u)))
    return FA_ERR_INVALID_ARG;
  if ((int64_t)cap * Hkv * D * 2 >= (1ll << 40)) return FA_ERR_INVALID_ARG;
  if (cap == 0) {
    // No cache: O = 0, no partials needed.
    return fa::record_cuda_status(fa::launch_decode(q, kcache, vcache, valid_len_dev, o, nullptr,
                                                    B, Hq, Hkv, 0, D, scale, nullptr, 0, stream),
                                  "decode_noalloc zero-fill launch");
  }
  const size_t need = fa::decode_scratch_floats(B, Hq, Hkv, cap, D);
  if (need > kNoAllocScratchFloats) return FA_ERR_TOO_LARGE;
  cudaError_t err = cudaSuccess;
  float* scratch = scratch_for_current_device(&err);
  if (!scratch) return fa::record_cuda_status(err, "decode_noalloc cudaGetSymbolAddress");
  return fa::record_cuda_status(fa::launch_decode(q, kcache, vcache, valid_len_dev, o, nullptr,
                                                  B, Hq, Hkv, cap, D, scale, scratch,
                                                  kNoAllocScratchFloats, stream),
                                "decode_noalloc launch");
}
