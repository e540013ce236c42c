// Decode attention with library-owned scratch, for callers that cannot allocate device
// memory.
//
// fg_decode_attn_q4kv takes its split-sequence scratch from the caller.  Some callers
// have no way to provide it: code that runs where cudaMalloc is off limits (inside a
// region that must not allocate, under an external allocator that owns all device memory,
// or in a host runtime that only passes existing buffers through).  This entry point runs
// the same kernels with the scratch taken from a fixed array in device global memory
// that the library defines statically, so the call itself allocates nothing.
//
// The array is FG_DECODE_ATTN_STATIC_SCRATCH_BYTES (4 MiB) and, like any static device
// variable, is held on every GPU that loads the library until the process exits.  Its
// device address is looked up once per device, with that device current, on the first
// call made on that device.  All calls share the one array: two calls that overlap on the
// GPU (different streams, or other host threads) race on it.  Every byte a call reads is
// written earlier by the same call, so nothing has to start at zero and the contents
// left by the previous call do not matter.
#include <mutex>
#include <string>

#include "fg_internal.h"

namespace fg {
namespace {

constexpr size_t kScratchFloats = FG_DECODE_ATTN_STATIC_SCRATCH_BYTES / sizeof(float);
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

struct DeviceScratch {
  bool ready = false;
  void* ptr = nullptr;   // device address of g_decode_scratch on this device
  int sms = 0;
};
std::mutex g_mu;
DeviceScratch g_dev[64];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Looks up the array's device address and the SM count for the current device, once.
int setup_current_device(DeviceScratch** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return FG_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return FG_ERR_ARCH;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceScratch& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
      set_last_error(cudaGetErrorString(e));
      return FG_ERR_CUDA;
    }
    if (major != 10 || minor != 3) {
      set_last_error("libfg is built for sm_103a (GB300); the current device is not compute 10.3");
      return FG_ERR_ARCH;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) {
      set_last_error(std::string("cudaGetSymbolAddress of the static scratch failed: ") +
                     cudaGetErrorString(e));
      return FG_ERR_CUDA;
    }
    d.ptr = p;
    d.sms = sms < kMaxSms ? sms : kMaxSms;   // the SM bound the workspace queries plan with
    d.ready = true;
  }
  *out = &d;
  return FG_OK;
}

}  // namespace
}  // namespace fg

using namespace fg;

extern "C" int fg_decode_attn_q4kv_static(const uint16_t* q, int64_t q_stride,
                                          const fg_kvcache* kv, int32_t len, float scale,
                                          uint16_t* out, void* stream) {
  if (!kv || !kv->k_codes || !kv->v_codes || !kv->k_ab || !kv->v_ab) return FG_ERR_ARG;
  if (!aligned16(kv->k_codes) || !aligned16(kv->v_codes) || !aligned16(kv->k_ab) ||
      !aligned16(kv->v_ab))
    return FG_ERR_ARG;
  if (kv->B < 0 || kv->cap <= 0 || kv->cap % 16 != 0 || kv->h <= 0 || kv->H <= 0 ||
      kv->h % 64 != 0 || kv->h % kv->H != 0)
    return FG_ERR_SHAPE;
  const int d = kv->h / kv->H;
  if (d != 64 && d != 128) return FG_ERR_SHAPE;
  if (len <= 0) return FG_ERR_SHAPE;
  if (len > kv->cap) return FG_ERR_CAPACITY;
  if (q_stride < kv->h || q_stride % 8 != 0) return FG_ERR_SHAPE;
  if (!(scale > 0.0f) || !isfinite(scale)) return FG_ERR_ARG;
  if (kv->B == 0) return FG_OK;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return FG_ERR_ARG;
  DeviceScratch* ds = nullptr;
  int rc = setup_current_device(&ds);
  if (rc) return rc;
  const size_t need = decode_attn_ws_bytes(*kv, len, ds->sms);
  if (need > FG_DECODE_ATTN_STATIC_SCRATCH_BYTES) {
    set_last_error("fg_decode_attn_q4kv_static: this call needs " + std::to_string(need) +
                   " bytes of split scratch, more than the static " +
                   std::to_string((size_t)FG_DECODE_ATTN_STATIC_SCRATCH_BYTES) +
                   " bytes; use fg_decode_attn_q4kv with a caller workspace");
    return FG_ERR_WORKSPACE;
  }
  int nk = 0;
  cudaError_t e = launch_decode_attn(q, q_stride, *kv, len, scale, out, ds->ptr, ds->sms,
                                     static_cast<cudaStream_t>(stream), &nk, nullptr);
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return FG_ERR_CUDA;
  }
  return FG_OK;
}
