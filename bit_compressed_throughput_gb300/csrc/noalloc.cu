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
// variable, is held on every GPU that loads the library until the process exits.  A call
// is rejected (FG_ERR_WORKSPACE, nothing launched) when fg_decode_attn_workspace_bytes --
// the split scratch planned for up to 192 SMs, never less than the current device's plan
// needs -- exceeds the array.  Its device address is looked up once per device, with that
// device current, on the first call made on that device, so make that first call before
// any stream capture.  All calls share the one array: two calls that overlap on the GPU
// (different streams, or other host threads) race on it.  Every byte a call reads is
// written earlier by the same call, so nothing has to start at zero and the contents
// left by the previous call do not matter.
#include <mutex>
#include <string>

#include "fg_internal.h"

namespace fg {
namespace {

constexpr size_t kScratchFloats = FG_DECODE_ATTN_STATIC_SCRATCH_BYTES / sizeof(float);
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

std::mutex g_mu;
void* g_scratch_ptr[64];   // device address of g_decode_scratch, per device (null: not yet)

// The array's device address on the current device, looked up once per device.  Host code
// must not pass g_decode_scratch itself to a kernel: in host code that name is a host-side
// stand-in, not a device address.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return FG_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return FG_ERR_ARCH;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) {
      set_last_error(std::string("cudaGetSymbolAddress of the static scratch failed: ") +
                     cudaGetErrorString(e));
      return FG_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FG_OK;
}

}  // namespace
}  // namespace fg

using namespace fg;

extern "C" int fg_decode_attn_q4kv_static(const uint16_t* q, int64_t q_stride,
                                          const fg_kvcache* kv, int32_t len, float scale,
                                          uint16_t* out, void* stream) {
  bool noop = false;
  int rc = check_decode_attn(q, q_stride, kv, len, scale, out, &noop);
  if (rc || noop) return rc;
  const size_t need = fg_decode_attn_workspace_bytes(kv, len);
  if (need > FG_DECODE_ATTN_STATIC_SCRATCH_BYTES) {
    set_last_error("fg_decode_attn_q4kv_static: this call needs " + std::to_string(need) +
                   " bytes of split scratch (fg_decode_attn_workspace_bytes), more than the "
                   "static " + std::to_string((size_t)FG_DECODE_ATTN_STATIC_SCRATCH_BYTES) +
                   " bytes; use fg_decode_attn_q4kv with a caller workspace");
    return FG_ERR_WORKSPACE;
  }
  int sms = 0;
  if ((rc = check_device(&sms))) return rc;
  void* scratch = nullptr;
  if ((rc = scratch_address(&scratch))) return rc;
  return run_decode_attn(q, q_stride, *kv, len, scale, out, scratch, sms,
                         static_cast<cudaStream_t>(stream));
}
