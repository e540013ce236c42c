// Device helpers shared by the kernels of libfg (sm_103a).
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace fg {

__device__ __forceinline__ float h2f(uint16_t u) { return __half2float(__ushort_as_half(u)); }
__device__ __forceinline__ uint16_t f2h(float f) { return __half_as_ushort(__float2half_rn(f)); }

// Two floats -> packed half2 bits (lo, hi), round to nearest even.
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_h2(uint32_t u) {
  __half2 h = *reinterpret_cast<__half2*>(&u);
  return __half22float2(h);
}

// Order key of an fp16 bit pattern: unsigned order == numeric order, -0 below +0.
__device__ __forceinline__ uint32_t order_key(uint32_t u) {
  return (u & 0x8000u) ? (0x7FFFu - (u & 0x7FFFu)) : (0x8000u + u);
}
__device__ __forceinline__ uint32_t key_to_bits(uint32_t k) {
  return (k >= 0x8000u) ? (k - 0x8000u) : (0x8000u | (0x7FFFu - k));
}

// Code of one value by the library's binary32 formula: rint((x-a)*15/(b-a)), one
// rounding per operation, ties to even, clamped to [0,15]; 0 for a constant group.
__device__ __forceinline__ uint32_t q4_code(float xf, float af, float bma) {
  if (bma == 0.0f) return 0u;
  float d = __fsub_rn(xf, af);
  float t = __fmul_rn(d, 15.0f);
  float r = __fdiv_rn(t, bma);
  float q = rintf(r);
  q = fminf(fmaxf(q, 0.0f), 15.0f);
  return (uint32_t)q;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

}  // namespace fg
