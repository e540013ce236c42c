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

// The same code with the division replaced, where that cannot change the result, by a
// multiply: y = fl(d * c15) with d = fl(x - a) and c15 = fl(15 * fl(1 / bma)).  Both y and
// fl(q), q = fl(d * 15) / bma, equal 15 d / bma times at most three (y) or two (fl(q))
// factors (1 + e), |e| <= 2^-24; since a <= x <= b makes 0 <= 15 d / bma <= 15 (1 + 2^-24),
// |y - fl(q)| <= 16 * 5 * 2^-24 < 2^-17.  So rint(y) == rint(fl(q)) unless y lies within
// 2^-17 of a half-integer; within 2^-16 of one (or y not a number) `near` is set and the
// caller must take the exact division (q4_code) instead.  rint(y) comes from adding
// 1.5 * 2^23: for 0 <= y < 2^22 the sum's unit in the last place is 1, so round-to-nearest-
// even leaves rint(y) in the low mantissa bits.  Valid for values of the group (a <= x <= b).
// No branch: the callers quantise many values in unrolled code and fix the rare near ties
// afterwards.
__device__ __forceinline__ uint32_t q4_code_fast(float xf, float af, float c15, bool& near) {
  const float y = __fmul_rn(__fsub_rn(xf, af), c15);
  const float t = __fadd_rn(y, 12582912.0f);
  near |= !(fabsf(__fsub_rn(y, __fsub_rn(t, 12582912.0f))) <= 0.5f - 0x1p-16f);
  return __float_as_uint(t) & 0xFu;
}

// ---- one quantisation group of 64 fp16 values, held 8 per thread (or 1 per thread)
// Order keys of the two fp16 values of a word, one per 16-bit lane (order_key on each).
__device__ __forceinline__ uint32_t order_keys2(uint32_t w) {
  const uint32_t neg = (w >> 15) & 0x00010001u;
  return w ^ (0x80008000u | (neg * 0x7FFFu));
}
// Min/max word of 8 fp16 values (four words): min key | (~max key) << 16.  Words of the
// parts of a group merge with __vminu2 (a 16-bit SIMD min of both halves).
__device__ __forceinline__ uint32_t q4_minmax8(const uint32_t (&w)[4]) {
  uint32_t kmin2 = order_keys2(w[0]), kmax2 = kmin2;
#pragma unroll
  for (int i = 1; i < 4; ++i) {
    const uint32_t k2 = order_keys2(w[i]);
    kmin2 = __vminu2(kmin2, k2);
    kmax2 = __vmaxu2(kmax2, k2);
  }
  const uint32_t kmin = min(kmin2 & 0xFFFFu, kmin2 >> 16);
  const uint32_t kmax = max(kmax2 & 0xFFFFu, kmax2 >> 16);
  return kmin | ((~kmax & 0xFFFFu) << 16);
}
// Min/max word of one fp16 value.
__device__ __forceinline__ uint32_t q4_minmax1(uint16_t u) {
  const uint32_t k = order_key(u);
  return k | ((~k & 0xFFFFu) << 16);
}
// The group's statistics word (a | b << 16, fp16 bits) from its merged min/max word.
__device__ __forceinline__ uint32_t q4_ab_word(uint32_t mm) {
  return key_to_bits(mm & 0xFFFFu) | (key_to_bits(~(mm >> 16) & 0xFFFFu) << 16);
}
// The per-group constants of the code formula: a, b - a and fl(15 * fl(1 / (b - a))).
struct Q4Group {
  float af, bma, c15;
};
__device__ __forceinline__ Q4Group q4_group(uint32_t abw) {
  Q4Group g;
  g.af = h2f((uint16_t)(abw & 0xFFFFu));
  g.bma = __fsub_rn(h2f((uint16_t)(abw >> 16)), g.af);
  g.c15 = __fmul_rn(15.0f, __frcp_rn(g.bma));
  return g;
}

// Packed codes of 8 fp16 values against their group: element 2i in the low nibble, 2i+1
// in the high nibble of byte i.  q4_codes8 takes the fast path and sets `near` when a code
// needs the exact division; q4_codes8_exact is that division for all 8 (a called function,
// kept out of the unrolled code that calls it rarely).
__device__ __forceinline__ uint32_t q4_codes8(const uint32_t (&w)[4], const Q4Group& g, bool& near) {
  if (g.bma == 0.0f) return 0u;                   // constant group
  uint32_t codes = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x2 = unpack_h2(w[i]);
    const uint32_t c0 = q4_code_fast(x2.x, g.af, g.c15, near);
    const uint32_t c1 = q4_code_fast(x2.y, g.af, g.c15, near);
    codes |= (c0 | (c1 << 4)) << (8 * i);
  }
  return codes;
}
static __device__ __noinline__ uint32_t q4_codes8_exact(uint4 v, float af, float bma) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t codes = 0;
  for (int i = 0; i < 4; ++i) {
    const float2 x2 = unpack_h2(w[i]);
    codes |= (q4_code(x2.x, af, bma) | (q4_code(x2.y, af, bma) << 4)) << (8 * i);
  }
  return codes;
}
// Fast path, then the exact one when any of the 8 codes is near a tie.
__device__ __forceinline__ uint32_t q4_codes8_checked(const uint32_t (&w)[4], const Q4Group& g) {
  bool near = false;
  const uint32_t c = q4_codes8(w, g, near);
  return near ? q4_codes8_exact(make_uint4(w[0], w[1], w[2], w[3]), g.af, g.bma) : c;
}

// ---- the same fast path two values per instruction (packed binary32 pairs, sm_100 and up):
// sub / mul / add .rn.f32x2 round each lane as the scalar operations do, so y, t and rint(y)
// are the same bits as in q4_code_fast.  The tie test takes the largest |y - rint(y)| of the
// 8 values (max.NaN keeps a NaN, which counts as near, as in q4_code_fast), and the code of a
// value is byte 0 of t = 1.5 * 2^23 + rint(y): one byte permute gathers four of them.
__device__ __forceinline__ uint64_t q4_pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void q4_unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t q4_sub2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t q4_mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t q4_add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float q4_max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint32_t q4_codes8_x2(const uint32_t (&w)[4], const Q4Group& g,
                                                 bool& near) {
  if (g.bma == 0.0f) return 0u;                   // constant group
  const uint64_t a2 = q4_pack2(g.af, g.af), c2 = q4_pack2(g.c15, g.c15);
  const uint64_t k2 = q4_pack2(12582912.0f, 12582912.0f);
  uint32_t tb[8];
  float dmax = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x2 = unpack_h2(w[i]);
    const uint64_t y = q4_mul2(q4_sub2(q4_pack2(x2.x, x2.y), a2), c2);
    const uint64_t t = q4_add2(y, k2);
    float d0, d1, t0, t1;
    q4_unpack2(q4_sub2(y, q4_sub2(t, k2)), d0, d1);
    q4_unpack2(t, t0, t1);
    dmax = q4_max_nan(dmax, q4_max_nan(fabsf(d0), fabsf(d1)));
    tb[2 * i] = __float_as_uint(t0);
    tb[2 * i + 1] = __float_as_uint(t1);
  }
  near |= !(dmax <= 0.5f - 0x1p-16f);
  const uint32_t ev = __byte_perm(__byte_perm(tb[0], tb[2], 0x0040),
                                  __byte_perm(tb[4], tb[6], 0x0040), 0x5410);
  const uint32_t od = __byte_perm(__byte_perm(tb[1], tb[3], 0x0040),
                                  __byte_perm(tb[5], tb[7], 0x0040), 0x5410);
  return (ev & 0x0F0F0F0Fu) | ((od & 0x0F0F0F0Fu) << 4);
}
__device__ __forceinline__ uint32_t q4_codes8_checked_x2(const uint32_t (&w)[4],
                                                         const Q4Group& g) {
  bool near = false;
  const uint32_t c = q4_codes8_x2(w, g, near);
  return near ? q4_codes8_exact(make_uint4(w[0], w[1], w[2], w[3]), g.af, g.bma) : c;
}

// Programmatic dependent launch: every library kernel lets the next kernel of the stream
// launch at once and waits for its predecessor's results (and for its predecessor to have
// finished reading what this kernel overwrites) before touching global data, so launch and
// setup overlap the previous kernel's tail.  Both are no-ops without the launch attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

}  // namespace fg
