// Group-wise 4-bit quantisation, restoration and KV-cache append (sm_103a).
//
// FlexGen stores weights and the KV cache as 4-bit codes in groups of 64 (weights along
// the output channel, K/V along the hidden dimension) with the group min a and max b,
// and restores FP16 values before compute [FlexGen review (jaehun.me), section
// "4-bit 압축은 정수 연산 가속과 같은가", restating paper §5].  The code formula is the
// library's binary32 reading documented in include/fg.h.
//
// Work split: 8 threads per group of 64, each owning 8 consecutive values (one 16-byte
// load, one 4-byte code store); the group min/max is a 3-step xor shuffle inside the
// 8-lane segment.  These kernels are HBM-bound: 2 bytes read and 0.5625 bytes written
// per element.
#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {

namespace {

constexpr int kThreads = 256;                 // 32 groups per CTA
constexpr int kGroupsPerCta = kThreads / 8;

// Quantise the 8 values held by this thread (part of a 64-group spread over 8 lanes).
// Returns the packed codes; *ab_out receives the group's statistics word.  The group min
// and max travel as one word (min key | ~max key << 16) reduced with a 16-bit SIMD min.
__device__ __forceinline__ uint32_t quantize8(const uint4 v, uint32_t* ab_out) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t mm = q4_minmax8(w);
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) mm = __vminu2(mm, __shfl_xor_sync(0xFFFFFFFFu, mm, o));
  *ab_out = q4_ab_word(mm);
  return q4_codes8_checked_x2(w, q4_group(*ab_out));
}

__global__ void __launch_bounds__(kThreads)
quantize_kernel(const uint16_t* __restrict__ x, int64_t ngroups, uint8_t* __restrict__ codes,
                uint32_t* __restrict__ ab) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t grp = (int64_t)blockIdx.x * kGroupsPerCta + (threadIdx.x >> 3);
  const int sub = threadIdx.x & 7;
  // Every lane of a warp takes part in the shuffles; lanes past the end use a dummy.
  const bool live = grp < ngroups;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (live) v = ldg_nc_v4(x + grp * 64 + sub * 8);
  uint32_t abw;
  const uint32_t c = quantize8(v, &abw);
  if (live) {
    reinterpret_cast<uint32_t*>(codes)[grp * 8 + sub] = c;
    if (sub == 0) ab[grp] = abw;
  }
}

// One CTA covers a block of positions of one (sequence b, head) of K or V (blockIdx.z):
// thread = (position, group of the head, 8-value slice), kPosPerThread positions apart,
// whose loads are all issued before any is used so that enough bytes are in flight per SM.
// The codes of the block's positions are then contiguous runs of the head-major cache
// (d/2 bytes per position) and so are their (a, b) words, so the writes coalesce; the
// reads are the head's d values of each source row.  Row r = b*T + t lives at r*row_stride.
constexpr int kPosPerThread = 4;
__global__ void __launch_bounds__(kThreads)
kv_append_kernel(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                 int64_t row_stride, int T, int pos, int H, int d, int cap, int ppc,
                 uint8_t* __restrict__ k_codes, uint8_t* __restrict__ v_codes,
                 uint32_t* __restrict__ k_ab, uint32_t* __restrict__ v_ab) {
  pdl_launch_dependents();
  pdl_wait();
  const int gph = d >> 6;                            // groups per head (1 or 2)
  const int b = blockIdx.x / H, head = blockIdx.x - b * H;
  const int p0 = threadIdx.x / (8 * gph);            // first position within the block
  const int pstep = kThreads / (8 * gph);            // ppc / kPosPerThread
  const int gs = (threadIdx.x >> 3) % gph, sub = threadIdx.x & 7;
  const uint16_t* src = blockIdx.z ? v_new : k_new;
  uint8_t* cdst = blockIdx.z ? v_codes : k_codes;
  uint32_t* adst = blockIdx.z ? v_ab : k_ab;
  uint4 v[kPosPerThread];
#pragma unroll
  for (int i = 0; i < kPosPerThread; ++i) {
    const int t = blockIdx.y * ppc + p0 + i * pstep;
    v[i] = make_uint4(0, 0, 0, 0);
    if (t < T)
      v[i] = ldg_nc_v4(src + ((int64_t)b * T + t) * row_stride + head * d + gs * 64 + sub * 8);
  }
#pragma unroll
  for (int i = 0; i < kPosPerThread; ++i) {
    const int t = blockIdx.y * ppc + p0 + i * pstep;
    // every lane of a warp takes part in the shuffles; positions past the end use a dummy
    uint32_t abw;
    const uint32_t c = quantize8(v[i], &abw);
    if (t < T) {
      const int64_t slot = ((int64_t)b * H + head) * cap + pos + t;
      reinterpret_cast<uint32_t*>(cdst + slot * (d >> 1) + gs * 32)[sub] = c;
      if (sub == 0) adst[slot * gph + gs] = abw;
    }
  }
}

// Short appends (decode: a few positions per sequence): 8 threads per group over the
// groups of the new rows (b, t) in row order, so every thread has work.
__global__ void __launch_bounds__(kThreads)
kv_append_rows_kernel(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                      int64_t row_stride, int T, int pos, int H, int d, int cap, int gpr,
                      int64_t ngroups, uint8_t* __restrict__ k_codes,
                      uint8_t* __restrict__ v_codes, uint32_t* __restrict__ k_ab,
                      uint32_t* __restrict__ v_ab) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t grp = (int64_t)blockIdx.x * kGroupsPerCta + (threadIdx.x >> 3);
  const int sub = threadIdx.x & 7;
  const bool live = grp < ngroups;
  const uint16_t* src = blockIdx.y ? v_new : k_new;
  int64_t row = 0;
  int gi = 0;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (live) {
    row = grp / gpr;
    gi = (int)(grp - row * gpr);
    v = ldg_nc_v4(src + row * row_stride + (int64_t)gi * 64 + sub * 8);
  }
  uint32_t abw;
  const uint32_t c = quantize8(v, &abw);
  if (live) {
    const int gph = d >> 6;
    const int64_t b = row / T;
    const int t = (int)(row - b * T);
    const int head = gi / gph, gs = gi - head * gph;
    const int64_t slot = ((b * H + head) * (int64_t)cap + pos + t);
    uint8_t* cdst = blockIdx.y ? v_codes : k_codes;
    uint32_t* adst = blockIdx.y ? v_ab : k_ab;
    reinterpret_cast<uint32_t*>(cdst + slot * (d >> 1) + gs * 32)[sub] = c;
    if (sub == 0) adst[slot * gph + gs] = abw;
  }
}

// Standalone restoration: fp16(a + q * ((b - a) / 15)), one rounding per binary32 op.
// kPerm: each run of 8 channels is stored in the order 0,4,1,5,2,6,3,7 (the order in which
// the CTA-pair GEMM's restore writes its A tiles, so that the GEMM can load them instead).
template <bool kPerm>
__global__ void __launch_bounds__(kThreads)
dequant_kernel(const uint8_t* __restrict__ codes, const uint32_t* __restrict__ ab,
               int64_t ngroups, uint16_t* __restrict__ y) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t grp = (int64_t)blockIdx.x * kGroupsPerCta + (threadIdx.x >> 3);
  const int sub = threadIdx.x & 7;
  if (grp >= ngroups) return;
  const uint32_t c = reinterpret_cast<const uint32_t*>(codes)[grp * 8 + sub];
  const uint32_t abw = ab[grp];
  const float af = h2f((uint16_t)(abw & 0xFFFFu)), bf = h2f((uint16_t)(abw >> 16));
  const float s = __fdiv_rn(__fsub_rn(bf, af), 15.0f);
  uint16_t xh[8];
#pragma unroll
  for (int n = 0; n < 8; ++n)
    xh[n] = f2h(__fadd_rn(af, __fmul_rn((float)((c >> (4 * n)) & 0xF), s)));
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = kPerm ? ((uint32_t)xh[i] | ((uint32_t)xh[i + 4] << 16))
                 : ((uint32_t)xh[2 * i] | ((uint32_t)xh[2 * i + 1] << 16));
  reinterpret_cast<uint4*>(y + grp * 64)[sub] = make_uint4(o[0], o[1], o[2], o[3]);
}

inline unsigned grid_for(int64_t ngroups) {
  return (unsigned)((ngroups + kGroupsPerCta - 1) / kGroupsPerCta);
}

}  // namespace

cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* codes,
                            uint32_t* ab, cudaStream_t st) {
  const int64_t ng = rows * (cols / 64);
  if (ng == 0) return cudaSuccess;
  return launch_pdl(quantize_kernel, dim3(grid_for(ng)), dim3(kThreads), 0, st, x, ng, codes, ab);
}

cudaError_t launch_dequant(const uint8_t* codes, const uint32_t* ab, int64_t rows, int64_t cols,
                           uint16_t* y, cudaStream_t st) {
  const int64_t ng = rows * (cols / 64);
  if (ng == 0) return cudaSuccess;
  return launch_pdl(dequant_kernel<false>, dim3(grid_for(ng)), dim3(kThreads), 0, st, codes, ab,
                    ng, y);
}

cudaError_t launch_dequant_pairperm(const uint8_t* codes, const uint32_t* ab, int64_t rows,
                                    int64_t cols, uint16_t* y, cudaStream_t st) {
  const int64_t ng = rows * (cols / 64);
  if (ng == 0) return cudaSuccess;
  return launch_pdl(dequant_kernel<true>, dim3(grid_for(ng)), dim3(kThreads), 0, st, codes, ab,
                    ng, y);
}

cudaError_t launch_kv_append(const uint16_t* k_new, const uint16_t* v_new, int64_t row_stride,
                             int32_t T, int32_t pos, const fg_kvcache& kv, cudaStream_t st) {
  if ((int64_t)kv.B * T == 0) return cudaSuccess;
  const int d = kv.h / kv.H;
  if (T < 8) {
    const int gpr = kv.h / 64;
    const int64_t ng = (int64_t)kv.B * T * gpr;
    dim3 grid(grid_for(ng), 2);
    return launch_pdl(kv_append_rows_kernel, grid, dim3(kThreads), 0, st, k_new, v_new, row_stride,
                      T, pos, kv.H, d, kv.cap, gpr, ng, kv.k_codes, kv.v_codes, kv.k_ab, kv.v_ab);
  }
  const int ppc = kPosPerThread * kThreads / (8 * (d / 64));   // 64 (d = 128) or 128
  const int64_t tblocks = (T + ppc - 1) / ppc;
  if (tblocks > 65535 || (int64_t)kv.B * kv.H > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)(kv.B * kv.H), (unsigned)tblocks, 2);
  return launch_pdl(kv_append_kernel, grid, dim3(kThreads), 0, st, k_new, v_new, row_stride, T, pos,
                    kv.H, d, kv.cap, ppc, kv.k_codes, kv.v_codes, kv.k_ab, kv.v_ab);
}

}  // namespace fg
