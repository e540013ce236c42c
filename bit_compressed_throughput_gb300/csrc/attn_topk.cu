// Top-K sparse decode attention over the 4-bit KV cache (sm_103a).
//
// For each sequence b and head hd: the scores of all cached positions t < len come from the
// 4-bit K, the softmax runs over all of them, and only the k positions with the highest
// scores contribute their values:
//   o = sum_{t in top-k} p_t v^_t,   p_t = exp(s_t - max s) / sum_t' exp(s_t' - max s)
// [论文阅读：FlexGen, §3.4 "4-bit 压缩权重和 KV cache": optional sparse attention that loads
// only the top 10% of the value cache; FlexGen paper explainer, §3.3 "Roadmap for the Deep
// Dive": Top-K sparse attention, an approximate method that cuts I/O volume].  Equal scores at
// the k-th place go to the lower position.  The V bytes read fall to k / len of the dense
// kernel's; K is read whole.
//
// Two kernels:
//   topk_scores_kernel  one thread per cached position: its K row (d/2 bytes of codes,
//                       consecutive threads read consecutive rows), per group
//                       s_g * sum_j c_j q_j + a_g * Q_g, scaled to base 2, into the workspace
//   topk_attend_kernel  one warp per (b, hd): the softmax maximum and denominator over all
//                       positions; the k-th largest score as a 32-step bitwise search over
//                       order-preserving keys (the largest key T with #{key >= T} >= k);
//                       the selected positions compacted in position order (keys above T,
//                       then keys equal to T from the lowest position); then the V rows of
//                       the selected positions, eight lanes per row (d/8 channels each),
//                       four rows per step, restored and weighted by p_t.
#include <math.h>

#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {

namespace {

constexpr int kScoreThreads = 128;

// float -> unsigned key with the same order (negative values reversed below the positives)
__device__ __forceinline__ uint32_t order_key_f32(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// exact small integer c (0..15) as a float: 2^23 + c as bits, minus 2^23
__device__ __forceinline__ float nib(uint32_t c) {
  return __uint_as_float(0x4B000000u | c) - 8388608.0f;
}

template <int D>
__global__ void __launch_bounds__(kScoreThreads)
topk_scores_kernel(const uint16_t* __restrict__ q, int64_t q_stride,
                   const uint8_t* __restrict__ kc, const uint32_t* __restrict__ kab, int H,
                   int cap, int len, float scale_log2, float* __restrict__ scores) {
  constexpr int NG = D / 64;
  __shared__ float qs[D];
  __shared__ float Qg[NG];
  pdl_launch_dependents();
  pdl_wait();
  const int bh = blockIdx.x;
  const int b = bh / H, hd = bh - b * H;
  for (int j = threadIdx.x; j < D; j += kScoreThreads)
    qs[j] = h2f(q[(int64_t)b * q_stride + (int64_t)hd * D + j]);
  __syncthreads();
  if (threadIdx.x < NG) {
    float s = 0.0f;
    for (int j = 0; j < 64; ++j) s += qs[threadIdx.x * 64 + j];
    Qg[threadIdx.x] = s;
  }
  __syncthreads();
  const int t = blockIdx.y * kScoreThreads + threadIdx.x;
  if (t >= len) return;
  const int64_t row = (int64_t)bh * cap + t;
  const uint4* cp = reinterpret_cast<const uint4*>(kc + row * (D / 2));
  float acc = 0.0f;
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    float dot = 0.0f;                                 // sum_j c_j q_j over the group
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4 u = ldg_nc_v4(cp + 2 * g + i);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
#pragma unroll
        for (int n = 0; n < 8; ++n)                 // nibble n of word e: channel 8e + n
          dot = fmaf(nib((w[e] >> (4 * n)) & 15u), qs[g * 64 + i * 32 + e * 8 + n], dot);
      }
    }
    const float2 ab = unpack_h2(kab[row * NG + g]);
    acc = fmaf((ab.y - ab.x) * (1.0f / 15.0f), dot, fmaf(ab.x, Qg[g], acc));
  }
  scores[(int64_t)bh * len + t] = acc * scale_log2;
}

template <int D>
__global__ void __launch_bounds__(32)
topk_attend_kernel(const float* __restrict__ scores, const uint8_t* __restrict__ vc,
                   const uint32_t* __restrict__ vab, int H, int cap, int len, int k,
                   uint16_t* __restrict__ out, int32_t* __restrict__ sel_out) {
  constexpr int NG = D / 64;
  constexpr int CPL = D / 8;                          // channels per lane of a row group
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);            // len keys
  int32_t* sel = reinterpret_cast<int32_t*>(smem + (size_t)len * 4);   // k positions
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x;
  const int bh = blockIdx.x;
  const float* sc = scores + (int64_t)bh * len;
  // ---- softmax statistics over all positions (base 2), keys into shared memory
  float m = -INFINITY;
  for (int t = lane; t < len; t += 32) {
    const float s = sc[t];
    keys[t] = order_key_f32(s);
    m = fmaxf(m, s);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  float z = 0.0f;
  for (int t = lane; t < len; t += 32) z += exp2f(sc[t] - m);
#pragma unroll
  for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
  __syncwarp();
  // ---- the k-th largest key: the largest T with #{key >= T} >= k, bit by bit
  uint32_t T = 0u;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t cand = T | (1u << bit);
    int c = 0;
    for (int t = lane; t < len; t += 32) c += (keys[t] >= cand) ? 1 : 0;
    c = __reduce_add_sync(0xFFFFFFFFu, c);
    if (c >= k) T = cand;
  }
  int above = 0;
  for (int t = lane; t < len; t += 32) above += (keys[t] > T) ? 1 : 0;
  above = __reduce_add_sync(0xFFFFFFFFu, above);
  const int eq_take = k - above;                      // >= 1 by the choice of T
  // ---- compaction in position order: every key above T, the first eq_take keys equal to T
  int n_sel = 0, n_eq = 0;
  for (int base = 0; base < len; base += 32) {
    const int t = base + lane;
    const uint32_t key = (t < len) ? keys[t] : 0u;
    const bool gt = t < len && key > T, eq = t < len && key == T;
    const uint32_t eqm = __ballot_sync(0xFFFFFFFFu, eq);
    const uint32_t below = (1u << lane) - 1u;
    const bool take = gt || (eq && n_eq + __popc(eqm & below) < eq_take);
    const uint32_t tm = __ballot_sync(0xFFFFFFFFu, take);
    if (take) sel[n_sel + __popc(tm & below)] = t;
    n_sel += __popc(tm);
    n_eq += __popc(eqm);
  }
  __syncwarp();
  if (sel_out)
    for (int i = lane; i < k; i += 32) sel_out[(int64_t)bh * k + i] = sel[i];
  // ---- values of the selected positions: lanes 8r..8r+7 take one row, CPL channels each
  const int pg = lane >> 3, cl = lane & 7;
  const int g = (cl * CPL) / 64;                      // the group of this lane's channels
  const float inv_z = 1.0f / z;
  float acc[CPL];
#pragma unroll
  for (int j = 0; j < CPL; ++j) acc[j] = 0.0f;
  const int64_t head_row0 = (int64_t)bh * cap;
#pragma unroll 4
  for (int i = pg; i < k; i += 4) {
    const int t = sel[i];
    const int64_t row = head_row0 + t;
    const float p = exp2f(sc[t] - m) * inv_z;
    const float2 ab = unpack_h2(vab[row * NG + g]);
    const float s = (ab.y - ab.x) * (1.0f / 15.0f);
    const uint8_t* vp = vc + row * (D / 2) + cl * (CPL / 2);
    uint32_t w[CPL / 8];
    if constexpr (CPL == 16) {
      const uint2 u = *reinterpret_cast<const uint2*>(vp);
      w[0] = u.x;
      w[(CPL / 8) - 1] = u.y;
    } else {
      w[0] = *reinterpret_cast<const uint32_t*>(vp);
    }
#pragma unroll
    for (int e = 0; e < CPL / 8; ++e)
#pragma unroll
      for (int n = 0; n < 8; ++n)
        acc[8 * e + n] = fmaf(p, fmaf(nib((w[e] >> (4 * n)) & 15u), s, ab.x), acc[8 * e + n]);
  }
  // ---- sum the four row groups (lanes cl, cl + 8, cl + 16, cl + 24) and store
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    acc[j] += __shfl_xor_sync(0xFFFFFFFFu, acc[j], 8);
    acc[j] += __shfl_xor_sync(0xFFFFFFFFu, acc[j], 16);
  }
  if (pg == 0) {
    uint16_t* o = out + (int64_t)bh * D + cl * CPL;
#pragma unroll
    for (int j = 0; j < CPL; j += 8) {
      uint4 v;
      v.x = pack_h2(acc[j], acc[j + 1]);
      v.y = pack_h2(acc[j + 2], acc[j + 3]);
      v.z = pack_h2(acc[j + 4], acc[j + 5]);
      v.w = pack_h2(acc[j + 6], acc[j + 7]);
      *reinterpret_cast<uint4*>(o + j) = v;
    }
  }
}

template <int D>
cudaError_t launch_topk_d(const uint16_t* q, int64_t q_stride, const fg_kvcache& kv, int32_t len,
                          int32_t k, float scale, uint16_t* out, int32_t* sel, float* ws,
                          cudaStream_t st) {
  const int64_t nbh = (int64_t)kv.B * kv.H;
  const float sl2 = scale * 1.4426950408889634f;
  const dim3 g1((unsigned)nbh, (unsigned)((len + kScoreThreads - 1) / kScoreThreads));
  cudaError_t e = launch_pdl(topk_scores_kernel<D>, g1, dim3(kScoreThreads), 0, st, q, q_stride,
                             kv.k_codes, reinterpret_cast<const uint32_t*>(kv.k_ab), kv.H,
                             kv.cap, len, sl2, ws);
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)len * 4 + (size_t)k * 4;
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(topk_attend_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(topk_attend_kernel<D>, dim3((unsigned)nbh), dim3(32), smem, st,
                    static_cast<const float*>(ws), kv.v_codes,
                    reinterpret_cast<const uint32_t*>(kv.v_ab), kv.H, kv.cap, len, k, out, sel);
}

}  // namespace

size_t decode_attn_topk_ws_bytes(const fg_kvcache& kv, int32_t len) {
  return (size_t)kv.B * kv.H * (size_t)len * sizeof(float);
}

cudaError_t launch_decode_attn_topk(const uint16_t* q, int64_t q_stride, const fg_kvcache& kv,
                                    int32_t len, int32_t k, float scale, uint16_t* out,
                                    int32_t* sel, void* ws, cudaStream_t st) {
  if ((int64_t)kv.B * kv.H >= (1ll << 31)) return cudaErrorInvalidValue;
  float* w = static_cast<float*>(ws);
  const int d = kv.h / kv.H;
  return (d == 128) ? launch_topk_d<128>(q, q_stride, kv, len, k, scale, out, sel, w, st)
                    : launch_topk_d<64>(q, q_stride, kv, len, k, scale, out, sel, w, st);
}

}  // namespace fg
