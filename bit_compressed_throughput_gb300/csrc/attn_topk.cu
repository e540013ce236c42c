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
//   scores   the dense decode kernel's scores-only instance (attn_decode.cu): K streamed
//            through its shared-memory ring, the scores on the tensor cores in base 2, each
//            written as an order-preserving key, and each work item's online-softmax state
//            (reference maximum m, sum l) kept for the denominator
//   topk_attend_kernel  one warp per (b, hd), no barriers (29 independent warps per SM,
//                       which this latency-bound work needs): the softmax denominator from
//                       the work items'
//                       (m, l); the keys once into shared memory; the k-th largest key by
//                       radix selection, eight bits per round from the top (a 256-bin
//                       histogram of the keys that share the bits found so far, then the bin
//                       holding the remaining rank); the selected positions compacted in
//                       position order (keys above T, then keys equal to T from the lowest
//                       position); then the V rows of the selected positions gathered 16 at a
//                       time into the dense kernel's tensor-core tile (weights 2^(s - M), the
//                       softmax denominator applied at the end).
#include <math.h>

#include "attn_q4.cuh"
#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {

namespace {

using q4attn::key_to_f32;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// sum over the lanes that share tig (the eight row owners of a tile)
__device__ __forceinline__ float warp_sum_gid(float v) {
  v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
  v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
  v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
  return v;
}

template <int D>
__global__ void __launch_bounds__(32)
topk_attend_kernel(const uint32_t* __restrict__ keys_g, const float2* __restrict__ ml,
                   int splits, const uint8_t* __restrict__ vc, const uint32_t* __restrict__ vab,
                   int H, int cap, int len, int k, uint16_t* __restrict__ out,
                   int32_t* __restrict__ sel_out) {
  constexpr int NW = D / 32, NG = D / 64;
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem);            // 256 radix counters
  uint32_t* keys = hist + 256;                                   // len keys
  int32_t* sel = reinterpret_cast<int32_t*>(keys + len);         // k positions
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x;
  const int bh = blockIdx.x;
  // ---- the softmax denominator from the work items' states: M = max m_s,
  // z = sum_s l_s 2^(m_s - M) (splits <= 16 < 32 lanes; every item saw a valid position)
  const float2 st = (lane < splits) ? ml[(int64_t)bh * splits + lane] : make_float2(-INFINITY, 0.0f);
  float m = st.x;
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  const float z = warp_sum((lane < splits) ? st.y * exp2f(st.x - m) : 0.0f);
  // ---- the keys once into shared memory
  const uint32_t* kg = keys_g + (int64_t)bh * len;
  for (int t = lane; t < len; t += 32) keys[t] = kg[t];
  __syncwarp();
  // ---- the k-th largest key, eight bits per round from the top: a histogram of the keys
  // that share the bits found so far, then the bin that holds the remaining rank
  uint32_t prefix = 0u, pmask = 0u;
  int rank = k;                                       // wanted rank among the matching keys
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
#pragma unroll
    for (int i = 0; i < 8; ++i) hist[lane * 8 + i] = 0u;
    __syncwarp();
    for (int t = lane; t < len; t += 32) {
      const uint32_t key = keys[t];
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncwarp();
    // lane l holds bins 255 - 8l .. 248 - 8l (descending), with the counts of all bins above
    uint32_t c[8], own = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      c[i] = hist[255 - 8 * lane - i];
      own += c[i];
    }
    uint32_t incl = own;                              // inclusive prefix over lanes 0..l
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    const uint32_t before = incl - own;
    const bool mine = before < (uint32_t)rank && incl >= (uint32_t)rank;
    const int owner = __ffs(__ballot_sync(0xFFFFFFFFu, mine)) - 1;
    int bin = 0, above = 0;
    if (mine) {
      uint32_t run = before;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (run + c[i] >= (uint32_t)rank) {
          bin = 255 - 8 * lane - i;
          above = (int)run;
          break;
        }
        run += c[i];
      }
    }
    bin = __shfl_sync(0xFFFFFFFFu, bin, owner);
    above = __shfl_sync(0xFFFFFFFFu, above, owner);
    rank -= above;
    prefix |= (uint32_t)bin << shift;
    pmask |= 255u << shift;
    __syncwarp();
  }
  const uint32_t T = prefix;                          // the k-th largest key
  const int eq_take = rank;                           // keys equal to T still to take
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
  // ---- values of the selected positions, 16 per tile on the tensor cores (the dense
  // kernel's arithmetic) with weights 2^(s - M) <= 2^8 (M trails the largest score by at
  // most 8, the lazy rescaling bound); the denominator divides at the end
  const int gid = lane >> 2, tig = lane & 3;
  float acc[2 * NW][4];
#pragma unroll
  for (int u = 0; u < 2 * NW; ++u)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[u][c] = 0.0f;
  float asum[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) asum[g] = 0.0f;
  const int64_t head_row0 = (int64_t)bh * cap;
#pragma unroll 1
  for (int i0 = 0; i0 < k; i0 += 16) {
    uint32_t vw[2][NW], va[2][NG];
    float p[2];
    bool valid[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int i = i0 + gid + 8 * r;
      valid[r] = i < k;
      const int t = sel[valid[r] ? i : k - 1];
      const int64_t row = head_row0 + t;
      const uint8_t* vp = vc + row * (D / 2) + tig * 4 * NW;
      if constexpr (NW == 4) {
        const uint4 u = ldg_nc_v4(vp);
        vw[r][0] = u.x; vw[r][1] = u.y; vw[r][2 % NW] = u.z; vw[r][3 % NW] = u.w;
      } else {
        const uint2 u = *reinterpret_cast<const uint2*>(vp);
        vw[r][0] = u.x; vw[r][1 % NW] = u.y;
      }
      if constexpr (NG == 2) {
        const uint2 u = *reinterpret_cast<const uint2*>(vab + row * NG);
        va[r][0] = u.x; va[r][NG - 1] = u.y;
      } else {
        va[r][0] = vab[row];
      }
      p[r] = valid[r] ? exp2f(key_to_f32(keys[t]) - m) : 0.0f;
    }
    q4attn::v_tile<D>(vw, va, p, valid, lane, acc, asum);
  }
#pragma unroll
  for (int g = 0; g < NG; ++g) asum[g] = warp_sum_gid(asum[g]);
  const float inv_z = 1.0f / z;
  uint16_t* o = out + (int64_t)bh * D;
  q4attn::v_channels<D>(acc, asum, lane, [&](int ch, float v) { o[ch] = f2h(v * inv_z); });
}

template <int D>
cudaError_t launch_attend(const fg_kvcache& kv, int32_t len, int32_t k, uint16_t* out,
                          int32_t* sel, const uint32_t* keys, const float2* ml, int splits,
                          cudaStream_t st) {
  const int64_t nbh = (int64_t)kv.B * kv.H;
  const size_t smem = 1024 + (size_t)len * 4 + (size_t)k * 4;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_attend_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(topk_attend_kernel<D>, dim3((unsigned)nbh), dim3(32), smem, st, keys, ml,
                    splits, kv.v_codes, reinterpret_cast<const uint32_t*>(kv.v_ab), kv.H, kv.cap,
                    len, k, out, sel);
}

// Workspace: the keys [B*H][len], then (16-byte aligned) the work items' (m, l).
size_t keys_bytes(const fg_kvcache& kv, int32_t len) {
  return ((size_t)kv.B * kv.H * (size_t)len * sizeof(uint32_t) + 15) & ~size_t(15);
}

}  // namespace

size_t decode_attn_topk_ws_bytes(const fg_kvcache& kv, int32_t len) {
  // the split count is at most the plan for kMaxSms SMs (decode_attn_splits)
  const int splits = decode_attn_splits(kv, len, kMaxSms);
  return keys_bytes(kv, len) + (size_t)kv.B * kv.H * splits * sizeof(float2);
}

cudaError_t launch_decode_attn_topk(const uint16_t* q, int64_t q_stride, const fg_kvcache& kv,
                                    int32_t len, int32_t k, float scale, uint16_t* out,
                                    int32_t* sel, void* ws, int nsm, cudaStream_t st) {
  if ((int64_t)kv.B * kv.H >= (1ll << 31)) return cudaErrorInvalidValue;
  uint32_t* keys = static_cast<uint32_t*>(ws);
  float2* ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) + keys_bytes(kv, len));
  int splits = 1;
  cudaError_t e = launch_decode_attn_scores(q, q_stride, kv, len, scale, keys, ml, nsm, st, &splits);
  if (e != cudaSuccess) return e;
  const int d = kv.h / kv.H;
  return (d == 128) ? launch_attend<128>(kv, len, k, out, sel, keys, ml, splits, st)
                    : launch_attend<64>(kv, len, k, out, sel, keys, ml, splits, st);
}

}  // namespace fg
