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
//   topk_scores_kernel  a warp per sixteen 16-position tiles of one (b, hd): the scores on the
//                       tensor cores from the 4-bit K (the dense kernel's arithmetic), in
//                       base 2, into the workspace
//   topk_attend_kernel  one warp per (b, hd): the scores read once into shared memory as
//                       order-preserving keys; the softmax maximum and denominator over all
//                       positions; the k-th largest key by radix selection, eight bits per
//                       round from the top (a 256-bin histogram of the keys that share the
//                       bits found so far, then the bin holding the remaining rank);
//                       the selected positions compacted in position order (keys above T,
//                       then keys equal to T from the lowest position); then the V rows of
//                       the selected positions gathered 16 at a time into the dense
//                       kernel's tensor-core tile (weights 2^(s - m), the softmax
//                       denominator applied at the end).
#include <math.h>

#include "attn_q4.cuh"
#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {

namespace {

constexpr int kScoreWarps = 4;            // warps per CTA of the score kernel
constexpr int kScoreTiles = 4;            // 16-position tiles loaded together
constexpr int kScoreBatches = 4;          // batches of kScoreTiles per warp

// float -> unsigned key with the same order (negative values reversed below the positives)
__device__ __forceinline__ uint32_t order_key_f32(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_f32(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

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

// One warp per kScoreBatches x kScoreTiles consecutive 16-position tiles of one (b, hd),
// kScoreTiles at a time, one query fragment for all of them: the K rows
// straight from global memory (lane (gid, tig): 16 bytes of rows gid and gid+8, a tile is one
// contiguous 1 KB run for d = 128), the scores on the tensor cores, lanes with tig == 0
// writing their two rows.  The loads of a batch are issued before its arithmetic.
template <int D>
__global__ void __launch_bounds__(kScoreWarps * 32)
topk_scores_kernel(const uint16_t* __restrict__ q, int64_t q_stride,
                   const uint8_t* __restrict__ kc, const uint32_t* __restrict__ kab, int H,
                   int cap, int len, float scale_log2, float* __restrict__ scores) {
  constexpr int NW = D / 32, NG = D / 64;
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int bh = blockIdx.x;
  const int b = bh / H, hd = bh - b * H;
  const int ntiles = (len + 15) / 16;
  const int tile_w = (blockIdx.y * kScoreWarps + warp) * kScoreTiles * kScoreBatches;
  if (tile_w >= ntiles) return;
  q4attn::QFrag<D> qf;
  q4attn::load_q_frag<D>(q + (int64_t)b * q_stride + (int64_t)hd * D, lane, scale_log2, qf);
#pragma unroll 1
  for (int tile0 = tile_w; tile0 < min(ntiles, tile_w + kScoreTiles * kScoreBatches);
       tile0 += kScoreTiles) {
    // tiles are whole 16 positions: rows past len stay below cap (a multiple of 16)
    uint32_t kw[kScoreTiles][2][NW], ka[kScoreTiles][2][NG];
#pragma unroll
    for (int i = 0; i < kScoreTiles; ++i) {
      if (tile0 + i >= ntiles) break;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int64_t row = (int64_t)bh * cap + (tile0 + i) * 16 + gid + 8 * r;
        const uint8_t* kp = kc + row * (D / 2) + tig * 4 * NW;
        if constexpr (NW == 4) {
          const uint4 u = ldg_nc_v4(kp);
          kw[i][r][0] = u.x; kw[i][r][1] = u.y; kw[i][r][2 % NW] = u.z; kw[i][r][3 % NW] = u.w;
        } else {
          const uint2 u = *reinterpret_cast<const uint2*>(kp);
          kw[i][r][0] = u.x; kw[i][r][1 % NW] = u.y;
        }
        if constexpr (NG == 2) {
          const uint2 u = *reinterpret_cast<const uint2*>(kab + row * NG);
          ka[i][r][0] = u.x; ka[i][r][NG - 1] = u.y;
        } else {
          ka[i][r][0] = kab[row];
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kScoreTiles; ++i) {
      if (tile0 + i >= ntiles) break;
      float sc[2];
      q4attn::tile_scores<D>(kw[i], ka[i], qf, sc);
      if (tig == 0) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int t = (tile0 + i) * 16 + gid + 8 * r;
          if (t < len) scores[(int64_t)bh * len + t] = sc[r];
        }
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(32)
topk_attend_kernel(const float* __restrict__ scores, const uint8_t* __restrict__ vc,
                   const uint32_t* __restrict__ vab, int H, int cap, int len, int k,
                   uint16_t* __restrict__ out, int32_t* __restrict__ sel_out) {
  constexpr int NW = D / 32, NG = D / 64;
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem);            // 256 radix counters
  uint32_t* keys = hist + 256;                                   // len keys
  int32_t* sel = reinterpret_cast<int32_t*>(keys + len);         // k positions
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x;
  const int bh = blockIdx.x;
  const float* sc = scores + (int64_t)bh * len;
  // ---- the scores once, as order keys in shared memory; the largest key
  uint32_t kmax = 0u;
  for (int t = lane; t < len; t += 32) {
    const uint32_t key = order_key_f32(sc[t]);
    keys[t] = key;
    kmax = max(kmax, key);
  }
  kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
  const float m = key_to_f32(kmax);
  __syncwarp();
  float z = 0.0f;                                     // softmax denominator (base 2)
  for (int t = lane; t < len; t += 32) z += exp2f(key_to_f32(keys[t]) - m);
  z = warp_sum(z);
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
  // kernel's arithmetic) with weights 2^(s - m) <= 1; the denominator divides at the end
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
cudaError_t launch_topk_d(const uint16_t* q, int64_t q_stride, const fg_kvcache& kv, int32_t len,
                          int32_t k, float scale, uint16_t* out, int32_t* sel, float* ws,
                          cudaStream_t st) {
  const int64_t nbh = (int64_t)kv.B * kv.H;
  const float sl2 = scale * 1.4426950408889634f;
  const int ntiles = (len + 15) / 16;
  const int per_cta = kScoreWarps * kScoreTiles * kScoreBatches;
  const dim3 g1((unsigned)nbh, (unsigned)((ntiles + per_cta - 1) / per_cta));
  cudaError_t e = launch_pdl(topk_scores_kernel<D>, g1, dim3(kScoreWarps * 32), 0, st, q, q_stride,
                             kv.k_codes, reinterpret_cast<const uint32_t*>(kv.k_ab), kv.H,
                             kv.cap, len, sl2, ws);
  if (e != cudaSuccess) return e;
  const size_t smem = 1024 + (size_t)len * 4 + (size_t)k * 4;
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
