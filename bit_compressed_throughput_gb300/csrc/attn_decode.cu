// Decode attention over the 4-bit KV cache (sm_103a).
//
// For each sequence b and head hd: o = sum_t softmax_t(scale * q . k^_t) v^_t over the
// cached positions t < len, where k^, v^ are restored from 4-bit codes with their
// group's (a, b) [FlexGen review (jaehun.me), "4-bit 압축은 정수 연산 가속과 같은가":
// KV grouped 64 along the hidden dimension, restored before compute].  Decoding
// attention is bound by reading the cache [FlexGen paper explainer, "Computation
// Delegation"]; this kernel streams each cached byte once.
//
// Algebra per group g of 64 channels (a = min, s = (b - a)/15, c = code):
//   q . k^  = sum_g ( s_g * sum_{j in g} c_j q_j  +  a_g * Q_g ),  Q_g = sum_{j in g} q_j
//   sum_t p_t v^_tj = sum_t (p_t s_tg) c_tj + sum_t p_t a_tg
// so the per-element work is a dot product of integer codes with fp16 weights.  The codes
// become exact fp16 integers by OR-ing the nibble into the mantissa of 1024.0 and
// subtracting 1024 (exact), and the dot products run on mma.sync m16n8k16 with fp32
// accumulation (the product of a 4-bit integer and an fp16 value is exact in fp32).
//
// One warp owns (b, hd, split): 16 positions per tile, lane (gid, tig) loads positions
// gid and gid+8 of the tile, 16 bytes of codes each for K and V (d = 128: 32 channels
// per lane).  The dot-product index order inside a tile is permuted to match what each
// lane loaded; q (K side) is permuted the same way, and the V side is transposed in
// registers with movmatrix.  Online softmax (base 2) across tiles; split-sequence
// partials are combined by a second kernel when one (b, hd) per warp would leave SMs idle.
#include <math.h>

#include <algorithm>

#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {
namespace {

constexpr int kWarps = 4;
constexpr int kTile = 16;

__device__ __forceinline__ uint32_t hsub_1024(uint32_t x) {
  __half2 a = *reinterpret_cast<__half2*>(&x);
  const uint32_t k = 0x64006400u;
  __half2 b = *reinterpret_cast<const __half2*>(&k);
  __half2 r = __hsub2(a, b);
  return *reinterpret_cast<uint32_t*>(&r);
}

// Pair i (0..3) of a code word as exact fp16 integers (c_i, c_{i+4}).
__device__ __forceinline__ uint32_t code_pair(uint32_t w, int i) {
  return hsub_1024(((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u);
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

template <int NW>
struct TileRegs {
  uint32_t k[2][NW], v[2][NW];   // codes of rows gid, gid+8
  uint32_t ka[2][2], va[2][2];   // (a,b) words of rows gid, gid+8, groups 0..NG-1
};

// D = head dim; NW = 32-bit code words per lane per row (D/32); NG = groups per head.
template <int D>
__global__ void __launch_bounds__(kWarps * 32)
decode_attn_kernel(const uint16_t* __restrict__ q, int64_t q_stride,
                   const uint8_t* __restrict__ kc, const uint8_t* __restrict__ vc,
                   const uint32_t* __restrict__ kab, const uint32_t* __restrict__ vab, int B,
                   int H, int cap, int len, int splits, int tiles_per_split, float scale_log2,
                   uint16_t* __restrict__ out, float* __restrict__ partial) {
  constexpr int NW = D / 32;
  constexpr int NG = D / 64;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int64_t item = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (item >= (int64_t)B * H * splits) return;
  const int split = (int)(item % splits);
  const int64_t bh = item / splits;
  const int b = (int)(bh / H), hd = (int)(bh % H);
  const int t_begin = split * tiles_per_split * kTile;
  const int t_end = min(len, t_begin + tiles_per_split * kTile);

  // ---- q: this lane's channels j = tig*8*NW + 8w + i + 4e, permuted into B fragments.
  const uint16_t* qh = q + (int64_t)b * q_stride + (int64_t)hd * D + tig * 8 * NW;
  uint32_t qw[NW * 4];
#pragma unroll
  for (int c = 0; c < NW; ++c) {
    const uint4 u = ldg_nc_v4(qh + 8 * c);
    qw[4 * c] = u.x; qw[4 * c + 1] = u.y; qw[4 * c + 2] = u.z; qw[4 * c + 3] = u.w;
  }
  // fp16 bits of channel 8w+i of this lane's chunk
  auto qval = [&](int w, int i) -> uint32_t {
    const uint32_t word = qw[4 * w + (i >> 1)];
    return (i & 1) ? (word >> 16) : (word & 0xFFFFu);
  };
  const int my_group = (NG == 2) ? (tig >> 1) : 0;
  float qsum = 0.0f;
#pragma unroll
  for (int w = 0; w < NW; ++w)
#pragma unroll
    for (int i = 0; i < 8; ++i) qsum += h2f((uint16_t)qval(w, i));
  // Sum over the lanes sharing this group: tig pairs (NG == 2) or all four (NG == 1).
  qsum += __shfl_xor_sync(0xFFFFFFFFu, qsum, 1);
  if (NG == 1) qsum += __shfl_xor_sync(0xFFFFFFFFu, qsum, 2);
  const float Q0 = __shfl_sync(0xFFFFFFFFu, qsum, lane & ~3);
  const float Q1 = (NG == 2) ? __shfl_sync(0xFFFFFFFFu, qsum, (lane & ~3) | 2) : 0.0f;

  uint32_t bq[2 * NW][2];
#pragma unroll
  for (int s = 0; s < 2 * NW; ++s) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int p = 2 * s + r, w = p >> 2, i = p & 3;
      const uint32_t v = qval(w, i) | (qval(w, i + 4) << 16);
      bq[s][r] = (gid == my_group) ? v : 0u;
    }
  }

  // ---- stream the tiles
  const int64_t head_row0 = ((int64_t)b * H + hd) * cap;      // slot of position 0
  const uint8_t* kbase = kc + head_row0 * (D / 2) + tig * 4 * NW;
  const uint8_t* vbase = vc + head_row0 * (D / 2) + tig * 4 * NW;
  const uint32_t* kabase = kab + head_row0 * NG;
  const uint32_t* vabase = vab + head_row0 * NG;

  auto load_tile = [&](int t0, TileRegs<NW>& R) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int t = t0 + gid + 8 * r;
      if (t < t_end) {
        if (NW == 4) {
          const uint4 uk = ldg_nc_v4(kbase + (int64_t)t * (D / 2));
          const uint4 uv = ldg_nc_v4(vbase + (int64_t)t * (D / 2));
          R.k[r][0] = uk.x; R.k[r][1] = uk.y; R.k[r][2 % NW] = uk.z; R.k[r][3 % NW] = uk.w;
          R.v[r][0] = uv.x; R.v[r][1] = uv.y; R.v[r][2 % NW] = uv.z; R.v[r][3 % NW] = uv.w;
        } else {
          const uint2 uk = *reinterpret_cast<const uint2*>(kbase + (int64_t)t * (D / 2));
          const uint2 uv = *reinterpret_cast<const uint2*>(vbase + (int64_t)t * (D / 2));
          R.k[r][0] = uk.x; R.k[r][1 % NW] = uk.y;
          R.v[r][0] = uv.x; R.v[r][1 % NW] = uv.y;
        }
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          R.ka[r][g] = kabase[(int64_t)t * NG + g];
          R.va[r][g] = vabase[(int64_t)t * NG + g];
        }
      } else {
#pragma unroll
        for (int w = 0; w < NW; ++w) { R.k[r][w] = 0u; R.v[r][w] = 0u; }
#pragma unroll
        for (int g = 0; g < NG; ++g) { R.ka[r][g] = 0u; R.va[r][g] = 0u; }
      }
    }
  };

  float m_run = -INFINITY, l_run = 0.0f;
  float acc[2 * NW][4];
#pragma unroll
  for (int u = 0; u < 2 * NW; ++u)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[u][c] = 0.0f;
  float asum[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) asum[g] = 0.0f;

  TileRegs<NW> cur, nxt;
  if (t_begin < t_end) load_tile(t_begin, cur);
  for (int t0 = t_begin; t0 < t_end; t0 += kTile) {
    if (t0 + kTile < t_end) load_tile(t0 + kTile, nxt);

    // ---- scores: K codes (rows t) x permuted q, one column per group
    float dk[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < 2 * NW; ++s) {
      const int p0 = 2 * s, p1 = 2 * s + 1;
      const uint32_t a0 = code_pair(cur.k[0][p0 >> 2], p0 & 3);
      const uint32_t a1 = code_pair(cur.k[1][p0 >> 2], p0 & 3);
      const uint32_t a2 = code_pair(cur.k[0][p1 >> 2], p1 & 3);
      const uint32_t a3 = code_pair(cur.k[1][p1 >> 2], p1 & 3);
      mma16816(dk, a0, a1, a2, a3, bq[s][0], bq[s][1]);
    }
    // lanes with tig == 0 hold D[t][0..1] for t = gid (dk[0], dk[1]) and gid+8 (dk[2], dk[3])
    float sc[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float2 ab0 = unpack_h2(cur.ka[r][0]);
      float v = (ab0.y - ab0.x) * (1.0f / 15.0f) * dk[2 * r] + ab0.x * Q0;
      if (NG == 2) {
        const float2 ab1 = unpack_h2(cur.ka[r][NG - 1]);
        v += (ab1.y - ab1.x) * (1.0f / 15.0f) * dk[2 * r + 1] + ab1.x * Q1;
      }
      v = __shfl_sync(0xFFFFFFFFu, v, lane & ~3);
      const int t = t0 + gid + 8 * r;
      sc[r] = (t < t_end) ? v * scale_log2 : -INFINITY;
    }
    float mx = fmaxf(sc[0], sc[1]);
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
    const float m_new = fmaxf(m_run, mx);
    const float corr = (m_run == -INFINITY) ? 0.0f : exp2f(m_run - m_new);
    const float p0 = exp2f(sc[0] - m_new), p1 = exp2f(sc[1] - m_new);
    float ps = p0 + p1;
    ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 4);
    ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 8);
    ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 16);
    if (m_new != m_run) {
      l_run *= corr;
#pragma unroll
      for (int u = 0; u < 2 * NW; ++u)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[u][c] *= corr;
#pragma unroll
      for (int g = 0; g < NG; ++g) asum[g] *= corr;
      m_run = m_new;
    }
    l_run += ps;

    // ---- V weights w_tg = p_t * s_tg (fp16) and the offset term sum_t p_t a_tg
    uint32_t wrow[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float p = r ? p1 : p0;
      const float2 ab0 = unpack_h2(cur.va[r][0]);
      const float w0 = p * (ab0.y - ab0.x) * (1.0f / 15.0f);
      asum[0] += p * ab0.x;
      float w1 = 0.0f;
      if (NG == 2) {
        const float2 ab1 = unpack_h2(cur.va[r][NG - 1]);
        w1 = p * (ab1.y - ab1.x) * (1.0f / 15.0f);
        asum[NG - 1] += p * ab1.x;
      }
      wrow[r] = pack_h2(w0, w1);
    }
    // B fragment: rows t = 2tig, 2tig+1 (and +8), column n = gid (group n)
    const uint32_t wa = __shfl_sync(0xFFFFFFFFu, wrow[0], 8 * tig);
    const uint32_t wb = __shfl_sync(0xFFFFFFFFu, wrow[0], 8 * tig + 4);
    const uint32_t wc = __shfl_sync(0xFFFFFFFFu, wrow[1], 8 * tig);
    const uint32_t wd = __shfl_sync(0xFFFFFFFFu, wrow[1], 8 * tig + 4);
    uint32_t bv0 = 0u, bv1 = 0u;
    if (gid < NG) {
      const uint32_t sel = gid ? 0x7632u : 0x5410u;   // pick the high or low halves
      bv0 = __byte_perm(wa, wb, sel);
      bv1 = __byte_perm(wc, wd, sel);
    }
    // ---- V codes transposed to (channel rows, position columns)
#pragma unroll
    for (int u = 0; u < 2 * NW; ++u) {
      const int px = 2 * u, py = 2 * u + 1;
      const uint32_t x0 = movtrans(code_pair(cur.v[0][px >> 2], px & 3));
      const uint32_t y0 = movtrans(code_pair(cur.v[0][py >> 2], py & 3));
      const uint32_t x1 = movtrans(code_pair(cur.v[1][px >> 2], px & 3));
      const uint32_t y1 = movtrans(code_pair(cur.v[1][py >> 2], py & 3));
      mma16816(acc[u], x0, y0, x1, y1, bv0, bv1);
    }
    cur = nxt;
  }

  // ---- epilogue: o_j = (acc + sum_t p_t a_tg) / l
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    asum[g] += __shfl_xor_sync(0xFFFFFFFFu, asum[g], 4);
    asum[g] += __shfl_xor_sync(0xFFFFFFFFu, asum[g], 8);
    asum[g] += __shfl_xor_sync(0xFFFFFFFFu, asum[g], 16);
  }
  if (tig != 0) return;
  const int g_lo = (NG == 2) ? (gid >> 2) : 0;        // group of channel row gid
  const float A = (NG == 2 && g_lo) ? asum[NG - 1] : asum[0];
  const float inv_l = (l_run > 0.0f) ? 1.0f / l_run : 0.0f;
  const int jbase = (gid >> 1) * 8 * NW + 4 * (gid & 1);
  if (splits == 1) {
    uint16_t* o = out + (int64_t)b * H * D + (int64_t)hd * D;
#pragma unroll
    for (int u = 0; u < 2 * NW; ++u) {
      const int px = 2 * u, py = 2 * u + 1;
      const float vx = (g_lo ? acc[u][1] : acc[u][0]) + A;
      const float vy = (g_lo ? acc[u][3] : acc[u][2]) + A;
      o[jbase + 8 * (px >> 2) + (px & 3)] = f2h(vx * inv_l);
      o[jbase + 8 * (py >> 2) + (py & 3)] = f2h(vy * inv_l);
    }
  } else {
    float* pp = partial + (bh * splits + split) * (int64_t)(D + 2);
#pragma unroll
    for (int u = 0; u < 2 * NW; ++u) {
      const int px = 2 * u, py = 2 * u + 1;
      pp[jbase + 8 * (px >> 2) + (px & 3)] = (g_lo ? acc[u][1] : acc[u][0]) + A;
      pp[jbase + 8 * (py >> 2) + (py & 3)] = (g_lo ? acc[u][3] : acc[u][2]) + A;
    }
    if (gid == 0) {
      pp[D] = m_run;
      pp[D + 1] = l_run;
    }
  }
}

// One warp per (b, hd): merge the split partials (m, l, unnormalised o) in base 2.
template <int D>
__global__ void __launch_bounds__(128)
decode_combine_kernel(const float* __restrict__ partial, int64_t nbh, int H, int splits,
                      uint16_t* __restrict__ out) {
  const int64_t bh = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (bh >= nbh) return;
  const float* pp = partial + bh * splits * (int64_t)(D + 2);
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, pp[s * (D + 2) + D]);
  float L = 0.0f;
  float o[D / 32];
#pragma unroll
  for (int c = 0; c < D / 32; ++c) o[c] = 0.0f;
  for (int s = 0; s < splits; ++s) {
    const float ms = pp[s * (D + 2) + D];
    const float wgt = (ms == -INFINITY) ? 0.0f : exp2f(ms - M);
    L += wgt * pp[s * (D + 2) + D + 1];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) o[c] += wgt * pp[s * (D + 2) + c * 32 + lane];
  }
  const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;
  const int64_t b = bh / H, hd = bh % H;
  uint16_t* op = out + b * H * D + hd * D;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) op[c * 32 + lane] = f2h(o[c] * inv);
}

constexpr int kTargetWarpsPerSm = 32;   // two waves of 16 resident warps

}  // namespace

int decode_attn_splits(const fg_kvcache& kv, int32_t len, int nsm) {
  const int64_t bh = (int64_t)kv.B * kv.H;
  if (bh == 0) return 1;
  const int ntiles = (len + kTile - 1) / kTile;
  const int64_t target = (int64_t)nsm * kTargetWarpsPerSm;
  int64_t splits = (target + bh - 1) / bh;
  const int min_tiles = 4;
  splits = std::min<int64_t>(splits, std::max(1, ntiles / min_tiles));
  splits = std::max<int64_t>(1, std::min<int64_t>(splits, ntiles));
  const int tps = (int)((ntiles + splits - 1) / splits);
  return (ntiles + tps - 1) / tps;
}

size_t decode_attn_ws_bytes(const fg_kvcache& kv, int32_t len, int nsm) {
  const int splits = decode_attn_splits(kv, len, nsm);
  if (splits <= 1) return 0;
  const int d = kv.h / kv.H;
  return (size_t)kv.B * kv.H * splits * (d + 2) * sizeof(float);
}

cudaError_t launch_decode_attn(const uint16_t* q, int64_t q_stride, const fg_kvcache& kv,
                               int32_t len, float scale, uint16_t* out, void* ws, int nsm,
                               cudaStream_t st, int* kernels_out, cudaEvent_t mid_event) {
  const int d = kv.h / kv.H;
  const int splits = decode_attn_splits(kv, len, nsm);
  const int ntiles = (len + kTile - 1) / kTile;
  const int tps = (ntiles + splits - 1) / splits;
  const int64_t items = (int64_t)kv.B * kv.H * splits;
  const unsigned grid = (unsigned)((items + kWarps - 1) / kWarps);
  const float sl2 = scale * 1.4426950408889634f;
  float* partial = static_cast<float*>(ws);
  if (d == 128)
    decode_attn_kernel<128><<<grid, kWarps * 32, 0, st>>>(
        q, q_stride, kv.k_codes, kv.v_codes, kv.k_ab, kv.v_ab, kv.B, kv.H, kv.cap, len, splits,
        tps, sl2, out, partial);
  else
    decode_attn_kernel<64><<<grid, kWarps * 32, 0, st>>>(
        q, q_stride, kv.k_codes, kv.v_codes, kv.k_ab, kv.v_ab, kv.B, kv.H, kv.cap, len, splits,
        tps, sl2, out, partial);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *kernels_out = 1;
  if (splits > 1) {
    if (mid_event) cudaEventRecord(mid_event, st);
    const int64_t nbh = (int64_t)kv.B * kv.H;
    const unsigned g2 = (unsigned)((nbh + 3) / 4);
    if (d == 128)
      decode_combine_kernel<128><<<g2, 128, 0, st>>>(partial, nbh, kv.H, splits, out);
    else
      decode_combine_kernel<64><<<g2, 128, 0, st>>>(partial, nbh, kv.H, splits, out);
    e = cudaGetLastError();
    *kernels_out = 2;
  }
  return e;
}

}  // namespace fg
