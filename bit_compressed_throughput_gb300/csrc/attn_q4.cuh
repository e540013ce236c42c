// Scores of cached positions against one query on the tensor cores, from 4-bit K codes
// (sm_103a): shared by the dense and the top-K decode attention.
//
// Per group g of 64 channels (a = min, s = (b - a)/15, c = code):
//   q . k^ = sum_g ( s_g * sum_{j in g} c_j q_j  +  a_g * Q_g ),  Q_g = sum_{j in g} q_j
// [FlexGen review (jaehun.me), "4-bit 압축은 정수 연산 가속과 같은가": KV grouped 64 along
// the hidden dimension, restored before compute].  A nibble masked in place is an exact fp16
// subnormal: c * 2^-24 (nibble at bit 0) or 16c * 2^-24 (nibble at bit 4), so one shift and
// four ANDs split a 32-bit word into four code pairs; the 16 is folded into q and 2^24 into the
// group scale.  The dot products run on mma.sync m16n8k16 with fp32 accumulation (the
// products are exact in fp32).
//
// Tile layout: 16 positions; lane (gid, tig) holds positions gid and gid+8, NW = d/32 words
// each (bytes tig*4*NW .. of the row: channels tig*8*NW + 8w + i of word w, nibble i).  The
// dot-product index order follows what the lane holds, and q is permuted the same way; every
// column n of the q operand carries group n & 1 (or group 0 when d = 64), so each lane's
// accumulator fragment holds its own rows' dot products for every group.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "fg_common.cuh"

namespace fg {
namespace q4attn {

// float -> unsigned key with the same order (negative values reversed below the positives)
__device__ __forceinline__ uint32_t order_key_f32(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_f32(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// The four pairs (c_i, c_{i+4}) of a code word as fp16 subnormals: pairs 0 and 2 hold
// c * 2^-24, pairs 1 and 3 hold 16c * 2^-24.
__device__ __forceinline__ void code_pairs(uint32_t w, uint32_t (&p)[4]) {
  const uint32_t w8 = w >> 8;
  p[0] = w & 0x000F000Fu;
  p[1] = w & 0x00F000F0u;
  p[2] = w8 & 0x000F000Fu;
  p[3] = w8 & 0x00F000F0u;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The query of one (sequence, head) as B fragments, with the per-group sums Q0, Q1 and the
// code-scale factor ck, all in the base-2 score scale.
template <int D>
struct QFrag {
  uint32_t bq[2 * (D / 32)][2];
  float Q0, Q1, ck;
};

// q_head: the head's d fp16 values (16-byte aligned).  Every lane of the warp calls it.
template <int D>
__device__ __forceinline__ void load_q_frag(const uint16_t* q_head, int lane, float scale_log2,
                                            QFrag<D>& f) {
  constexpr int NW = D / 32, NG = D / 64;
  const int gid = lane >> 2, tig = lane & 3;
  const uint16_t* qh = q_head + tig * 8 * NW;
  uint32_t qw[NW * 4];
#pragma unroll
  for (int c = 0; c < NW; ++c) {
    const uint4 u = ldg_nc_v4(qh + 8 * c);
    qw[4 * c] = u.x; qw[4 * c + 1] = u.y; qw[4 * c + 2] = u.z; qw[4 * c + 3] = u.w;
  }
  auto qval = [&](int w, int i) -> uint32_t {       // fp16 bits of channel 8w+i of the chunk
    const uint32_t word = qw[4 * w + (i >> 1)];
    return (i & 1) ? (word >> 16) : (word & 0xFFFFu);
  };
  const int my_group = (NG == 2) ? (tig >> 1) : 0;
  // q for pairs with factor 1, q/16 (exact) for pairs with factor 16
  float qsum = 0.0f;
#pragma unroll
  for (int s = 0; s < 2 * NW; ++s) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int p = 2 * s + r, w = p >> 2, i = p & 3;
      uint32_t v = qval(w, i) | (qval(w, i + 4) << 16);
      const float2 fq = unpack_h2(v);
      qsum += fq.x + fq.y;
      if (i & 1) {
        const uint32_t k16 = 0x2C002C00u;               // half2(1/16, 1/16)
        __half2 h = __hmul2(*reinterpret_cast<__half2*>(&v), *reinterpret_cast<const __half2*>(&k16));
        v = *reinterpret_cast<uint32_t*>(&h);
      }
      f.bq[s][r] = (NG == 1 || (gid & 1) == my_group) ? v : 0u;
    }
  }
  // sum over the lanes sharing this group: tig pairs (NG == 2) or all four (NG == 1)
  qsum += __shfl_xor_sync(0xFFFFFFFFu, qsum, 1);
  if (NG == 1) qsum += __shfl_xor_sync(0xFFFFFFFFu, qsum, 2);
  // scores in base 2: the softmax scale rides on the group sums and the code scale
  f.Q0 = __shfl_sync(0xFFFFFFFFu, qsum, lane & ~3) * scale_log2;
  f.Q1 = (NG == 2) ? __shfl_sync(0xFFFFFFFFu, qsum, (lane & ~3) | 2) * scale_log2 : 0.0f;
  // the dot products come out as 2^-24 * sum_j c_j q_j: the code scale (b - a)/15 takes
  // the 2^24 back
  f.ck = (16777216.0f / 15.0f) * scale_log2;
}

// Base-2 scores of the lane's two rows (gid, gid+8) of a 16-position tile from their code
// words kw[r][0..NW) and group statistics ka[r][0..NG).
template <int D>
__device__ __forceinline__ void tile_scores(const uint32_t (&kw)[2][D / 32],
                                            const uint32_t (&ka)[2][D / 64], const QFrag<D>& f,
                                            float (&sc)[2]) {
  constexpr int NW = D / 32, NG = D / 64;
  float dk[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    uint32_t c0[4], c1[4];                           // rows gid and gid+8
    code_pairs(kw[0][w], c0);
    code_pairs(kw[1][w], c1);
    mma16816(dk, c0[0], c1[0], c0[1], c1[1], f.bq[2 * w][0], f.bq[2 * w][1]);
    mma16816(dk, c0[2], c1[2], c0[3], c1[3], f.bq[2 * w + 1][0], f.bq[2 * w + 1][1]);
  }
  // dk[2r] (group 0) and dk[2r+1] (group 1, or group 0 again) belong to row gid + 8r
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float2 ab0 = unpack_h2(ka[r][0]);
    float dot = (ab0.y - ab0.x) * dk[2 * r];
    float off = ab0.x * f.Q0;
    if (NG == 2) {
      const float2 ab1 = unpack_h2(ka[r][NG - 1]);
      dot = fmaf(ab1.y - ab1.x, dk[2 * r + 1], dot);
      off = fmaf(ab1.x, f.Q1, off);
    }
    sc[r] = fmaf(dot, f.ck, off);
  }
}

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// Values of one 16-position tile: sum_t p_t v^_tj = sum_t (p_t s_tg) c_tj + sum_t p_t a_tg.
// The lane holds rows gid and gid+8 (code words vw[r], statistics va[r]) with weights p[r];
// rows with valid[r] false take (a, b) = (0, 0), so their bytes contribute exact zeros.  The
// weights w_tg = p_t (b - a)_tg / 15 go to fp16 B fragments (rows 2tig, 2tig+1 and +8, column
// n carrying group n & 1); each packed code word is transposed with movmatrix (the lane then
// holds 4 channels at two positions) and split into code pairs, the A operand.
// acc[2w+h] row gid accumulates channel cb + 2h times 2^-24, row gid+8 channel cb + 2h + 1
// times 2^-20 (cb = 8*NW*(gid>>1) + 8w + 4*(gid&1)), in columns 2tig (group 0) and 2tig+1
// (group 1); asum[g] accumulates sum_t p_t a_tg over the lane's rows.
template <int D>
__device__ __forceinline__ void v_tile(const uint32_t (&vw)[2][D / 32],
                                       const uint32_t (&va)[2][D / 64], const float (&p)[2],
                                       const bool (&valid)[2], int lane,
                                       float (&acc)[2 * (D / 32)][4], float (&asum)[D / 64]) {
  constexpr int NW = D / 32, NG = D / 64;
  const int gid = lane >> 2, tig = lane & 3;
  uint32_t wrow[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float pr = p[r];
    const float p15 = pr * (1.0f / 15.0f);
    const float2 ab0 = unpack_h2(valid[r] ? va[r][0] : 0u);
    const float w0 = p15 * (ab0.y - ab0.x);
    asum[0] = fmaf(pr, ab0.x, asum[0]);
    float w1 = w0;
    if (NG == 2) {
      const float2 ab1 = unpack_h2(valid[r] ? va[r][NG - 1] : 0u);
      w1 = p15 * (ab1.y - ab1.x);
      asum[NG - 1] = fmaf(pr, ab1.x, asum[NG - 1]);
    }
    wrow[r] = pack_h2(w0, w1);
  }
  const uint32_t wa = __shfl_sync(0xFFFFFFFFu, wrow[0], 8 * tig);
  const uint32_t wb = __shfl_sync(0xFFFFFFFFu, wrow[0], 8 * tig + 4);
  const uint32_t wc = __shfl_sync(0xFFFFFFFFu, wrow[1], 8 * tig);
  const uint32_t wd = __shfl_sync(0xFFFFFFFFu, wrow[1], 8 * tig + 4);
  const uint32_t sel = (NG == 2 && (gid & 1)) ? 0x7632u : 0x5410u;
  const uint32_t bv0 = __byte_perm(wa, wb, sel);
  const uint32_t bv1 = __byte_perm(wc, wd, sel);
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    uint32_t c0[4], c1[4];
    code_pairs(movtrans(vw[0][w]), c0);
    code_pairs(movtrans(vw[1][w]), c1);
    mma16816(acc[2 * w], c0[0], c0[1], c1[0], c1[1], bv0, bv1);
    mma16816(acc[2 * w + 1], c0[2], c0[3], c1[2], c1[3], bv0, bv1);
  }
}

// The accumulated values per output channel: calls emit(ch, value) for the channels lane tig
// owns (the accumulators u with u % 4 == tig), value = the row's accumulator (times 2^24 or
// 2^20) plus the offset sum of its group.  asum must already hold the warp-wide sums.
template <int D, typename Emit>
__device__ __forceinline__ void v_channels(const float (&acc)[2 * (D / 32)][4],
                                           const float (&asum)[D / 64], int lane, Emit emit) {
  constexpr int NW = D / 32, NG = D / 64;
  const int gid = lane >> 2, tig = lane & 3;
  const int g_lane = (NG == 2) ? (gid >> 2) : 0;     // group of every channel of row gid
  const float A = (NG == 2 && g_lane) ? asum[NG - 1] : asum[0];
  const int cbase = 8 * NW * (gid >> 1) + 4 * (gid & 1);
#pragma unroll
  for (int u = 0; u < 2 * NW; ++u) {
    if ((u & 3) != tig) continue;
    const int ch = cbase + 8 * (u >> 1) + 2 * (u & 1);
    emit(ch, (g_lane ? acc[u][1] : acc[u][0]) * 16777216.0f + A);
    emit(ch + 1, (g_lane ? acc[u][3] : acc[u][2]) * 1048576.0f + A);
  }
}

}  // namespace q4attn
}  // namespace fg
