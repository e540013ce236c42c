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
// so the per-element work is a dot product of integer codes with fp16 weights.  A nibble
// masked in place is an exact fp16 subnormal: c * 2^-24 (nibble at bit 0) or 16c * 2^-24
// (nibble at bit 4), so one shift and one AND per pair of codes suffice, with no offset to
// remove; the 16 is folded into q (K side) or into the epilogue (V side), and 2^24 into the
// group scale.  The dot products run on mma.sync m16n8k16 with fp32 accumulation (the
// products are exact in fp32).
//
// Memory pipeline: a warp owns a flattened stream of 32-position slots (two 16-position
// tiles) over its work items (b, hd, split).  Lane 0 keeps kRing slots in flight with 1-D
// bulk async copies (K codes, V codes, K and V group statistics: four contiguous runs in
// the head-major cache) into a per-warp shared-memory ring, completing on one mbarrier
// per slot; the warp computes on one slot while the others land.  The stream runs across
// item boundaries, so the ring never drains between items.  Copies cover whole
// 16-position tiles (the cache capacity is a multiple of 16); positions at or past the
// end are masked with selects, so never-written cache slots cannot leak into the result.
//
// Inside a tile, lane (gid, tig) reads positions gid and gid+8 (16 bytes of codes each
// for K and V when d = 128).  K side: the dot-product index order is permuted to match
// what each lane holds and q is permuted the same way; every column of the q operand
// carries a group's q, so each lane's accumulator fragment holds its own rows' scores.
// V side: each packed code word is transposed with movmatrix (a lane then holds four
// channels at two positions) before it is split into code pairs.  Online softmax (base
// 2) per item; split items write (m, l, unnormalised o) partials that a second kernel
// combines.
//
// Every mbarrier wait is bounded; on timeout the warp sets the device error word read by
// fg_check_device_error, drains its copies and stops.
#include <math.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "attn_q4.cuh"
#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {

__device__ unsigned int g_attn_error = 0;

namespace {

constexpr int kWarps = 4;
constexpr int kTile = 16;                 // positions per mma step
constexpr int kSub = 3;                   // tiles per ring slot
constexpr int kSlotPos = kSub * kTile;    // positions per ring slot
constexpr int kRing = 2;                  // slots per warp (K and V)
constexpr int kRingScores = 4;            // slots per warp of the scores-only instance (K)
constexpr int kPlanWarpsPerSm = 16;       // resident warps per SM assumed by the split plan
constexpr long long kWaitCycles = 1ll << 32;

// A slot holds K codes, V codes, K statistics, V statistics (SC: K codes and statistics).
template <int D, bool SC>
struct Ring {
  static constexpr int NG = D / 64;                     // groups per head
  static constexpr int ROW_CODE = D / 2;                // code bytes of one position
  static constexpr int ROW_AB = NG * 4;                 // statistics bytes of one position
  static constexpr int ROW_BYTES = (SC ? 1 : 2) * (ROW_CODE + ROW_AB);
  static constexpr int CODE_BYTES = kSlotPos * ROW_CODE;
  static constexpr int AB_BYTES = kSlotPos * ROW_AB;
  static constexpr int KAB_OFF = (SC ? 1 : 2) * CODE_BYTES;     // K statistics in a slot
  static constexpr int DEPTH = SC ? kRingScores : kRing;
  static constexpr int SLOT = kSlotPos * ROW_BYTES;
  static constexpr int WARP_BYTES = DEPTH * SLOT;
  static constexpr int CTA_BYTES = kWarps * WARP_BYTES + kWarps * DEPTH * 8;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}


// 2^x on the special-function unit; inputs are <= 8 (lazy rescaling) or -inf, results that
// would be subnormal flush to zero, which only drops terms below 2^-126 of the largest.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void bar_init(uint32_t bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void bar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool bar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait; false (and the device error word set) if it ran out.  The non-blocking
// test_wait goes first: a slot's copies have usually landed by the time it is consumed.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
  {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    if (ok) return true;
  }
  const long long t0 = clock64();
  while (!bar_try(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(&g_attn_error, 1u);
      return false;
    }
  }
  return true;
}
// One contiguous run global -> shared through the bulk-copy engine, completing on `bar`.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Loads N consecutive 32-bit words from shared memory (N = 1, 2 or 4).
template <int N>
__device__ __forceinline__ void load_words(const uint8_t* p, uint32_t (&w)[N]) {
  if constexpr (N == 4) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
  } else if constexpr (N == 2) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    w[0] = u.x; w[1] = u.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  }
}

// Work item -> (b, hd, position range).
struct Item {
  int b, hd, split, t_begin, t_end, nslots;
};
__device__ __forceinline__ Item item_of(int item, int H, int len, int splits, int tps) {
  Item it;
  const int bh = item / splits;
  it.split = item - bh * splits;
  it.b = bh / H;
  it.hd = bh - it.b * H;
  it.t_begin = it.split * tps * kTile;
  it.t_end = min(len, it.t_begin + tps * kTile);
  it.nslots = (it.t_end - it.t_begin + kSlotPos - 1) / kSlotPos;
  return it;
}

// D = head dim; NW = 32-bit code words per lane per row (D/32); NG = groups per head.
// SC: the scores-only instance (top-K attention): no V; every valid score goes to keys
// (order keys of the base-2 scores, row b*H + hd of len) and each work item's softmax state
// (m, l) to ml; out and partial are unused.
template <int D, bool SC>
__global__ void __launch_bounds__(kWarps * 32, 4)
decode_attn_kernel(const uint16_t* __restrict__ q, int64_t q_stride,
                   const uint8_t* __restrict__ kc, const uint8_t* __restrict__ vc,
                   const uint32_t* __restrict__ kab, const uint32_t* __restrict__ vab, int B,
                   int H, int cap, int len, int splits, int tps, float scale_log2,
                   uint16_t* __restrict__ out, float* __restrict__ partial,
                   uint32_t* __restrict__ keys, float2* __restrict__ ml) {
  using R = Ring<D, SC>;
  constexpr int kRing = R::DEPTH;
  constexpr int NW = D / 32;
  constexpr int NG = D / 64;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  uint8_t* ring = smem + warp * R::WARP_BYTES;
  const uint32_t bar0 = smem_u32(smem + kWarps * R::WARP_BYTES) + warp * kRing * 8;
  const int items = B * H * splits;                     // < 2^31 (checked on the host)
  const int nwarps = gridDim.x * kWarps;
  const int first = blockIdx.x * kWarps + warp;

  if (lane == 0) {
    for (int s = 0; s < kRing; ++s) bar_init(bar0 + 8 * s);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  pdl_launch_dependents();
  pdl_wait();

  // ---- issue cursor (used by lane 0 only): kRing slots ahead of the compute cursor
  int ii = first, islot = 0, is = 0, issued = 0;
  Item iitem = item_of(ii < items ? ii : 0, H, len, splits, tps);
  auto issue = [&]() {
    if (ii >= items) return;
    const uint32_t bar = bar0 + 8 * is;
    uint8_t* slot = ring + is * R::SLOT;
    const int t0 = iitem.t_begin + islot * kSlotPos;
    // whole 16-position tiles up to the one holding t_end - 1: never past cap, since
    // t_end <= cap and cap is a multiple of 16
    const int rows = min(kSlotPos, (iitem.t_end - t0 + kTile - 1) / kTile * kTile);
    const int64_t row0 = ((int64_t)iitem.b * H + iitem.hd) * cap + t0;
    // the slot was last read through the generic proxy; order that before the copy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    bar_expect_tx(bar, (uint32_t)(rows * R::ROW_BYTES));
    bulk_copy(smem_u32(slot), kc + row0 * R::ROW_CODE, rows * R::ROW_CODE, bar);
    bulk_copy(smem_u32(slot + R::KAB_OFF), kab + row0 * NG, rows * R::ROW_AB, bar);
    if constexpr (!SC) {
      bulk_copy(smem_u32(slot + R::CODE_BYTES), vc + row0 * R::ROW_CODE, rows * R::ROW_CODE, bar);
      bulk_copy(smem_u32(slot + 2 * R::CODE_BYTES + R::AB_BYTES), vab + row0 * NG,
                rows * R::ROW_AB, bar);
    }
    ++issued;
    if (++is == kRing) is = 0;
    if (++islot == iitem.nslots) {
      ii += nwarps;
      islot = 0;
      if (ii < items) iitem = item_of(ii, H, len, splits, tps);
    }
  };
  if (lane == 0)
    for (int r = 0; r < kRing; ++r) issue();

  int cs = 0, consumed = 0;             // compute cursor: ring slot, slots consumed
  uint32_t cph = 0;                     // parity of the slot's current phase
  bool ok = true;
  for (int ci = first; ci < items && ok; ci += nwarps) {
    const Item it = item_of(ci, H, len, splits, tps);

    // ---- q as B fragments (permuted to the lanes' code words), group sums, code scale
    q4attn::QFrag<D> qf;
    q4attn::load_q_frag<D>(q + (int64_t)it.b * q_stride + (int64_t)it.hd * D, lane, scale_log2,
                           qf);

    float m_run = -INFINITY;
    float l_run = 0.0f;                 // this lane's rows only; summed over gid at the end
    float acc[2 * NW][4];
#pragma unroll
    for (int u = 0; u < 2 * NW; ++u)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[u][c] = 0.0f;
    float asum[NG];                     // sum_t p_t a_tg over this lane's rows
#pragma unroll
    for (int g = 0; g < NG; ++g) asum[g] = 0.0f;

    // One ring slot in three phases: scores of every tile, one softmax step, then the V
    // accumulation of every tile.  The tiles of a phase are independent, so their
    // latencies overlap.  MASK (the item's last slot, which reaches past t_end): rows at
    // or past t_end are masked, including whole tiles the copy skipped, whose stale bytes
    // are still finite codes and whose statistics are replaced by zeros.
    auto process = [&](const uint8_t* slot, int ts, auto mask_tag) {
      constexpr bool MASK = decltype(mask_tag)::value;
      auto valid = [&](int sub, int r) {
        return !MASK || ts + sub * kTile + gid + 8 * r < it.t_end;
      };
      // ---- phase 1: scores, K codes (rows t) x permuted q
      float sc[kSub][2];
#pragma unroll
      for (int sub = 0; sub < kSub; ++sub) {
        uint32_t kw[2][NW], ka[2][NG];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int row = sub * kTile + gid + 8 * r;
          load_words<NW>(slot + row * R::ROW_CODE + tig * 4 * NW, kw[r]);
          load_words<NG>(slot + R::KAB_OFF + row * R::ROW_AB, ka[r]);
        }
        float t_sc[2];
        q4attn::tile_scores<D>(kw, ka, qf, t_sc);
        sc[sub][0] = valid(sub, 0) ? t_sc[0] : -INFINITY;
        sc[sub][1] = valid(sub, 1) ? t_sc[1] : -INFINITY;
        if constexpr (SC) {
          // every lane of a row holds its score; lane tig == 0 stores it
          if (tig == 0) {
            uint32_t* kr = keys + ((int64_t)it.b * H + it.hd) * len + ts + sub * kTile;
            if (valid(sub, 0)) kr[gid] = q4attn::order_key_f32(t_sc[0]);
            if (valid(sub, 1)) kr[gid + 8] = q4attn::order_key_f32(t_sc[1]);
          }
        }
      }
      // ---- phase 2: lazy rescaling: the reference maximum moves only when a score
      // exceeds it by more than 2^8, so p stays <= 256 and the accumulators rarely need
      // scaling; the warp maximum is taken only then
      float mloc = fmaxf(sc[0][0], sc[0][1]);
#pragma unroll
      for (int sub = 1; sub < kSub; ++sub) mloc = fmaxf(mloc, fmaxf(sc[sub][0], sc[sub][1]));
      if (__any_sync(0xFFFFFFFFu, mloc > m_run + 8.0f)) {
        float mx = mloc;
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
        const float corr = (m_run == -INFINITY) ? 0.0f : ex2(m_run - mx);
        l_run *= corr;
#pragma unroll
        for (int u = 0; u < 2 * NW; ++u)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[u][c] *= corr;
#pragma unroll
        for (int g = 0; g < NG; ++g) asum[g] *= corr;
        m_run = mx;
      }
      // invalid rows hold -inf scores, and ex2(-inf) = 0
      float p[kSub][2];
#pragma unroll
      for (int sub = 0; sub < kSub; ++sub) {
        p[sub][0] = ex2(sc[sub][0] - m_run);
        p[sub][1] = ex2(sc[sub][1] - m_run);
        l_run += p[sub][0] + p[sub][1];
      }
      // ---- phase 3: V weights w_tg = p_t (b - a)_tg / 15 (fp16), the offset term
      // sum_t p_t a_tg, and the V codes (channel rows, position columns)
      if constexpr (!SC) {
#pragma unroll
      for (int sub = 0; sub < kSub; ++sub) {
        uint32_t vw[2][NW], va[2][NG];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int row = sub * kTile + gid + 8 * r;
          load_words<NW>(slot + R::CODE_BYTES + row * R::ROW_CODE + tig * 4 * NW, vw[r]);
          load_words<NG>(slot + 2 * R::CODE_BYTES + R::AB_BYTES + row * R::ROW_AB, va[r]);
        }
        const bool vr[2] = {valid(sub, 0), valid(sub, 1)};
        q4attn::v_tile<D>(vw, va, p[sub], vr, lane, acc, asum);
      }
      }
    };

    for (int j = 0; j < it.nslots; ++j) {
      ok = __all_sync(0xFFFFFFFFu, bar_wait(bar0 + 8 * cs, cph));
      if (!ok) break;
      const uint8_t* slot = ring + cs * R::SLOT;
      const int ts = it.t_begin + j * kSlotPos;
      if (ts + kSlotPos <= it.t_end)
        process(slot, ts, std::false_type{});
      else
        process(slot, ts, std::true_type{});
      // every lane has consumed the words it loaded from this slot: refill it kRing slots
      // ahead (releasing it any earlier would let the copy race the slot's last readers)
      __syncwarp();
      if (lane == 0) issue();
      ++consumed;
      if (++cs == kRing) {
        cs = 0;
        cph ^= 1u;
      }
    }
    if (!ok) break;

    // ---- epilogue of the item: o_j = (acc + sum_t p_t a_tg) / l
    float l = l_run;
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 4);
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 8);
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 16);
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      asum[g] += __shfl_xor_sync(0xFFFFFFFFu, asum[g], 4);
      asum[g] += __shfl_xor_sync(0xFFFFFFFFu, asum[g], 8);
      asum[g] += __shfl_xor_sync(0xFFFFFFFFu, asum[g], 16);
    }
    if constexpr (SC) {
      if (lane == 0) ml[ci] = make_float2(m_run, l);
      __syncwarp();
      continue;
    }
    const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
    uint16_t* o = out + (int64_t)it.b * H * D + (int64_t)it.hd * D;
    float* pp = partial + (int64_t)ci * (D + 2);
    if (splits == 1)
      q4attn::v_channels<D>(acc, asum, lane, [&](int ch, float v) { o[ch] = f2h(v * inv_l); });
    else
      q4attn::v_channels<D>(acc, asum, lane, [&](int ch, float v) { pp[ch] = v; });
    if (splits > 1 && lane == 0) {
      pp[D] = m_run;
      pp[D + 1] = l;
    }
    __syncwarp();
  }

  // ---- drain: every issued copy must land before the warp's shared memory is released
  if (lane == 0) {
    for (int g = consumed; g < issued; ++g) {
      const uint32_t bar = bar0 + 8 * (uint32_t)(g % kRing);
      const long long t0 = clock64();
      while (!bar_try(bar, (uint32_t)((g / kRing) & 1))) {
        if (clock64() - t0 > kWaitCycles) {
          atomicOr(&g_attn_error, 2u);
          break;
        }
      }
    }
  }
}

// One warp per (b, hd): merge the split partials (m, l, unnormalised o) in base 2.
template <int D>
__global__ void __launch_bounds__(128)
decode_combine_kernel(const float* __restrict__ partial, int64_t nbh, int H, int splits,
                      uint16_t* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
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

template <int D, bool SC>
int resident_ctas() {
  static int occ = [] {
    int n = 0;
    // the rings exceed the 48 KB default; prefer the carveout that admits the most CTAs
    cudaFuncSetAttribute(decode_attn_kernel<D, SC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Ring<D, SC>::CTA_BYTES);
    cudaFuncSetAttribute(decode_attn_kernel<D, SC>,
                         cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_attn_kernel<D, SC>, kWarps * 32,
                                                      Ring<D, SC>::CTA_BYTES) != cudaSuccess ||
        n < 1)
      n = 1;
    return n;
  }();
  return occ;
}

}  // namespace

// Sequence splits: the fewest that minimise the busiest warp's work, with the resident
// warps (nsm * kPlanWarpsPerSm) taking items round-robin.  Work is counted in tiles: an
// item costs about one tile more than its tiles (q preparation and its epilogue), and
// splitting about four (the partials and the combine kernel).
static int plan_splits(const fg_kvcache& kv, int32_t len, int nsm) {
  const int64_t bh = (int64_t)kv.B * kv.H;
  if (bh == 0) return 1;
  const int ntiles = (len + kTile - 1) / kTile;
  const int64_t warps = (int64_t)std::max(nsm, 1) * kPlanWarpsPerSm;
  int best = 1;
  int64_t best_cost = -1;
  for (int s = 1; s <= std::min(ntiles, 16); ++s) {
    const int tps = (ntiles + s - 1) / s;
    if (s > 1 && (s - 1) * tps >= ntiles) break;           // an empty split
    const int64_t rounds = (bh * s + warps - 1) / warps;
    const int64_t cost = rounds * (tps + 1) + (s > 1 ? 4 : 0);
    if (best_cost < 0 || cost < best_cost) {
      best = s;
      best_cost = cost;
    }
  }
  const int tps = (ntiles + best - 1) / best;
  return (ntiles + tps - 1) / tps;
}

// The device's plan, capped by the plan for kMaxSms SMs: the workspace query sizes for the
// latter, and partial bytes grow with the split count.
int decode_attn_splits(const fg_kvcache& kv, int32_t len, int nsm) {
  return std::min(plan_splits(kv, len, nsm), plan_splits(kv, len, kMaxSms));
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
  if (items >= (1ll << 31)) return cudaErrorInvalidValue;   // work items are 32-bit
  const float sl2 = scale * 1.4426950408889634f;
  float* partial = static_cast<float*>(ws);
  const int64_t want = (items + kWarps - 1) / kWarps;
  if (d == 128) {
    const unsigned grid =
        (unsigned)std::min<int64_t>(want, (int64_t)nsm * resident_ctas<128, false>());
    cudaError_t e0 = launch_pdl(decode_attn_kernel<128, false>, dim3(grid), dim3(kWarps * 32),
                                Ring<128, false>::CTA_BYTES, st, q, q_stride, kv.k_codes,
                                kv.v_codes, kv.k_ab, kv.v_ab, kv.B, kv.H, kv.cap, len, splits, tps,
                                sl2, out, partial, nullptr, nullptr);
    if (e0 != cudaSuccess) return e0;
  } else {
    const unsigned grid =
        (unsigned)std::min<int64_t>(want, (int64_t)nsm * resident_ctas<64, false>());
    cudaError_t e0 = launch_pdl(decode_attn_kernel<64, false>, dim3(grid), dim3(kWarps * 32),
                                Ring<64, false>::CTA_BYTES, st, q, q_stride, kv.k_codes,
                                kv.v_codes, kv.k_ab, kv.v_ab, kv.B, kv.H, kv.cap, len, splits, tps,
                                sl2, out, partial, nullptr, nullptr);
    if (e0 != cudaSuccess) return e0;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *kernels_out = 1;
  if (splits > 1) {
    if (mid_event) cudaEventRecord(mid_event, st);
    const int64_t nbh = (int64_t)kv.B * kv.H;
    const unsigned g2 = (unsigned)((nbh + 3) / 4);
    if (d == 128)
      e = launch_pdl(decode_combine_kernel<128>, dim3(g2), dim3(128), 0, st, partial, nbh, kv.H,
                     splits, out);
    else
      e = launch_pdl(decode_combine_kernel<64>, dim3(g2), dim3(128), 0, st, partial, nbh, kv.H,
                     splits, out);
    *kernels_out = 2;
  }
  return e;
}

cudaError_t launch_decode_attn_scores(const uint16_t* q, int64_t q_stride, const fg_kvcache& kv,
                                      int32_t len, float scale, uint32_t* keys, float2* ml,
                                      int nsm, cudaStream_t st, int* splits_out) {
  const int d = kv.h / kv.H;
  const int splits = decode_attn_splits(kv, len, nsm);
  const int ntiles = (len + kTile - 1) / kTile;
  const int tps = (ntiles + splits - 1) / splits;
  const int64_t items = (int64_t)kv.B * kv.H * splits;
  if (items >= (1ll << 31)) return cudaErrorInvalidValue;   // work items are 32-bit
  *splits_out = splits;
  const float sl2 = scale * 1.4426950408889634f;
  const int64_t want = (items + kWarps - 1) / kWarps;
  if (d == 128) {
    const unsigned grid =
        (unsigned)std::min<int64_t>(want, (int64_t)nsm * resident_ctas<128, true>());
    return launch_pdl(decode_attn_kernel<128, true>, dim3(grid), dim3(kWarps * 32),
                      Ring<128, true>::CTA_BYTES, st, q, q_stride, kv.k_codes, kv.v_codes,
                      kv.k_ab, kv.v_ab, kv.B, kv.H, kv.cap, len, splits, tps, sl2,
                      (uint16_t*)nullptr, (float*)nullptr, keys, ml);
  }
  const unsigned grid =
      (unsigned)std::min<int64_t>(want, (int64_t)nsm * resident_ctas<64, true>());
  return launch_pdl(decode_attn_kernel<64, true>, dim3(grid), dim3(kWarps * 32),
                    Ring<64, true>::CTA_BYTES, st, q, q_stride, kv.k_codes, kv.v_codes, kv.k_ab,
                    kv.v_ab, kv.B, kv.H, kv.cap, len, splits, tps, sl2, (uint16_t*)nullptr,
                    (float*)nullptr, keys, ml);
}

cudaError_t attn_read_error(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_attn_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_attn_error, &zero, sizeof(unsigned int));
}

}  // namespace fg
