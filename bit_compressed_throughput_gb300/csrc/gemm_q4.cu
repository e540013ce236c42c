// Dequant-fused GEMM on the 5th-generation tensor cores (sm_103a):
//   Y[M][N] = epi( X[M][K] * W^[K][N] + bias )
// where W^ is restored to fp16 from 4-bit codes grouped 64 along the output channel N
// with per-group (a, b) [FlexGen review (jaehun.me), "4-bit 압축은 정수 연산 가속과 같은가":
// weights grouped along the output channel, restored to FP16 before compute, no INT4
// matmul].  The block schedule's batch reuse makes the projections and the MLP dense
// contractions over M = g*s (prefill) or M = B (decode) rows.
//
// Persistent kernel: one CTA per SM loops over output tiles 128 x 256 (K step 64).
//   warp 0      TMA producer: X tile (128B swizzle, K-major), packed code tile (128B
//               swizzle) and the tile's group statistics, one transaction per stage, into a
//               6-deep ring; owns the TMEM allocation (512 columns)
//   warp 1      one thread issues tcgen05.mma (kind::f16, M=128, N=256, K=16) into one of
//               two double-buffered 128 x 256 fp32 accumulators and commits to mbarriers
//   warps 2-9   restore codes -> fp16 B tile in a 2-deep shared-memory ring (MN-major,
//               128B swizzle: one k-row of 64 output channels = one 128-byte swizzle row =
//               one group); two restore warps per SM sub-partition hide each other's
//               latency
//   warps 10-13 epilogue of the previous tile (tcgen05.ld, bias / ReLU / residual, fp16
//               store) while the other accumulator fills
// The restore, not the MMA, bounds this kernel: with the restore skipped the same
// pipeline runs at about 84% of the measured dense fp16 peak.
// Restoration per pair of codes: the nibble is OR-ed into mantissa bits 6..9 of 1.0h so
// that the half equals 1 + q/16, then one HFMA2 gives (1 + q/16)*(16s) + (a - 16s) = a + q*s.
// Within each 8-channel chunk the pairs land as (n0,n4,n1,n5,n2,n6,n3,n7); the epilogue
// undoes that order when it packs the accumulator columns back to fp16.
//
// Small M (decode) also splits K: work units are (split, tile); partial fp32 tiles go to
// the caller's workspace and a reduce kernel applies the epilogue.
//
// Every mbarrier wait is bounded (about 2 s); on timeout the CTA raises an abort flag,
// sets the device error word, drains its outstanding copies and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {

__device__ unsigned int g_gemm_error = 0;

namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int UM = 128;                     // rows per MMA
constexpr int RS = 6;                       // raw ring: X tile + code tile
constexpr int BS = 2;                       // restored B ring
constexpr int RW = 8;                       // restore warps
constexpr int RT = RW * 32;                 // restore threads
constexpr int EW0 = 2 + RW;                 // first epilogue warp
constexpr int THREADS = (EW0 + 4) * 32;
constexpr int ITEMS = BK * BN / 32 / RT;    // 16-byte code chunks per restore thread
constexpr int A_BYTES = BM * BK * 2;        // 16 KB
constexpr int B_BYTES = BK * BN * 2;        // 32 KB
constexpr int C_BYTES = BK * BN / 2;        // 8 KB of codes (128-byte rows)
constexpr int S_BYTES = BK * (BN / 64) * 4;  // 1 KB of (a, b) words
constexpr int SMEM_BYTES = RS * (A_BYTES + C_BYTES + S_BYTES) + BS * B_BYTES +
                           1024 /*align*/ + 256 /*barriers*/;
constexpr uint32_t TMEM_COLS = 2 * (BM / UM) * BN;   // two accumulator buffers
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(TMEM_COLS == 512, "TMEM budget");
static_assert(ITEMS * RT * 32 == BK * BN, "restore coverage");
constexpr long long kWaitCycles = 1ll << 32;
constexpr int SWZ_GROUP_M = 8;

// instruction descriptor: D f32, A f16 K-major, B f16 MN-major, N = 256, M = 128
constexpr uint32_t IDESC = (1u << 4) | (1u << 16) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(UM >> 4) << 24);

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait.  Returns false (and raises the CTA abort flag) on timeout or when another
// warp already aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      atomicOr(&g_gemm_error, 1u);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x),
      "r"(y), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor: start, leading / stride byte offsets (>> 4), the
// descriptor version bit of this architecture, 128-byte swizzle layout.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t x, uint32_t s, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&x), *reinterpret_cast<__half2*>(&s),
                      *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Restore 8 codes (one word) of one group to 4 half2 in (n0,n4),(n1,n5),(n2,n6),(n3,n7).
__device__ __forceinline__ uint4 restore8(uint32_t w, uint32_t s16, uint32_t c) {
  uint4 o;
  o.x = hfma2_u32(((w << 6) & 0x03C003C0u) | 0x3C003C00u, s16, c);
  o.y = hfma2_u32(((w << 2) & 0x03C003C0u) | 0x3C003C00u, s16, c);
  o.z = hfma2_u32(((w >> 2) & 0x03C003C0u) | 0x3C003C00u, s16, c);
  o.w = hfma2_u32(((w >> 6) & 0x03C003C0u) | 0x3C003C00u, s16, c);
  return o;
}

struct EpiArgs {
  const uint16_t* bias;
  const uint16_t* residual;
  uint16_t* Y;
  float* partial;     // split-K: [splits][M][N] fp32, else null
  int epi;
};

// Bias / ReLU / residual on 8 consecutive outputs and the fp16 store.
__device__ __forceinline__ void epilogue8(const EpiArgs& ea, float (&v)[8], int64_t row, int n,
                                          int N) {
  if (ea.bias) {
    const uint4 bu = ldg_nc_v4(ea.bias + n);
    const uint32_t bw[4] = {bu.x, bu.y, bu.z, bu.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = unpack_h2(bw[i]);
      v[2 * i] += f.x;
      v[2 * i + 1] += f.y;
    }
  }
  if (ea.epi == FG_EPI_RELU) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = fmaxf(v[i], 0.0f);
  } else if (ea.epi == FG_EPI_RESIDUAL) {
    const uint4 ru = *reinterpret_cast<const uint4*>(ea.residual + row * N + n);
    const uint32_t rw[4] = {ru.x, ru.y, ru.z, ru.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = unpack_h2(rw[i]);
      v[2 * i] += f.x;
      v[2 * i + 1] += f.y;
    }
  }
  uint4 o;
  o.x = pack_h2(v[0], v[1]);
  o.y = pack_h2(v[2], v[3]);
  o.z = pack_h2(v[4], v[5]);
  o.w = pack_h2(v[6], v[7]);
  *reinterpret_cast<uint4*>(ea.Y + row * N + n) = o;
}

__device__ __forceinline__ void unit_coords(int u, int tiles_m, int tiles_n, int kblocks,
                                            int kb_per_split, int& m0, int& n0, int& split,
                                            int& kb_begin, int& kb_end) {
  const int tiles = tiles_m * tiles_n;
  split = u / tiles;
  const int lin = u - split * tiles;
  // grouped raster: SWZ_GROUP_M m-tiles share a wave of n-tiles
  const int group_span = SWZ_GROUP_M * tiles_n;
  const int grp = lin / group_span;
  const int first_m = grp * SWZ_GROUP_M;
  const int gm = min(SWZ_GROUP_M, tiles_m - first_m);
  const int within = lin - grp * group_span;
  m0 = (first_m + within % gm) * BM;
  n0 = (within / gm) * BN;
  kb_begin = split * kb_per_split;
  kb_end = min(kblocks, kb_begin + kb_per_split);
}

__global__ void __launch_bounds__(THREADS, 1)
gemm_q4_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmC,
                  const __grid_constant__ CUtensorMap tmS, int M, int N, int K, int tiles_m, int tiles_n,
                  int kblocks, int kb_per_split, int units, EpiArgs ea) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;                                  // RS x A_BYTES
  uint8_t* sC = sA + RS * A_BYTES;                     // RS x C_BYTES
  uint8_t* sB = sC + RS * C_BYTES;                     // BS x B_BYTES
  uint32_t* sS = reinterpret_cast<uint32_t*>(sB + BS * B_BYTES);    // RS x 256 words
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + BS * B_BYTES + RS * S_BYTES);
  // bars: full_raw[RS], empty_raw[RS], full_b[BS], empty_b[BS], acc_full[2], acc_empty[2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * RS + 2 * BS + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(bars);
  auto full_raw = [&](int s) { return bar0 + 8u * s; };
  auto empty_raw = [&](int s) { return bar0 + 8u * (RS + s); };
  auto full_b = [&](int s) { return bar0 + 8u * (2 * RS + s); };
  auto empty_b = [&](int s) { return bar0 + 8u * (2 * RS + BS + s); };
  auto acc_full = [&](int s) { return bar0 + 8u * (2 * RS + 2 * BS + s); };
  auto acc_empty = [&](int s) { return bar0 + 8u * (2 * RS + 2 * BS + 2 + s); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < RS; ++s) {
      mbar_init(full_raw(s), 1);
      mbar_init(empty_raw(s), 1);
    }
    for (int s = 0; s < BS; ++s) {
      mbar_init(full_b(s), RT);                    // every restore thread arrives
      mbar_init(empty_b(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(acc_full(s), 1);
      mbar_init(acc_empty(s), 4);                  // one arrival per epilogue warp
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        int m0, n0, split, kbb, kbe;
        unit_coords(u, tiles_m, tiles_n, kblocks, kb_per_split, m0, n0, split, kbb, kbe);
        for (int kb = kbb; kb < kbe; ++kb, ++it) {
          const int s = it % RS;
          if (it >= RS && !mbar_wait(empty_raw(s), ((it / RS) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(full_raw(s), A_BYTES + C_BYTES + S_BYTES);
          tma_load_2d(smem_u32(sA + s * A_BYTES), &tmA, kb * BK, m0, full_raw(s));
          tma_load_2d(smem_u32(sC + s * C_BYTES), &tmC, n0 / 2, kb * BK, full_raw(s));
          tma_load_2d(smem_u32(sS + s * (S_BYTES / 4)), &tmS, n0 / 64, kb * BK, full_raw(s));
        }
      }
      // Drain: every issued load must have landed before this CTA can exit.
      for (int i = max(0, it - RS); i < it; ++i) {
        const long long t0 = clock64();
        while (!mbar_try(full_raw(i % RS), (i / RS) & 1)) {
          if (clock64() - t0 > kWaitCycles) {
            atomicOr(&g_gemm_error, 2u);
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0, tl = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++tl) {
        int m0, n0, split, kbb, kbe;
        unit_coords(u, tiles_m, tiles_n, kblocks, kb_per_split, m0, n0, split, kbb, kbe);
        const int acc = tl & 1;
        if (tl >= 2 && !mbar_wait(acc_empty(acc), ((tl >> 1) & 1) ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t tacc = tmem + acc * ((BM / UM) * BN);
        for (int kb = kbb; kb < kbe; ++kb, ++it) {
          const int s = it % RS, bs = it % BS;
          if (!mbar_wait(full_raw(s), (it / RS) & 1, abort_flag) ||
              !mbar_wait(full_b(bs), (it / BS) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + s * A_BYTES);
          const uint32_t b_base = smem_u32(sB + bs * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bd = smem_desc(b_base + kk * 16 * 128, 64 * 128, 1024);
            const uint32_t accum = (kb > kbb || kk > 0) ? 1u : 0u;
#pragma unroll
            for (int hh = 0; hh < BM / UM; ++hh) {
              if (m0 + hh * UM >= M) break;         // rows past M: nothing to compute
              const uint64_t ad = smem_desc(a_base + hh * (UM * 128) + kk * 32, 16, 1024);
              umma_f16(tacc + hh * BN, ad, bd, accum);
            }
          }
          umma_commit(empty_raw(s));
          umma_commit(empty_b(bs));
        }
        umma_commit(acc_full(acc));
      }
    }
  } else if (warp < EW0) {
    // ------------------------------------------------------------ restore codes -> B
    const int tid = threadIdx.x - 64;                 // 0 .. RT-1
    // items of this thread: k-row and 16-byte code chunk c (32 output channels) of the
    // 64 x 256 tile; 8 consecutive lanes take 8 consecutive k at one c, which keeps the
    // swizzled code loads, the statistics loads and the swizzled B stores free of bank
    // conflicts
    int ik[ITEMS], ic[ITEMS];
#pragma unroll
    for (int t = 0; t < ITEMS; ++t) {
      const int item = t * RT + tid;
      ik[t] = (item & 7) | (((item >> 6) & 7) << 3);
      ic[t] = (item >> 3) & 7;
    }
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      int m0, n0, split, kbb, kbe;
      unit_coords(u, tiles_m, tiles_n, kblocks, kb_per_split, m0, n0, split, kbb, kbe);
      for (int kb = kbb; kb < kbe; ++kb, ++it) {
        const int s = it % RS, bs = it % BS;
        if (!mbar_wait(full_raw(s), (it / RS) & 1, abort_flag) ||
            (it >= BS && !mbar_wait(empty_b(bs), ((it / BS) & 1) ^ 1, abort_flag))) {
          ok = false;
          break;
        }
        const uint8_t* cs = sC + s * C_BYTES;
        const uint32_t* ss = sS + s * (S_BYTES / 4);
        uint8_t* bsm = sB + bs * B_BYTES;
#pragma unroll
        for (int t = 0; t < ITEMS; ++t) {
          const int k = ik[t], c = ic[t], sw = k & 7;
          const uint4 cw = *reinterpret_cast<const uint4*>(cs + k * 128 + ((c ^ sw) << 4));
          const float2 abf = unpack_h2(ss[k * (BN / 64) + (c >> 1)]);
          const float sc16 = (abf.y - abf.x) * (16.0f / 15.0f);
          const uint32_t s16 = pack_h2(sc16, sc16);
          const float cf = abf.x - sc16;
          const uint32_t cc = pack_h2(cf, cf);
          uint8_t* brow = bsm + (c >> 1) * (BK * 128) + k * 128;
          const int jc0 = (c & 1) * 4;
          *reinterpret_cast<uint4*>(brow + (((jc0 + 0) ^ sw) << 4)) = restore8(cw.x, s16, cc);
          *reinterpret_cast<uint4*>(brow + (((jc0 + 1) ^ sw) << 4)) = restore8(cw.y, s16, cc);
          *reinterpret_cast<uint4*>(brow + (((jc0 + 2) ^ sw) << 4)) = restore8(cw.z, s16, cc);
          *reinterpret_cast<uint4*>(brow + (((jc0 + 3) ^ sw) << 4)) = restore8(cw.w, s16, cc);
        }
        // make the stores visible to the tensor core's (async) proxy, then arrive
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(full_b(bs));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int lane_base = 32 * (warp & 3);            // TMEM lanes this warp may read
    int tl = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++tl) {
      int m0, n0, split, kbb, kbe;
      unit_coords(u, tiles_m, tiles_n, kblocks, kb_per_split, m0, n0, split, kbb, kbe);
      const int acc = tl & 1;
      if (!mbar_wait(acc_full(acc), (tl >> 1) & 1, abort_flag)) break;
      __syncwarp();
      tc_fence_after();
      for (int hh = 0; hh < BM / UM; ++hh) {
      const int64_t row = (int64_t)m0 + hh * UM + lane_base + lane;
      const bool row_ok = row < M;
      for (int cc = 0; cc < BN / 32; ++cc) {
        const int nb = n0 + cc * 32;
        // loads that do not depend on the accumulator go first
        uint4 bias4[4], res4[4];
        if (!ea.partial && nb < N) {
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            bias4[g8] = ea.bias ? ldg_nc_v4(ea.bias + nb + g8 * 8) : make_uint4(0, 0, 0, 0);
            res4[g8] = (ea.epi == FG_EPI_RESIDUAL && row_ok)
                           ? *reinterpret_cast<const uint4*>(ea.residual + row * N + nb + g8 * 8)
                           : make_uint4(0, 0, 0, 0);
          }
        }
        uint32_t r[32];
        const uint32_t taddr =
            tmem + ((uint32_t)lane_base << 16) + acc * ((BM / UM) * BN) + hh * BN + cc * 32;
        __syncwarp();
        tmem_ld16(taddr, r);
        tmem_ld16(taddr + 16, r + 16);
        tmem_wait_ld();
        if (!row_ok || nb >= N) continue;
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8) {
          const int n = nb + g8 * 8;
          float v[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v[i] = __uint_as_float(r[8 * g8 + 2 * i]);
            v[i + 4] = __uint_as_float(r[8 * g8 + 2 * i + 1]);
          }
          if (ea.partial) {
            float* pp = ea.partial + ((int64_t)split * M + row) * N + n;
            reinterpret_cast<float4*>(pp)[0] = make_float4(v[0], v[1], v[2], v[3]);
            reinterpret_cast<float4*>(pp)[1] = make_float4(v[4], v[5], v[6], v[7]);
            continue;
          }
          const uint32_t bw[4] = {bias4[g8].x, bias4[g8].y, bias4[g8].z, bias4[g8].w};
          const uint32_t rw[4] = {res4[g8].x, res4[g8].y, res4[g8].z, res4[g8].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 fb = unpack_h2(bw[i]), fr = unpack_h2(rw[i]);
            v[2 * i] += fb.x + fr.x;
            v[2 * i + 1] += fb.y + fr.y;
          }
          if (ea.epi == FG_EPI_RELU) {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = fmaxf(v[i], 0.0f);
          }
          uint4 o;
          o.x = pack_h2(v[0], v[1]);
          o.y = pack_h2(v[2], v[3]);
          o.z = pack_h2(v[4], v[5]);
          o.w = pack_h2(v[6], v[7]);
          *reinterpret_cast<uint4*>(ea.Y + row * N + n) = o;
        }
      }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(acc));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                 : "memory");
  }
}

// Sum the split-K partials and apply bias / ReLU / residual: 8 outputs per thread.
__global__ void __launch_bounds__(256)
gemm_reduce_kernel(const float* __restrict__ partial, int splits, int64_t M, int N, EpiArgs ea) {
  const int64_t idx = (int64_t)blockIdx.x * 256 + threadIdx.x;
  const int64_t chunks = M * (N / 8);
  if (idx >= chunks) return;
  const int64_t row = idx / (N / 8);
  const int n = (int)(idx - row * (N / 8)) * 8;
  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < splits; ++s) {
    const float4* pp = reinterpret_cast<const float4*>(partial + ((int64_t)s * M + row) * N + n);
    const float4 x = pp[0], y = pp[1];
    v[0] += x.x; v[1] += x.y; v[2] += x.z; v[3] += x.w;
    v[4] += y.x; v[5] += y.y; v[6] += y.z; v[7] += y.w;
  }
  epilogue8(ea, v, row, n, N);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

cudaError_t get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

cudaError_t make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                        uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                        uint32_t box_outer, CUtensorMapSwizzle swz) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

GemmPlan gemm_plan(int64_t M, int64_t K, int64_t N, int nsm) {
  GemmPlan p{};
  p.M = M; p.N = N; p.K = K;
  p.tiles_m = (int)((M + BM - 1) / BM);
  p.tiles_n = (int)((N + BN - 1) / BN);
  p.kblocks = (int)((K + BK - 1) / BK);
  const int64_t tiles = (int64_t)p.tiles_m * p.tiles_n;
  int splits = 1;
  // Split K only when the tile grid leaves more than a quarter of the SMs idle, keeping
  // at least 8 k-blocks per split so the pipeline stays full.
  if (tiles > 0 && tiles * 4 < (int64_t)nsm * 3) {
    splits = (int)std::max<int64_t>(1, nsm / tiles);
    splits = std::min(splits, std::max(1, p.kblocks / 8));
  }
  p.kb_per_split = std::max(1, (p.kblocks + splits - 1) / splits);
  p.splits = std::max(1, (p.kblocks + p.kb_per_split - 1) / p.kb_per_split);
  p.ws_bytes = (p.splits > 1) ? (size_t)p.splits * M * N * sizeof(float) : 0;
  p.units = tiles * p.splits;
  p.grid = (int)std::min<int64_t>(p.units, nsm);
  return p;
}

cudaError_t launch_gemm(const GemmPlan& p, const uint16_t* X, const fg_q4mat& W,
                        const uint16_t* bias, int epi, const uint16_t* residual, uint16_t* Y,
                        void* ws, cudaStream_t st, cudaEvent_t mid_event) {
  if (p.M == 0) return cudaSuccess;
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  static cudaError_t attr_err = cudaFuncSetAttribute(
      gemm_q4_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap tmA, tmC, tmS;
  e = make_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X, (uint64_t)p.K, (uint64_t)p.M,
                  (uint64_t)p.K * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = make_map_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, W.codes, (uint64_t)(p.N / 2),
                  (uint64_t)p.K, (uint64_t)(p.N / 2), BN / 2, BK, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = make_map_2d(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT32, W.ab, (uint64_t)(p.N / 64),
                  (uint64_t)p.K, (uint64_t)(p.N / 64) * 4, BN / 64, BK,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  const EpiArgs final_ea{bias, residual, Y, nullptr, epi};
  EpiArgs ea = final_ea;
  if (p.splits > 1) ea.partial = static_cast<float*>(ws);
  gemm_q4_tc_kernel<<<(unsigned)p.grid, THREADS, SMEM_BYTES, st>>>(
      tmA, tmC, tmS, (int)p.M, (int)p.N, (int)p.K, p.tiles_m, p.tiles_n, p.kblocks,
      p.kb_per_split, (int)p.units, ea);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1) return e;
  if (mid_event) cudaEventRecord(mid_event, st);
  const int64_t chunks = p.M * (p.N / 8);
  gemm_reduce_kernel<<<(unsigned)((chunks + 255) / 256), 256, 0, st>>>(
      static_cast<const float*>(ws), p.splits, p.M, (int)p.N, final_ea);
  return cudaGetLastError();
}

cudaError_t gemm_read_error(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_gemm_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(unsigned int));
}

}  // namespace fg
