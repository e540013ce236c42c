// Dequant-fused GEMM on CTA pairs (sm_103a): the tiled product for more than 128 tokens,
// with each 2-CTA cluster sharing one tensor-core tile of 256 channels x up to 256 tokens.
//   Y[M][N] = epi( X[M][K] * W^[K][N] + bias ),  W^ restored from 4-bit codes grouped 64
//   along the output channel with per-group (a, b) [FlexGen review (jaehun.me), "4-bit
//   압축은 정수 연산 가속과 같은가"].
//
// As in gemm_q4.cu the tensor core computes Y^T = W^T X^T, restored weights as the MMA's A
// operand (MN-major, 128B swizzle) and activations as its B operand (K-major, 128B swizzle).
// A cluster of two CTAs on two SMs owns a tile of 256 output channels x tn = 2 tnh tokens
// (tnh <= 128, chosen per launch so that the tiles cover M with little padding: 144 tokens
// make one tile of 144):
//   CTA r (r = 0, 1) restores channels c0 + 128 r .. + 127 into its own shared memory (its
//   half of the MMA's M = 256) and loads tokens t0 + tnh r .. + tnh - 1 of X (its half of
//   the MMA's N = tn).  One thread of CTA 0 issues tcgen05.mma.cta_group::2: each SM's tensor
//   core multiplies its own A half by both B halves, so every SM reads from shared memory
//   its 16 KB A slot and its X half (16 KB at tnh = 128) per k-block, against 16 + 32 KB for
//   the 128 x 256 tile of one CTA, and each X element is loaded once per 256 channels instead
//   of once per 128.  Each CTA's TMEM holds its 128 channels x tn tokens of the accumulator,
//   which its own epilogue reads.
// Ring depths are set per launch: many token tiles (prefill) reuse each code tile from L2 and
// take 6 k-block slots and 4 code stages; one or two token tiles (decode) stream the 4-bit
// weights from HBM and take 12 code stages over 5 or 6 slots.
//
// Roles (16 warps per CTA; warp w issues on scheduler w % 4).  The MMA issuer shares its
// scheduler only with the two single-thread producers and one epilogue warp: with restore
// warps beside it, the four MMAs and the commit of a k-block took ~450 cycles to issue
// against ~365 here (measured on a GB300).
//   warp 1      CTA 0 only: issues the pair's MMAs (M = 256, N = tn, K = 16) and commits each
//               k-block to the k-block barrier of both CTAs
//   warp 5      TMA producer of this CTA's X half (tnh tokens x 64 k) into the k-block ring
//   warp 9      TMA producer of this CTA's code tiles and group statistics
//   warp 8      owns the pair's TMEM (tcgen05.alloc.cta_group::2, 512 columns = two
//               256-column accumulators)
//   warps 0, 2, 3, 4, 6, 7, 10, 11: four restore groups of two warps, group g restoring the
//               k-blocks it == g (mod 4) into A slot it % r, as in gemm_q4.cu; a group that has
//               written its slot and seen its CTA's X half land arrives, one arrival per warp,
//               on CTA 0's barrier of that k-block, which therefore completes when both CTAs'
//               A and X halves are in place
//   warps 12-15 epilogue of the previous tile from this CTA's TMEM (warp w reads lane quarter
//               w % 4), overlapped with the next tile through the double-buffered accumulator;
//               each warp arrives on CTA 0's accumulator-empty barrier when it has read its
//               lanes
// Each CTA drains its own TMA loads (they complete on its own barriers), CTA 0 waits for the
// last of its MMAs, and the pair meets at a cluster barrier before freeing TMEM together.
//
// Every mbarrier wait is bounded (about 2 s of clock64); on timeout the CTA raises its abort
// flag and sets the device error word (read by fg_check_device_error); the other CTA's waits
// then run out too, and both reach the final drain and cluster barrier.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "fg_common.cuh"
#include "fg_internal.h"
#include "gemm_tc.cuh"

namespace fg {

__device__ unsigned int g_gemm_pair_error = 0;

namespace {

constexpr int TCH = 128;                    // output channels per CTA (half of the MMA's M)
constexpr int TNH_MAX = 128;                // tokens per CTA (half of the MMA's N), run time
constexpr int ACC_COLS = 256;               // TMEM columns per accumulator buffer (N <= 256)
constexpr int BK = 64;
constexpr int R_MAX = 8;                    // k-block ring (A slot + X half), run-time depth
constexpr int RC_MAX = 16;                  // code ring (codes + group statistics), run time
constexpr int RW = 8;                       // restore warps
constexpr int RT = RW * 32;
constexpr int RG = 4;                       // restore groups
constexpr int RTG = RT / RG;                // threads per restore group (two warps)
constexpr int ITEMS = RG;                   // 16-byte code chunks per thread per k-block
constexpr int EW0 = 12;                     // first epilogue warp
constexpr int THREADS = 16 * 32;
constexpr int kMmaWarp = 1, kXWarp = 5, kCodeWarp = 9, kTmemWarp = 8;
// Restore warps 0, 2, 3, 4, 6, 7, 10, 11 -> restore index 0..7 (-1: another role).
__device__ __forceinline__ int restore_index(int warp) {
  switch (warp) {
    case 0: return 0;
    case 2: return 1;
    case 3: return 2;
    case 4: return 3;
    case 6: return 4;
    case 7: return 5;
    case 10: return 6;
    case 11: return 7;
    default: return -1;
  }
}
constexpr int W_BYTES = TCH * BK * 2;       // 16 KB restored A slot
constexpr int C_BYTES = BK * TCH / 2;       // 4 KB of codes (64-byte rows)
constexpr int S_BYTES = BK * 4 * 4;         // 1 KB: (a, b) words of 4 groups x 64 k-rows
constexpr int CS_BYTES = C_BYTES + S_BYTES; // one code stage
constexpr int SMEM_BYTES = 232448;          // the whole per-CTA budget
constexpr int BAR_BYTES = 1024;
constexpr int POOL_BYTES = SMEM_BYTES - 1024 /*align*/ - BAR_BYTES;
// barriers: full[R] (CTA 0: the k-block's A and X halves of both CTAs), xfull[R] (this CTA's
// X half landed), mma_done[R] (the k-block's MMAs done: slot reusable), full_c[RC], free_c[RC],
// acc_full[2], acc_empty[2] (CTA 0: both CTAs' epilogues read the accumulator), drain, and
// with fp16 weights afull[2][R] (this CTA's two 64-channel halves of the A slot landed)
// and uq_full[QD] (a unit-schedule ring entry published: the dynamic order below)
constexpr int QD = 16;
constexpr int NBARS = 5 * R_MAX + 2 * RC_MAX + 5 + QD;
constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;   // two accumulator buffers of 256 columns
constexpr int FULL_ARRIVALS = 2 * (RTG / 32);   // one per restore warp of a group, both CTAs
constexpr int EMPTY_ARRIVALS = 2 * 4;           // one per epilogue warp, both CTAs
static_assert(NBARS * 8 + 8 + QD * 4 <= BAR_BYTES, "barriers, TMEM slot, abort flag, schedule");
// Dynamic order: CTA 0's X producer runs at most R_MAX k-blocks ahead of the MMAs (slot
// reuse), which run at most 2 units ahead of both CTAs' epilogues (accumulator reuse), and
// every other role sits between the two; so the producer that publishes schedule entries is
// fewer than R_MAX + 3 entries (one unit holds at least one k-block) ahead of any reader, and
// a ring of QD entries is never overwritten before it is read nor waited on a lap early.
static_assert(QD >= R_MAX + 3, "unit schedule ring depth");
static_assert(W_BYTES % 1024 == 0, "128B-swizzled slots stay 1024-aligned");
static_assert(CS_BYTES % 512 == 0, "64B-swizzled code stages stay 512-byte aligned");
static_assert(RTG * ITEMS * 32 == BK * TCH, "restore coverage: 32 codes per item");
static_assert(RTG % 32 == 0, "restore groups are whole warps");
// Code stage c always goes to restore group c % RG, so a group waits on every lap of its
// stages in order.  Otherwise a group could wait on lap L of a stage whose lap L - 1 (another
// group's k-block) had not landed yet: a parity wait cannot tell lap L from lap L - 2 and
// would pass at once on stale codes (TMA loads complete in any order).
// (The host picks the code ring depth rc as a multiple of RG.)
static_assert(RC_MAX % RG == 0, "code ring depth in whole restore-group rounds");
static_assert(RG == kPairStageKb, "a code stage of several k-blocks gives one to each group");
static_assert((RG & (RG - 1)) == 0, "stage positions by mask");
// The A-slot waits need no such rule: MMAs complete in order, and with a ring depth r >= RG
// (checked on the host) a group has seen the MMAs of k-block it - RG - r done before it waits
// on those of it - r.
static_assert(TMEM_COLS == 512, "TMEM budget: two 256-column accumulators");
constexpr long long kWaitCycles = 1ll << 32;

// instruction descriptor: D f32, A and B f16, A MN-major, B K-major, M = 256 (the pair),
// N = tn (both CTAs' tokens)
__host__ __device__ constexpr uint32_t pair_idesc(int tn) {
  return (1u << 4) | (1u << 15) | ((uint32_t)(tn >> 3) << 17) | ((uint32_t)(2 * TCH >> 4) << 24);
}

__device__ __forceinline__ bool pwait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      atomicOr(&g_gemm_pair_error, 1u);
      return false;
    }
  }
  return true;
}

// Wait for a phase whatever the abort flag says (draining copies or MMAs in flight).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(&g_gemm_pair_error, 2u);
      return;
    }
  }
}

// Unit schedule (dynamic order): CTA 0 writes an entry of CTA 1's ring and arrives on its
// barrier with cluster-scope release; readers wait with cluster-scope acquire.
__device__ __forceinline__ void st_cluster_u32(uint32_t cl_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cl_addr), "r"(v) : "memory");
}
__device__ __forceinline__ void mbar_arrive_release_cluster(uint32_t cl_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cl_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_acq_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool uwait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const long long t0 = clock64();
  while (!mbar_try_acq_cluster(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      atomicOr(&g_gemm_pair_error, 4u);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void transpose8x8_h(uint32_t (&w)[4], int lane) {
  const bool b0 = lane & 1, b1 = lane & 2, b2 = lane & 4;
  const uint32_t sel = b0 ? 0x3276u : 0x5410u;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t x = __shfl_xor_sync(0xFFFFFFFFu, w[q], 1);
    w[q] = __byte_perm(w[q], x, sel);
  }
  {
    const uint32_t y0 = __shfl_xor_sync(0xFFFFFFFFu, b1 ? w[0] : w[1], 2);
    const uint32_t y1 = __shfl_xor_sync(0xFFFFFFFFu, b1 ? w[2] : w[3], 2);
    if (b1) { w[0] = y0; w[2] = y1; } else { w[1] = y0; w[3] = y1; }
  }
  {
    const uint32_t z0 = __shfl_xor_sync(0xFFFFFFFFu, b2 ? w[0] : w[2], 4);
    const uint32_t z1 = __shfl_xor_sync(0xFFFFFFFFu, b2 ? w[1] : w[3], 4);
    if (b2) { w[0] = z0; w[1] = z1; } else { w[2] = z0; w[3] = z1; }
  }
}

__device__ __forceinline__ uint32_t hadd2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hadd2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

struct PUnit {
  int t0, c0, split, kb_begin, kb_end;     // c0: the pair's first channel
};

struct PArgs {
  int M, N, K;
  int tiles_t, pairs, kblocks, kb_per_split, units;
  int tnh;             // tokens per CTA: a multiple of 8, <= 128 (the MMA's N = 2 tnh)
  int r;               // k-block ring depth, RG <= r <= R_MAX
  int rc;              // code ring depth in stages, <= RC_MAX (a multiple of RG when sk = 1)
  int sk;              // k-blocks per code stage: 1, or RG (whole stages in every unit)
  int xslot;           // bytes per X slot: tnh * 128 rounded up to 1024
  int grp;             // token tiles per raster group
  int w16;             // 1: A slots are loaded by TMA from restored fp16 weights (no restore)
  unsigned int* ctr;   // dynamic order: the launch's ticket counter (zeroed before the launch);
                       // null: static order
};

// Work unit u -> split, token tile, channel pair and k-block range.  Within a split the
// units run in raster groups of `grp` token tiles x every channel pair, token tile fastest:
// the clusters working at one time (76 on a GB300) cover grp token tiles and 76 / grp
// channel pairs, so each k-block of X is read from HBM once for 76 / grp clusters and each
// k-block of codes once for grp.
__device__ __forceinline__ PUnit pair_unit(int u, int tn, const PArgs& ka) {
  PUnit r;
  const int tiles = ka.tiles_t * ka.pairs;
  r.split = u / tiles;
  const int lin = u - r.split * tiles;
  const int span = ka.grp * ka.pairs;
  const int g = lin / span;
  const int first = g * ka.grp;
  const int gn = min(ka.grp, ka.tiles_t - first);
  const int within = lin - g * span;
  r.t0 = (first + within % gn) * tn;
  r.c0 = (within / gn) * (2 * TCH);
  r.kb_begin = r.split * ka.kb_per_split;
  r.kb_end = min(ka.kblocks, r.kb_begin + ka.kb_per_split);
  return r;
}


__global__ void __launch_bounds__(THREADS, 1)
gemm_q4_pair_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmC,
                    const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmA,
                    const PArgs ka, const EpiArgs ea) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int R = ka.r, RC = ka.rc, TNH = ka.tnh, TN = 2 * ka.tnh, XS = ka.xslot;
  const int SK = ka.sk, SB = ka.sk * CS_BYTES;         // code stage: SK k-blocks
  uint8_t* sW = smem;                                  // R x W_BYTES (restored weights)
  uint8_t* sX = sW + R * W_BYTES;                      // R x XS (this CTA's X half)
  uint8_t* sC = sX + R * XS;                           // RC x SB (SK codes, SK statistics)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + POOL_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* uq = abort_flag + 1;                   // unit schedule ring (QD entries)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int r) { return bar0 + 8u * r; };
  auto xfull = [&](int r) { return bar0 + 8u * (R_MAX + r); };
  auto mma_done = [&](int r) { return bar0 + 8u * (2 * R_MAX + r); };
  auto full_c = [&](int c) { return bar0 + 8u * (3 * R_MAX + c); };
  auto free_c = [&](int c) { return bar0 + 8u * (3 * R_MAX + RC_MAX + c); };
  auto acc_full = [&](int a) { return bar0 + 8u * (3 * R_MAX + 2 * RC_MAX + a); };
  auto acc_empty = [&](int a) { return bar0 + 8u * (3 * R_MAX + 2 * RC_MAX + 2 + a); };
  const uint32_t drain = bar0 + 8u * (3 * R_MAX + 2 * RC_MAX + 4);
  auto afull = [&](int hf, int r) { return bar0 + 8u * (3 * R_MAX + 2 * RC_MAX + 5 + hf * R_MAX + r); };
  auto uq_full = [&](int i) { return bar0 + 8u * (5 * R_MAX + 2 * RC_MAX + 5 + i); };

  if (threadIdx.x == 0) {
    for (int r = 0; r < R; ++r) {
      mbar_init(full(r), ka.w16 ? 2 : FULL_ARRIVALS);   // fp16 weights: one relay per CTA
      mbar_init(xfull(r), 1);
      mbar_init(mma_done(r), 1);
      mbar_init(afull(0, r), 1);
      mbar_init(afull(1, r), 1);
    }
    for (int c = 0; c < RC; ++c) {
      mbar_init(full_c(c), 1);
      mbar_init(free_c(c), SK * RTG);            // the SK groups of the stage's k-blocks
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full(a), 1);
      mbar_init(acc_empty(a), EMPTY_ARRIVALS);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < QD; ++i) mbar_init(uq_full(i), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kTmemWarp) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  // both CTAs' barriers are initialised and the pair's TMEM allocated before either CTA
  // touches the other's barriers
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();

  // Schedule position q -> work unit (ka.units: none left; -1: a wait gave up).  Static
  // order: cluster cl takes units cl, cl + ncl, ...  Dynamic order (prefill, many token
  // tiles): CTA 0's X producer takes the launch counter's next ticket when it starts a unit
  // and publishes it in both CTAs' ring entry q % QD; every role of both CTAs reads the same
  // sequence.  Tickets follow the raster order, so whatever the clusters' relative speeds
  // the units in flight stay one window of the raster, the window whose tiles L2 holds; in
  // static order a cluster that runs ahead drifts into the next raster window, and the
  // clusters sharing a tile no longer read it at the same time.
  auto unit_static = [&](int q) -> int {
    const int64_t u = cl + (int64_t)q * ncl;
    return u < ka.units ? (int)u : ka.units;
  };
  auto unit_fetch = [&](int q) -> int {                // CTA 0's X producer (one thread)
    if (!ka.ctr) return unit_static(q);
    const int u = (int)min(atomicAdd(ka.ctr, 1u), (unsigned)ka.units);
    const int i = q % QD;
    uq[i] = u;
    st_cluster_u32(mapa_shared(smem_u32((const void*)(uq + i)), 1), (uint32_t)u);
    mbar_arrive_release_cluster(mapa_shared(uq_full(i), 1));
    mbar_arrive(uq_full(i));
    return u;
  };
  auto unit_read = [&](int q) -> int {                 // one thread
    if (!ka.ctr) return unit_static(q);
    if (!uwait(uq_full(q % QD), (uint32_t)((q / QD) & 1), abort_flag)) return -1;
    return uq[q % QD];
  };
  auto unit_read_warp = [&](int q) -> int {            // the whole warp
    if (!ka.ctr) return unit_static(q);
    if (!__all_sync(0xFFFFFFFFu, uwait(uq_full(q % QD), (uint32_t)((q / QD) & 1), abort_flag)))
      return -1;
    return uq[q % QD];
  };

  if (warp == kXWarp || warp == kCodeWarp) {
    // ------------------------------------------------------------ TMA producers
    // this CTA's X half into the k-block ring, or its codes + statistics into the code ring
    if (lane == 0) {
      const bool is_x = (warp == kXWarp);
      const int depth = is_x ? R : RC;
      const int nunits = (is_x || !ka.w16) ? ka.units : 0;   // fp16 weights: no code copies
      const int step = is_x ? 1 : SK;                 // k-blocks per load (X) or stage (codes)
      int it = 0, s = 0;                              // loads issued; slot
      uint32_t ph = 0;                                // lap parity of slot s
      for (int q = 0; nunits > 0; ++q) {
        const int u = (is_x && rank == 0) ? unit_fetch(q) : unit_read(q);
        if (u < 0 || u >= ka.units) break;
        const PUnit w = pair_unit(u, TN, ka);
        const int c0 = w.c0 + (int)rank * TCH;
        bool ok = true;
        for (int kb = w.kb_begin; kb < w.kb_end; kb += step, ++it) {
          // a slot is free once the MMAs of k-block it - R are done (X); a code stage once
          // the restorers of the k-blocks of stage it - RC consumed it
          if (it >= depth && !pwait(is_x ? mma_done(s) : free_c(s), ph ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          if (is_x) {
            mbar_expect_tx(xfull(s), (uint32_t)(TNH * BK * 2));
            tma_load_2d(smem_u32(sX + s * XS), &tmX, kb * BK, w.t0 + (int)rank * TNH, xfull(s));
          } else {
            // one box of SK x 64 code rows and one of their statistics
            uint8_t* cs = sC + s * SB;
            mbar_expect_tx(full_c(s), (uint32_t)SB);
            tma_load_2d(smem_u32(cs), &tmC, c0 / 2, kb * BK, full_c(s));
            tma_load_2d(smem_u32(cs + SK * C_BYTES), &tmS, (c0 / 256) * 4, kb * BK, full_c(s));
          }
          if (++s == depth) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
      }
      // every load this thread issued lands on this CTA's own barrier: wait for the last
      // `depth` of them (earlier ones were waited for before their slots were reused)
      for (int i = max(0, it - depth); i < it; ++i)
        drain_wait(is_x ? xfull(i % depth) : full_c(i % depth), (uint32_t)((i / depth) & 1));
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (CTA 0)
    if (lane == 0 && rank == 0) {
      // descriptors of slot 0; a slot offset, and the K16 step, add (bytes >> 4) to the
      // start-address field (all addresses are below 256 KB)
      const uint64_t adesc0 = smem_desc(smem_u32(sW), 64 * 128, 1024);
      const uint64_t bdesc0 = smem_desc(smem_u32(sX), 16, 1024);
      const uint32_t idesc = pair_idesc(TN);
      int tl = 0, r = 0;
      uint32_t ph = 0;
      bool ok = true, issued = false;
      for (int q = 0; ok; ++q, ++tl) {
        const int u = unit_read(q);
        if (u < 0 || u >= ka.units) break;
        const PUnit w = pair_unit(u, TN, ka);
        const int acc = tl & 1;
        if (tl >= 2 && !pwait(acc_empty(acc), ((tl >> 1) & 1) ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t tacc = tmem + acc * ACC_COLS;
        uint32_t accumulate = 0u;
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if (!pwait(full(r), ph, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = adesc0 + (uint64_t)r * (W_BYTES >> 4);
          const uint64_t bd = bdesc0 + (uint64_t)r * (uint64_t)(XS >> 4);
          umma2_f16(tacc, ad, bd, idesc, accumulate);
          umma2_f16(tacc, ad + 128, bd + 2, idesc, 1u);
          umma2_f16(tacc, ad + 256, bd + 4, idesc, 1u);
          umma2_f16(tacc, ad + 384, bd + 6, idesc, 1u);
          umma2_commit_mc(mma_done(r), (uint16_t)0x3);
          issued = true;
          accumulate = 1u;
          if (++r == R) {
            r = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        umma2_commit_mc(acc_full(acc), (uint16_t)0x3);
      }
      // the pair frees TMEM only after every MMA this thread issued has completed
      if (issued) {
        umma2_commit_mc(drain, (uint16_t)0x1);
        drain_wait(drain, 0u);
      }
    }
  } else if (restore_index(warp) >= 0 && ka.w16) {
    // ------------------------------------------------------------ fp16 weights
    // Restore warp 0 relays, restore warps 1 and 2 load the two 64-channel halves of this
    // CTA's 128 channels x 64 k of restored weights into the A slot (the layout the restore
    // writes: two 8 KB halves, k-rows of 128 bytes, 128B swizzle), each copy on a barrier of
    // its own; a slot is refilled once the MMAs of k-block it - R are done.  The relay
    // arrives on CTA 0's barrier of a k-block once this CTA's X half and both A halves landed.
    const int ri = restore_index(warp);
    if (lane == 0 && ri <= 2) {
      int it = 0, r = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int q = 0; ok; ++q) {
        const int u = unit_read(q);
        if (u < 0 || u >= ka.units) break;
        const PUnit w = pair_unit(u, TN, ka);
        const int c0 = w.c0 + (int)rank * TCH;
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++it) {
          if (ri == 0) {
            if (!pwait(xfull(r), ph, abort_flag) || !pwait(afull(0, r), ph, abort_flag) ||
                !pwait(afull(1, r), ph, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_cluster(mapa_shared(full(r), 0));
          } else {
            const int hf = ri - 1;
            if (it >= R && !pwait(mma_done(r), ph ^ 1, abort_flag)) {
              ok = false;
              break;
            }
            mbar_expect_tx(afull(hf, r), (uint32_t)(W_BYTES / 2));
            tma_load_2d(smem_u32(sW + r * W_BYTES + hf * (W_BYTES / 2)), &tmA, c0 + 64 * hf,
                        kb * BK, afull(hf, r));
          }
          if (++r == R) {
            r = 0;
            ph ^= 1;
          }
        }
      }
      // every copy this thread issued lands on this CTA's own barrier before the CTA exits
      if (ri > 0)
        for (int i = max(0, it - R); i < it; ++i)
          drain_wait(afull(ri - 1, i % R), (uint32_t)((i / R) & 1));
    }
  } else if (restore_index(warp) >= 0) {
    // ------------------------------------------------------------ restore codes -> A
    // Item -> (k-row, 16-byte code chunk = 32 channels) as in gemm_q4.cu: each 8-lane phase
    // takes the two chunks of one 64-channel group on four k-rows whose (k & 3) differ and
    // whose (k & 1, k & 4) differ (conflict-free 64B-swizzled loads and 128B-swizzled stores).
    const int tid = 32 * restore_index(warp) + lane;
    const int grp = tid / RTG, tg = tid % RTG;
    int code_off[ITEMS], stat_k[ITEMS], w_off[ITEMS], sw[ITEMS], cl4[ITEMS];
#pragma unroll
    for (int t = 0; t < ITEMS; ++t) {
      const int item = tg + t * RTG;
      const int cbit = item & 1, rsel = (item >> 1) & 3, quad = (item >> 3) & 1;
      const int j = (item >> 4) & 1;
      const int k = (item >> 5) * 8 + (quad ? 2 + rsel : (rsel < 2 ? rsel : rsel + 4));
      const int c = 2 * j + cbit;
      code_off[t] = k * 64 + ((c ^ ((k >> 1) & 3)) << 4);
      stat_k[t] = k * 4 + j;
      w_off[t] = j * (BK * 128) + k * 128;
      sw[t] = k & 7;
      cl4[t] = cbit * 4;
    }
    int it = 0, c = 0, r = 0, rg = 0;
    uint32_t phc = 0, phr = 0;
    bool ok = true;
    for (int q = 0; ok; ++q) {
      const int u = unit_read_warp(q);
      if (u < 0 || u >= ka.units) break;
      const PUnit w = pair_unit(u, TN, ka);
      const int g0 = ((w.c0 + (int)rank * TCH) >> 6) & 3;   // first group in the stats box
      for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++it) {
        // code stage c holds SK consecutive k-blocks of the unit; this is its j-th.  With
        // SK = RG each group takes one k-block of every stage (it == g mod RG), so every group
        // waits on every lap of every stage in order
        const int j = (kb - w.kb_begin) & (SK - 1);
        const int cc_ = c, cr = r;
        const uint32_t cphc = phc, cphr = phr;
        const bool mine = (rg == grp);
        if (j == SK - 1 && ++c == RC) { c = 0; phc ^= 1; }
        if (++r == R) { r = 0; phr ^= 1; }
        if (++rg == RG) rg = 0;
        if (!mine) continue;
        if (!pwait(full_c(cc_), cphc, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* cs = sC + cc_ * SB + j * C_BYTES;
        const uint32_t* ss =
            reinterpret_cast<const uint32_t*>(sC + cc_ * SB + SK * C_BYTES + j * S_BYTES);
        uint4 cw[ITEMS];
        uint32_t abw[ITEMS];
#pragma unroll
        for (int t = 0; t < ITEMS; ++t) {
          cw[t] = *reinterpret_cast<const uint4*>(cs + code_off[t]);
          abw[t] = ss[stat_k[t] + g0];
        }
        // the A slot is free once the MMAs of k-block it - R are done
        if (it >= R && !pwait(mma_done(cr), cphr ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* wb = sW + cr * W_BYTES;
#pragma unroll
        for (int t = 0; t < ITEMS; ++t) {
          const float2 abf = unpack_h2(abw[t]);
          const float sc16 = (abf.y - abf.x) * (16.0f / 15.0f);
          const uint32_t s16 = pack_h2(sc16, sc16);
          const float cf = abf.x - sc16;
          const uint32_t ccst = pack_h2(cf, cf);
          uint8_t* wrow = wb + w_off[t];
          const int u0 = cl4[t], z = sw[t];
          *reinterpret_cast<uint4*>(wrow + (((u0 + 0) ^ z) << 4)) = restore8(cw[t].x, s16, ccst);
          *reinterpret_cast<uint4*>(wrow + (((u0 + 1) ^ z) << 4)) = restore8(cw[t].y, s16, ccst);
          *reinterpret_cast<uint4*>(wrow + (((u0 + 2) ^ z) << 4)) = restore8(cw[t].z, s16, ccst);
          *reinterpret_cast<uint4*>(wrow + (((u0 + 3) ^ z) << 4)) = restore8(cw[t].w, s16, ccst);
        }
        mbar_arrive(free_c(cc_));                     // the code stage's words are consumed
        // the restored stores become visible to the tensor core's (async) proxy; once this
        // CTA's X half of the k-block has landed too, one arrival per warp on CTA 0's
        // barrier of the k-block, whose MMA then makes this SM's tensor core read the slots
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        int good = 1;
        if (lane == 0) {
          good = pwait(xfull(cr), cphr, abort_flag) ? 1 : 0;
          if (good) mbar_arrive_cluster(mapa_shared(full(cr), 0));
        }
        if (!__shfl_sync(0xFFFFFFFFu, good, 0)) {
          ok = false;
          break;
        }
      }
    }
  } else if (warp >= EW0) {
    // ------------------------------------------------------------ epilogue
    // TMEM lane L of this CTA holds its restored row L: channel (L & ~7) + kPerm[L & 7] of
    // its 128, kPerm = (0,4,1,5,2,6,3,7); column n holds token t0 + n.
    const int lane_base = 32 * (warp & 3);
    const int L = lane_base + lane;
    const int ch_in_tile = (L & ~7) + ((L & 7) >> 1) + ((L & 1) << 2);
    const int64_t N = ka.N;
    const bool add_res = !ea.partial && ea.epi == FG_EPI_RESIDUAL;
    const uint32_t empty_cl[2] = {mapa_shared(acc_empty(0), 0), mapa_shared(acc_empty(1), 0)};
    int tl = 0;
    for (int q = 0;; ++q, ++tl) {
      const int u = unit_read_warp(q);
      if (u < 0 || u >= ka.units) break;
      const PUnit w = pair_unit(u, TN, ka);
      const int c0 = w.c0 + (int)rank * TCH;
      const int acc = tl & 1;
      const int ntok = min(TN, ka.M - w.t0);
      if (add_res) {
        for (int i = 32 * (warp & 3) + lane; i < 2 * ntok; i += 128)
          prefetch_l2(ea.residual + (int64_t)(w.t0 + (i >> 1)) * N + c0 + (i & 1) * 64);
      }
      // the warp-collective TMEM loads below need the whole warp: decide for all its lanes
      if (!__all_sync(0xFFFFFFFFu, pwait(acc_full(acc), (tl >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      const int64_t ch = c0 + ch_in_tile;
      const float bias_f = (!ea.partial && ea.bias) ? h2f(ea.bias[ch]) : 0.0f;
      const int64_t chb = c0 + lane_base + (lane & ~7);
      for (int cb = 0; cb < ntok; cb += 32) {
        uint32_t r[32];
        __syncwarp();
        const uint32_t taddr = tmem + ((uint32_t)lane_base << 16) + acc * ACC_COLS + cb;
        tmem_ld16(taddr, r);
        tmem_ld16(taddr + 16, r + 16);
        tmem_wait_ld();
        if (ea.partial) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (cb + i >= ntok) break;
            ea.partial[((int64_t)w.split * ka.M + w.t0 + cb + i) * N + ch] = __uint_as_float(r[i]);
          }
          continue;
        }
        uint32_t hv[16];
        if (ea.epi == FG_EPI_RELU) {
#pragma unroll
          for (int k = 0; k < 16; ++k)
            hv[k] = pack_h2(fmaxf(__uint_as_float(r[2 * k]) + bias_f, 0.0f),
                            fmaxf(__uint_as_float(r[2 * k + 1]) + bias_f, 0.0f));
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k)
            hv[k] = pack_h2(__uint_as_float(r[2 * k]) + bias_f, __uint_as_float(r[2 * k + 1]) + bias_f);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t q[4] = {hv[4 * j], hv[4 * j + 1], hv[4 * j + 2], hv[4 * j + 3]};
          transpose8x8_h(q, lane);
          uint4 o;
          o.x = __byte_perm(q[0], q[1], 0x5410);          // channels 0, 1
          o.y = __byte_perm(q[2], q[3], 0x5410);          // 2, 3
          o.z = __byte_perm(q[0], q[1], 0x7632);          // 4, 5
          o.w = __byte_perm(q[2], q[3], 0x7632);          // 6, 7
          const int tt = cb + 8 * j + (lane & 7);
          if (tt < ntok) {
            const int64_t t = w.t0 + tt;
            if (ea.epi == FG_EPI_RESIDUAL) {
              const uint4 rv = *reinterpret_cast<const uint4*>(ea.residual + t * N + chb);
              o.x = hadd2_u32(o.x, rv.x);
              o.y = hadd2_u32(o.y, rv.y);
              o.z = hadd2_u32(o.z, rv.z);
              o.w = hadd2_u32(o.w, rv.w);
            }
            *reinterpret_cast<uint4*>(ea.Y + t * N + chb) = o;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(empty_cl[acc]);
    }
  }

  // both CTAs are done with the pair's TMEM (CTA 0's MMAs drained above, every epilogue read
  // done) before it is freed
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == kTmemWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                 : "memory");
  }
}

int g_max_clusters = -1;
std::once_flag g_max_clusters_once;

cudaLaunchConfig_t pair_config(unsigned grid, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

}  // namespace

// Clusters of two that can be resident at once (one CTA per SM), queried once.
int pair_max_clusters() {
  std::call_once(g_max_clusters_once, [] {
    if (cudaFuncSetAttribute(gemm_q4_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config(2, nullptr, attr);
    cfg.numAttrs = 1;                                  // the cluster shape only
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_q4_pair_kernel, &cfg) == cudaSuccess && n > 0)
      g_max_clusters = n;
  });
  return g_max_clusters;
}

// Ring depths for a plan.  With many token tiles (prefill) each code tile is reused from L2
// by the token tiles of a raster group: 6 k-block slots keep the tensor pipe fed and code
// stages of one k-block (4 of them) suffice.  With one or two token tiles (decode) the 4-bit
// weights stream from HBM: a thread that issues TMA copies from HBM manages one every
// ~600 cycles whatever its size, so a code stage carries RG k-blocks (a 256-row code box and
// its statistics: two copies per 4 k-blocks) and the ring gets at least 12 k-blocks of codes
// in flight (~60 KB per SM) over 5 or 6 slots.  Stages of RG k-blocks need every unit to hold
// whole stages (the planner rounds kb_per_split to RG when K allows).
static bool pair_rings(const GemmPlan& p, int tnh, int* r_out, int* rc_out, int* sk_out,
                       int* xslot_out) {
  const int xslot = (tnh * BK * 2 + 1023) / 1024 * 1024;
  const bool stream = p.tiles_t <= 2;
  const int sk = (stream && p.kblocks % RG == 0 && p.kb_per_split % RG == 0) ? RG : 1;
  auto rc_for = [&](int r) {
    const int n = std::min(RC_MAX, (POOL_BYTES - r * (W_BYTES + xslot)) / (sk * CS_BYTES));
    return sk == 1 ? n / RG * RG : n;
  };
  int r = 6, rc = 4;
  if (stream) {
    for (r = 6; r > RG && rc_for(r) * sk < 12; --r) {
    }
    rc = rc_for(r);
  }
  if (r < RG || r > R_MAX || rc < 2 || rc > RC_MAX || (sk == 1 && rc % RG != 0) ||
      r * (W_BYTES + xslot) + rc * sk * CS_BYTES > POOL_BYTES)
    return false;
  *r_out = r;
  *rc_out = rc;
  *sk_out = sk;
  *xslot_out = xslot;
  return true;
}

// Raster group: X is 3.6x the bytes of the 4-bit codes per k-block and tile, so the clusters
// working at one time should span many channel pairs and few token tiles; up to 4 token tiles,
// fewer when the group's X would pass 64 MB (half the L2), e.g. 2 at K = 49152.  Measured at
// the OPT-175B prefill shapes (18432 tokens): 4 (2 at K = 49152) is 3.5-4% faster than 8,
// 16 or groups of channel pairs; at the 6.7B shapes the group size makes no difference.
// With fp16 weights a channel pair's A tiles are as many bytes as a token tile of X, and the
// DRAM bytes per wave, g X tiles + 76 / g weight tiles, are least near g = 8, whatever K:
// 8 token tiles there (in the OPT-175B bench 1% faster than 4, and another 1% faster than
// capping the group at 64 MB of X, which gave 2 at K = 49152; A/B runs in one call).
static int pair_raster_group(const GemmPlan& p, bool w16) {
  if (w16) return 8;
  const double x_tile = (double)p.tn * p.K * 2.0;
  return (int)std::max(1.0, std::min(4.0, 64e6 / x_tile));
}

cudaError_t launch_gemm_pair(const GemmPlan& p, const fg_q4mat& W, const uint16_t* X,
                             const EpiArgs& ea, cudaStream_t st, const uint16_t* w16, void* ws) {
  const int maxcl = pair_max_clusters();
  if (maxcl <= 0) return cudaErrorInvalidConfiguration;
  const int tnh = p.tn / 2;
  int r = 0, rc = 0, sk = 1, xslot = 0;
  if (p.tn % 16 != 0 || tnh < 72 || tnh > TNH_MAX || p.tiles_c % 2 != 0 ||
      !pair_rings(p, tnh, &r, &rc, &sk, &xslot))
    return cudaErrorInvalidConfiguration;
  CUtensorMap tmX, tmC, tmS;
  cudaError_t e = make_map_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X, (uint64_t)p.K,
                              (uint64_t)p.M, (uint64_t)p.K * 2, BK, (uint32_t)tnh,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = make_map_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, W.codes, (uint64_t)(p.N / 2),
                  (uint64_t)p.K, (uint64_t)(p.N / 2), TCH / 2, (uint32_t)(BK * sk),
                  CU_TENSOR_MAP_SWIZZLE_64B);
  if (e != cudaSuccess) return e;
  e = make_map_2d(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT32, W.ab, (uint64_t)(p.N / 64),
                  (uint64_t)p.K, (uint64_t)(p.N / 64) * 4, 4, (uint32_t)(BK * sk),
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  // restored fp16 weights [K][N]: boxes of 64 channels x 64 k-rows (or the code map again)
  CUtensorMap tmA = tmC;
  if (w16) {
    e = make_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, w16, (uint64_t)p.N, (uint64_t)p.K,
                    (uint64_t)p.N * 2, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
  }
  // dynamic order for plans of several token tiles: the ticket counter in the workspace,
  // zeroed on the stream before the launch
  unsigned int* ctr = nullptr;
  if (p.tiles_t >= 2) {
    if (!ws || p.sched_off % 16 != 0) return cudaErrorInvalidValue;
    ctr = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + p.sched_off);
    e = cudaMemsetAsync(ctr, 0, sizeof(unsigned int), st);
    if (e != cudaSuccess) return e;
  }
  const PArgs ka{(int)p.M,  (int)p.N, (int)p.K, p.tiles_t, p.tiles_c / 2, p.kblocks,
                 p.kb_per_split, (int)p.units, tnh, r, rc, sk, xslot, pair_raster_group(p, w16),
                 w16 ? 1 : 0, ctr};
  const int64_t clusters = std::min<int64_t>(p.units, maxcl);
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config((unsigned)(2 * clusters), st, attr);
  return cudaLaunchKernelEx(&cfg, gemm_q4_pair_kernel, tmX, tmC, tmS, tmA, ka, ea);
}

cudaError_t gemm_pair_read_error(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_gemm_pair_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_gemm_pair_error, &zero, sizeof(unsigned int));
}

}  // namespace fg
