// Dequant-fused GEMM on the 5th-generation tensor cores (sm_103a):
//   Y[M][N] = epi( X[M][K] * W^[K][N] + bias )
// where W^ is restored to fp16 from 4-bit codes grouped 64 along the output channel N
// with per-group (a, b) [FlexGen review (jaehun.me), "4-bit 압축은 정수 연산 가속과 같은가":
// weights grouped along the output channel, restored to FP16 before compute, no INT4
// matmul].  The block schedule's batch reuse makes the projections and the MLP dense
// contractions over M = g*s (prefill) or M = B (decode) rows.
//
// The tensor core computes the transposed product Y^T = W^T X^T: the restored weights are
// the MMA's A operand (M = 128 output channels) and the activations its B operand
// (N = up to 256 tokens).  Against the straight orientation (tokens as M, channels as N)
// this halves the codes restored per MMA cycle at 256 tokens per tile, needs no padding
// when the token count is small (decode: N = B), and keeps the restored tile in the
// layout the codes already have: one k-row of 64 output channels is one 128-byte swizzle
// row of an MN-major operand, one quantisation group.
//
// Persistent kernel: one CTA per SM loops over (split, token tile, channel tile) units,
// K step 64.  Two rings in shared memory: a k-block ring of R slots, each an X tile and a
// restored A tile, freed together by one MMA commit; and a code ring of RC stages (codes +
// group statistics), freed by the restorers once they have consumed the words.  Depths
// follow the token tile: R = 4, RC = 6 at tn = 256; R = 6, RC = 16 at tn = 64, where the
// codes stream from HBM and need more bytes in flight.
//   warp 0      TMA producer of X tiles (tn x 64, 128B swizzle, K-major); owns TMEM
//   warp 1      one thread issues tcgen05.mma (kind::f16, M=128, N=tn, K=16) into one of
//               two double-buffered fp32 accumulators; it waits once per k-block, on a
//               barrier that completes when the A slot is restored AND the X tile landed
//   warp 15     with tn <= 128, a second issuing thread: the two take alternate k-blocks
//               into their own accumulators (one thread cannot keep the tensor pipe busy
//               with N <= 128 MMAs); the epilogue adds the pair
//   warp 2      TMA producer of code tiles (64B swizzle) and the group statistics of the
//               aligned 256-channel block
//   warps 3-10  four groups of two warps restore every fourth k-block: codes -> fp16 A
//               tile (MN-major, 128B swizzle), four 16-byte code chunks (32 channels each)
//               per thread per k-block
//   warps 11-14 epilogue of the previous tile (tcgen05.ld: one TMEM lane per output
//               channel, 32 tokens per batch; bias / ReLU / residual, fp16 store); with a
//               residual the tile's rows are prefetched to L2 while the accumulator fills
// Barrier polls take the non-blocking test_wait first: on the MMA issuer's path the phase
// is nearly always complete, and test_wait returns several times sooner than try_wait.
// Restoration per pair of codes: the nibble is OR-ed into mantissa bits 6..9 of 1.0h so
// that the half equals 1 + q/16, then one HFMA2 gives (1 + q/16)*(16s) + (a - 16s) = a + q*s.
// Within each 8-channel chunk the pairs land as (n0,n4,n1,n5,n2,n6,n3,n7), so accumulator
// lane 8u+p holds channel 8u+kPerm[p]; the epilogue maps lanes back to channels.
//
// Few work units (decode) split K: partial fp32 tiles go to the caller's workspace and a
// reduce kernel applies the epilogue.
//
// Every mbarrier wait is bounded (about 2 s); on timeout the CTA raises an abort flag,
// sets the device error word, drains its outstanding copies and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "fg_common.cuh"
#include "fg_internal.h"
#include "gemm_tc.cuh"

namespace fg {

__device__ unsigned int g_gemm_error = 0;

namespace {

constexpr int TCH = 128;                    // output channels per tile (MMA M)
constexpr int TN_MAX = 256;                 // tokens per tile (MMA N), runtime tn <= 256
constexpr int BK = 64;
constexpr int RA_MAX = 10;                  // restored-A ring (k-block barriers)
constexpr int RC_MAX = 16;                  // code ring: codes + group statistics
constexpr int RW = 8;                       // restore warps
constexpr int RT = RW * 32;                 // restore threads
constexpr int RG = 4;                       // restore groups: k-blocks restored concurrently
constexpr int RTG = RT / RG;                // threads per restore group
constexpr int ITEMS = RG;                   // 16-byte code chunks per thread per k-block
constexpr int RW0 = 3;                      // first restore warp
constexpr int EW0 = RW0 + RW;               // first epilogue warp
constexpr int MW1 = EW0 + 4;                // second MMA issuer warp (token tiles <= 128)
constexpr int THREADS = (MW1 + 1) * 32;
constexpr int W_BYTES = TCH * BK * 2;       // 16 KB restored
constexpr int C_BYTES = BK * TCH / 2;       // 4 KB of codes (64-byte rows)
constexpr int S_BYTES = BK * 4 * 4;         // 1 KB: (a, b) words of 4 groups x 64 k-rows
constexpr int CS_BYTES = C_BYTES + S_BYTES; // one code stage
constexpr int SMEM_BYTES = 232448;          // the whole per-CTA budget
constexpr int BAR_BYTES = 512 + 1024;       // barriers, then the epilogue's exchange words
constexpr int XCH_OFF = 512;
constexpr int POOL_BYTES = SMEM_BYTES - 1024 /*align*/ - BAR_BYTES;
constexpr uint32_t TMEM_COLS = 2 * TN_MAX;  // two accumulator buffers
static_assert((2 * RA_MAX + 2 * RC_MAX + 5) * 8 + 8 <= XCH_OFF, "barrier space");
static_assert(TMEM_COLS == 512, "TMEM budget");
static_assert(RTG * ITEMS * 32 == BK * TCH, "restore coverage: 32 codes per item");
static_assert(CS_BYTES % 512 == 0, "64B-swizzled code stages stay 512-byte aligned");
// The code ring's depth is a multiple of the restore groups (launch_gemm rounds it down), so
// stage c always goes to group c % RG and a group waits on every lap of its stages in order.
// Otherwise a group could wait on lap L of a stage whose lap L - 1 (another group's k-block)
// had not landed yet: a parity wait cannot tell lap L from lap L - 2 and would pass at once
// on stale codes, since TMA loads complete in any order.  The restored-A ring needs ra >= RG
// instead: MMAs complete in order, so a group that saw the MMAs of k-block it - RG - ra done
// has seen the slot's previous lap (k-block it - 2 ra) done as well.
static_assert(RC_MAX % RG == 0, "code ring depth in whole restore-group rounds");
constexpr long long kWaitCycles = 1ll << 32;
constexpr int SWZ_GROUP = 8;                // token tiles per raster group

// instruction descriptor: D f32, A and B f16, A MN-major, B K-major, M = 128, N = tn
__host__ __device__ constexpr uint32_t make_idesc(int tn) {
  return (1u << 4) | (1u << 15) | ((uint32_t)(tn >> 3) << 17) | ((uint32_t)(TCH >> 4) << 24);
}

// Bounded wait.  Returns false (and raises the CTA abort flag) on timeout or when another
// warp already aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_test(bar, parity)) return true;            // fast path: phase already complete
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

// 8 x 8 fp16 transpose inside each 8-lane group of a warp.  On entry lane p of the group
// holds w[q] = (D[p][2q], D[p][2q+1]) for columns (tokens) 0..7 of its row p; on return it
// holds w[q] = (D[2q][p], D[2q+1][p]), column p of every row.  Three exchanges, each swapping
// one lane-index bit with one element-index bit (half of a word, then word bit 0, then word
// bit 1).
__device__ __forceinline__ void transpose8x8_h(uint32_t (&w)[4], int lane) {
  const bool b0 = lane & 1, b1 = lane & 2, b2 = lane & 4;
  const uint32_t sel = b0 ? 0x3276u : 0x5410u;        // (x.hi, w.hi) or (w.lo, x.lo)
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

// Bias / ReLU / residual on 8 consecutive outputs and the fp16 store (reduce kernel);
// returns the stored fp16 words.
__device__ __forceinline__ uint4 epilogue8(const EpiArgs& ea, float (&v)[8], int64_t row, int n,
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
  return o;
}

struct Unit {
  int t0, c0, split, kb_begin, kb_end;
};

// Work unit u -> token tile, channel tile and k-block range.  Grouped raster: SWZ_GROUP
// token tiles share a wave of channel tiles, so a wave of CTAs touches few X tiles.
__device__ __forceinline__ Unit unit_coords(int u, int tn, int tiles_t, int tiles_c,
                                            int kblocks, int kb_per_split) {
  Unit r;
  const int tiles = tiles_t * tiles_c;
  r.split = u / tiles;
  const int lin = u - r.split * tiles;
  const int group_span = SWZ_GROUP * tiles_c;
  const int grp = lin / group_span;
  const int first_t = grp * SWZ_GROUP;
  const int gt = min(SWZ_GROUP, tiles_t - first_t);
  const int within = lin - grp * group_span;
  r.t0 = (first_t + within % gt) * tn;
  r.c0 = (within / gt) * TCH;
  r.kb_begin = r.split * kb_per_split;
  r.kb_end = min(kblocks, r.kb_begin + kb_per_split);
  return r;
}

struct KArgs {
  int M, N, K, tn;
  uint32_t idesc;
  int tiles_t, tiles_c, kblocks, kb_per_split, units;
  int ra;              // restored-A ring depth (the k-block barriers)
  int rx;              // X ring depth, <= ra
  int ni;              // MMA issuers: 2 for tn <= 128 (k-blocks alternate, 2 accumulators)
  int rc;              // code ring depth
};

// KV: the K/V append in the epilogue (a separate instance, so that the plain GEMM carries
// none of its code: the larger kernel measured a few percent slower even when the append
// never ran).
template <bool KV>
__global__ void __launch_bounds__(THREADS, 1)
gemm_q4_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmC,
                  const __grid_constant__ CUtensorMap tmS, const KArgs ka, const EpiArgs ea) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int tn = ka.tn, R = ka.ra, RX = ka.rx, RC = ka.rc, XB = tn * 128;
  uint8_t* sW = smem;                                  // R x W_BYTES (restored weights)
  uint8_t* sX = sW + R * W_BYTES;                      // RX x XB (activations)
  uint8_t* sC = sX + RX * XB;                          // RC x CS_BYTES (codes | statistics)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + POOL_BYTES);
  // bars: full[RA_MAX], mma_done[RA_MAX], full_c[RC_MAX], free_c[RC_MAX], acc_full[2],
  // acc_empty[2].  K-block it uses A slot it % R and X slot it % RX (RX <= R).  full(it % R)
  // completes when the restore group has written the A slot AND the X tile has landed (the
  // X producer's expect_tx arrival plus the TMA bytes), so the MMA issuer waits once per
  // k-block.  mma_done(it % R) completes when the MMAs of k-block it are done: its A slot may
  // be rewritten and its X slot refilled.  The X producer issues k-block it after the MMAs
  // of k-block it - RX, hence after those of it - R, so its arrival always lands in k-block
  // it's phase of full(it % R).
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * RA_MAX + 2 * RC_MAX + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // K/V append: per-token min/max words of the four epilogue warps, two buffers
  uint32_t* xch = reinterpret_cast<uint32_t*>(smem + POOL_BYTES + XCH_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int r) { return bar0 + 8u * r; };
  auto mma_done = [&](int r) { return bar0 + 8u * (RA_MAX + r); };
  auto full_c = [&](int c) { return bar0 + 8u * (2 * RA_MAX + c); };
  auto free_c = [&](int c) { return bar0 + 8u * (2 * RA_MAX + RC_MAX + c); };
  auto acc_full = [&](int a) { return bar0 + 8u * (2 * RA_MAX + 2 * RC_MAX + a); };
  auto acc_empty = [&](int a) { return bar0 + 8u * (2 * RA_MAX + 2 * RC_MAX + 2 + a); };
  const uint32_t xchg = bar0 + 8u * (2 * RA_MAX + 2 * RC_MAX + 4);

  if (threadIdx.x == 0) {
    for (int r = 0; r < R; ++r) {
      mbar_init(full(r), RTG + 1);                 // one restore group + the X producer
      mbar_init(mma_done(r), 1);
    }
    for (int c = 0; c < RC; ++c) {
      mbar_init(full_c(c), 1);
      mbar_init(free_c(c), RTG);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full(a), ka.ni);               // one commit per MMA issuer
      mbar_init(acc_empty(a), 4);                  // one arrival per epilogue warp
    }
    mbar_init(xchg, 4);                            // one arrival per epilogue warp
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
  pdl_launch_dependents();
  pdl_wait();

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ TMA producers
    // warp 0: X tiles into the X ring; warp 2: codes + statistics into the code ring
    if (lane == 0) {
      const bool is_x = (warp == 0);
      const int depth = is_x ? RX : RC;
      int it = 0, s = 0;                              // k-block, slot in this ring
      uint32_t ph = 0;                                // lap parity of slot s (code ring)
      int kr = 0;                                     // X: A-ring position of k-block it
      int fa = R - RX;                                // X: A-ring position of it - RX
      uint32_t fph = 1;                               //    and its lap parity
      bool ok = true;
      for (int u = blockIdx.x; u < ka.units && ok; u += gridDim.x) {
        const Unit w = unit_coords(u, tn, ka.tiles_t, ka.tiles_c, ka.kblocks, ka.kb_per_split);
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++it) {
          if (is_x) {
            // the X slot is free once the MMAs of k-block it - RX are done
            if (it >= RX && !mbar_wait(mma_done(fa), fph, abort_flag)) {
              ok = false;
              break;
            }
            mbar_expect_tx(full(kr), (uint32_t)XB);
            tma_load_2d(smem_u32(sX + s * XB), &tmX, kb * BK, w.t0, full(kr));
            if (++kr == R) kr = 0;
            if (++fa == R) {
              fa = 0;
              fph ^= 1;
            }
          } else {
            if (it >= RC && !mbar_wait(free_c(s), ph ^ 1, abort_flag)) {
              ok = false;
              break;
            }
            uint8_t* cs = sC + s * CS_BYTES;
            mbar_expect_tx(full_c(s), (uint32_t)CS_BYTES);
            tma_load_2d(smem_u32(cs), &tmC, w.c0 / 2, kb * BK, full_c(s));
            tma_load_2d(smem_u32(cs + C_BYTES), &tmS, (w.c0 / 256) * 4, kb * BK, full_c(s));
          }
          if (++s == depth) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      // Drain: every issued load must have landed before this CTA can exit.  X tiles land
      // on the k-block barriers, which the MMA issuer consumes on the normal path; after an
      // abort their phases may also lack restore arrivals, so those waits are short.
      if (!is_x || !ok) {
        const long long limit = is_x ? (1ll << 26) : kWaitCycles;
        const int dep = is_x ? R : RC;
        for (int i = max(0, it - depth); i < it; ++i) {
          const uint32_t bar = is_x ? full(i % dep) : full_c(i % dep);
          const long long t0 = clock64();
          while (!mbar_try(bar, (i / dep) & 1)) {
            if (clock64() - t0 > limit) {
              atomicOr(&g_gemm_error, 2u);
              break;
            }
          }
        }
      }
    }
  } else if (warp == 1 || warp == MW1) {
    // ------------------------------------------------------------ MMA issuers
    // With ni = 2 (token tiles of at most 128), issuer mi takes the k-blocks it == mi
    // (mod 2), which restore group mi restores, into its own accumulator (columns
    // acc * 256 + mi * 128): a single issuing thread cannot keep the tensor pipe busy with
    // N <= 128 MMAs.  The epilogue adds the two accumulators.
    const int mi = (warp == 1) ? 0 : 1;
    if (lane == 0 && mi < ka.ni) {
      // descriptors of slot 0; a slot offset, and the K16 step, add (bytes >> 4) to the
      // start-address field (all addresses are below 256 KB)
      const uint64_t adesc0 = smem_desc(smem_u32(sW), 64 * 128, 1024);
      const uint64_t bdesc0 = smem_desc(smem_u32(sX), 16, 1024);
      // descriptors of the current slot advance with the ring; parity by bit test (ni is
      // 1 or 2): this thread's bookkeeping sits on the MMA stream's critical path
      const uint64_t a_step = W_BYTES >> 4, b_step = (uint64_t)(XB >> 4);
      uint64_t ad = adesc0, bd = bdesc0;
      int tl = 0, r = 0, rx = 0;                      // A slot, X slot
      uint32_t ph = 0, par = 0;                       // lap parity of A slot r; k-block parity
      const uint32_t mask = (ka.ni == 2) ? 1u : 0u;
      bool ok = true;
      for (int u = blockIdx.x; u < ka.units && ok; u += gridDim.x, ++tl) {
        const Unit w = unit_coords(u, tn, ka.tiles_t, ka.tiles_c, ka.kblocks, ka.kb_per_split);
        const int acc = tl & 1;
        if (tl >= 2 && !mbar_wait(acc_empty(acc), ((tl >> 1) & 1) ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t tacc = tmem + acc * TN_MAX + mi * 128;
        uint32_t accumulate = 0u;
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if ((par & mask) == (uint32_t)mi) {
            if (!mbar_wait(full(r), ph, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            umma_f16(tacc, ad, bd, ka.idesc, accumulate);
            umma_f16(tacc, ad + 128, bd + 2, ka.idesc, 1u);
            umma_f16(tacc, ad + 256, bd + 4, ka.idesc, 1u);
            umma_f16(tacc, ad + 384, bd + 6, ka.idesc, 1u);
            umma_commit(mma_done(r));
            accumulate = 1u;
          }
          ++par;
          if (++r == R) {
            r = 0;
            ph ^= 1;
            ad = adesc0;
          } else {
            ad += a_step;
          }
          if (++rx == RX) {
            rx = 0;
            bd = bdesc0;
          } else {
            bd += b_step;
          }
        }
        umma_commit(acc_full(acc));
      }
    }
  } else if (warp < EW0) {
    // ------------------------------------------------------------ restore codes -> A
    // RG groups of RTG threads; group g restores the k-blocks it == g (mod RG), so RG
    // k-blocks are in restoration at once.  Item -> (k-row, 16-byte code chunk c = 32
    // channels).  Each 8-lane phase takes the two chunks of one 64-channel group on four
    // k-rows whose (k & 3) differ and whose (k & 1, k & 4) differ, which keeps the
    // 64B-swizzled code loads and the 128B-swizzled restored stores free of bank conflicts.
    const int tid = threadIdx.x - 32 * RW0;           // 0 .. RT-1
    const int grp = tid / RTG, tg = tid % RTG;
    int code_off[ITEMS], stat_k[ITEMS], w_off[ITEMS], sw[ITEMS], cl4[ITEMS];
#pragma unroll
    for (int t = 0; t < ITEMS; ++t) {
      const int item = tg + t * RTG;                  // 0 .. 255
      const int cl = item & 1, rsel = (item >> 1) & 3, quad = (item >> 3) & 1;
      const int j = (item >> 4) & 1;
      const int k = (item >> 5) * 8 + (quad ? 2 + rsel : (rsel < 2 ? rsel : rsel + 4));
      const int c = 2 * j + cl;
      code_off[t] = k * 64 + ((c ^ ((k >> 1) & 3)) << 4);
      stat_k[t] = k * 4 + j;
      w_off[t] = j * (BK * 128) + k * 128;
      sw[t] = k & 7;
      cl4[t] = cl * 4;
    }
    // ring positions of k-block it: code stage c (lap parity phc) and slot r (parity phr);
    // the slot is free once the MMAs of k-block it - R (same slot, parity phr ^ 1) are done
    int it = 0, c = 0, r = 0, rg = 0;
    uint32_t phc = 0, phr = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < ka.units && ok; u += gridDim.x) {
      const Unit w = unit_coords(u, tn, ka.tiles_t, ka.tiles_c, ka.kblocks, ka.kb_per_split);
      const int g0 = (w.c0 >> 6) & 3;                 // first group of the tile in the box
      for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++it) {
        const int cc_ = c, cr = r;
        const uint32_t cphc = phc, cphr = phr;
        const bool mine = (rg == grp);
        if (++c == RC) { c = 0; phc ^= 1; }
        if (++r == R) { r = 0; phr ^= 1; }
        if (++rg == RG) rg = 0;
        if (!mine) continue;
        if (!mbar_wait(full_c(cc_), cphc, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* cs = sC + cc_ * CS_BYTES;
        const uint32_t* ss = reinterpret_cast<const uint32_t*>(cs + C_BYTES);
        uint4 cw[ITEMS];
        uint32_t abw[ITEMS];
#pragma unroll
        for (int t = 0; t < ITEMS; ++t) {
          cw[t] = *reinterpret_cast<const uint4*>(cs + code_off[t]);
          abw[t] = ss[stat_k[t] + g0];
        }
        if (it >= R && !mbar_wait(mma_done(cr), cphr ^ 1, abort_flag)) {
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
        // the code stage may be refilled: its words have been consumed by the stores above
        mbar_arrive(free_c(cc_));
        // make the stores visible to the tensor core's (async) proxy, then arrive
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(full(cr));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // TMEM lane L holds restored row L of the tile: channel (L & ~7) + kPerm[L & 7] with
    // kPerm = (0,4,1,5,2,6,3,7), the order restore8 leaves the pairs in.
    const int lane_base = 32 * (warp & 3);            // TMEM lanes this warp may read
    const int L = lane_base + lane;
    const int ch_in_tile = (L & ~7) + ((L & 7) >> 1) + ((L & 1) << 2);
    const int64_t N = ka.N;
    const bool add_res = !ea.partial && ea.epi == FG_EPI_RESIDUAL;
    const int q = warp & 3;                           // TMEM lane quarter
    int tl = 0;
    uint32_t xph = 0;                                 // K/V exchanges so far
    bool fail = false;
    for (int u = blockIdx.x; u < ka.units; u += gridDim.x, ++tl) {
      const Unit w = unit_coords(u, tn, ka.tiles_t, ka.tiles_c, ka.kblocks, ka.kb_per_split);
      const int acc = tl & 1;
      const int ntok = min(tn, ka.M - w.t0);          // valid tokens of this tile
      if (add_res) {
        // pull this tile's residual rows (2 x 128 bytes per token) into L2 while the
        // accumulator fills
        for (int i = 32 * (warp & 3) + lane; i < 2 * ntok; i += 128)
          prefetch_l2(ea.residual + (int64_t)(w.t0 + (i >> 1)) * N + w.c0 + (i & 1) * 64);
      }
      // the warp-collective TMEM loads below need the whole warp: decide for all its lanes
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(acc_full(acc), (tl >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      const int64_t ch = w.c0 + ch_in_tile;
      const float bias_f = (!ea.partial && ea.bias) ? h2f(ea.bias[ch]) : 0.0f;
      // first channel of this lane's 8-lane group (channels in natural order after the
      // transpose)
      const int64_t chb = w.c0 + lane_base + (lane & ~7);
      // a K or V tile of the QKV projection (h is a multiple of 128: no tile straddles)
      const bool kv_tile = KV && ea.kv.k_codes != nullptr && !ea.partial && w.c0 >= ea.kv.h;
      const KvCol kcol = kv_tile ? kv_col(ea.kv, (int)chb) : KvCol{};
      for (int cb = 0; cb < ntok; cb += 32) {
        // columns past tn (at most cb + 31 <= 255) stay inside this accumulator's 256
        uint32_t r[32];
        __syncwarp();
        const uint32_t taddr = tmem + ((uint32_t)lane_base << 16) + acc * TN_MAX + cb;
        tmem_ld16(taddr, r);
        tmem_ld16(taddr + 16, r + 16);
        tmem_wait_ld();
        if (ka.ni == 2) {
          // second issuer's accumulator, columns + 128 (tn <= 128 so cb + 31 < 128 + 128)
          uint32_t r2[16];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tmem_ld16(taddr + 128 + 16 * h, r2);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              r[16 * h + i] = __float_as_uint(__uint_as_float(r[16 * h + i]) + __uint_as_float(r2[i]));
          }
        }
        if (ea.partial) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (cb + i >= ntok) break;
            ea.partial[((int64_t)w.split * ka.M + w.t0 + cb + i) * N + ch] = __uint_as_float(r[i]);
          }
          continue;
        }
        // bias (and ReLU) in fp32 on this lane's channel, then fp16 pairs along tokens
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
        // per 8-token block: transpose so this lane holds token 8j + (lane & 7) for the
        // group's 8 channels, undo the restore order (positions 0..7 hold channels
        // 0,4,1,5,2,6,3,7), add the residual row segment and store 16 bytes
        uint4 ov[4];                                  // the stored fp16 outputs
        uint32_t mmv[4];                              // their min/max over the warp's channels
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t u[4] = {hv[4 * j], hv[4 * j + 1], hv[4 * j + 2], hv[4 * j + 3]};
          transpose8x8_h(u, lane);
          uint4 o;
          o.x = __byte_perm(u[0], u[1], 0x5410);          // channels 0, 1
          o.y = __byte_perm(u[2], u[3], 0x5410);          // 2, 3
          o.z = __byte_perm(u[0], u[1], 0x7632);          // 4, 5
          o.w = __byte_perm(u[2], u[3], 0x7632);          // 6, 7
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
          ov[j] = o;
          if (kv_tile) {
            const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
            uint32_t mm = q4_minmax8(ow);
            mm = __vminu2(mm, __shfl_xor_sync(0xFFFFFFFFu, mm, 8));
            mmv[j] = __vminu2(mm, __shfl_xor_sync(0xFFFFFFFFu, mm, 16));
          }
        }
        if (!kv_tile) continue;
        // ---- K/V append.  A 64-channel group is two lane quarters (q, q ^ 1): lanes 0..7
        // publish the quarter's min/max of tokens 8j + lane, then read the partner's
        uint32_t* xb = xch + (xph & 1) * 128;
        if (lane < 8) {
#pragma unroll
          for (int j = 0; j < 4; ++j) xb[32 * q + 8 * j + lane] = mmv[j];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(xchg);
        if (!mbar_wait(xchg, xph & 1, abort_flag)) {
          fail = true;
          break;
        }
        ++xph;
        // codes of the four tokens' words on the fast path; words with a code near a tie
        // are redone with the exact division after the unrolled loop
        uint32_t abv[4], cwv[4], nmask = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          abv[j] = q4_ab_word(__vminu2(mmv[j], xb[32 * (q ^ 1) + 8 * j + (lane & 7)]));
          const uint32_t ow[4] = {ov[j].x, ov[j].y, ov[j].z, ov[j].w};
          bool nr = false;
          cwv[j] = q4_codes8(ow, q4_group(abv[j]), nr);
          nmask |= (uint32_t)nr << j;
        }
        if (nmask) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if ((nmask >> j) & 1u) {
              const Q4Group g = q4_group(abv[j]);
              cwv[j] = q4_codes8_exact(ov[j], g.af, g.bma);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int tt = cb + 8 * j + (lane & 7);
          if (tt < ntok) {
            const int kr = kv_row(ea.kv, w.t0 + tt);
            *kv_codes_at(ea.kv, kcol, kr) = cwv[j];
            if ((chb & 63) == 0) *kv_ab_at(ea.kv, kcol, kr) = abv[j];
          }
        }
      }
      if (fail) break;
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

// Sum the split-K partials and apply bias / ReLU / residual: 8 outputs per thread.  With
// a K/V append the 8 threads of a lane segment hold one 64-channel group of a row (N and
// the chunk count are multiples of 64 and 8), quantised as the standalone quantiser does.
__global__ void __launch_bounds__(256)
gemm_reduce_kernel(const float* __restrict__ partial, int splits, int64_t M, int N, EpiArgs ea) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t idx = (int64_t)blockIdx.x * 256 + threadIdx.x;
  const int64_t chunks = M * (N / 8);
  const bool live = idx < chunks;               // whole lane segments are live or not
  const int64_t row = live ? idx / (N / 8) : 0;
  const int n = live ? (int)(idx - row * (N / 8)) * 8 : 0;
  uint4 o = make_uint4(0, 0, 0, 0);
  if (live) {
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < splits; ++s) {
      const float4* pp = reinterpret_cast<const float4*>(partial + ((int64_t)s * M + row) * N + n);
      const float4 x = pp[0], y = pp[1];
      v[0] += x.x; v[1] += x.y; v[2] += x.z; v[3] += x.w;
      v[4] += y.x; v[5] += y.y; v[6] += y.z; v[7] += y.w;
    }
    o = epilogue8(ea, v, row, n, N);
  }
  if (ea.kv.k_codes == nullptr || !__any_sync(0xFFFFFFFFu, live && n >= ea.kv.h)) return;
  const uint32_t w[4] = {o.x, o.y, o.z, o.w};
  uint32_t mm = q4_minmax8(w);
#pragma unroll
  for (int k = 1; k < 8; k <<= 1) mm = __vminu2(mm, __shfl_xor_sync(0xFFFFFFFFu, mm, k));
  if (live && n >= ea.kv.h) {
    const uint32_t abw = q4_ab_word(mm);
    const KvCol col = kv_col(ea.kv, n);
    const int kr = kv_row(ea.kv, (int)row);
    *kv_codes_at(ea.kv, col, kr) = q4_codes8_checked(w, q4_group(abw));
    if ((n & 63) == 0) *kv_ab_at(ea.kv, col, kr) = abw;
  }
}

// One CTA per output row: the split-K sum and the epilogue as gemm_reduce_kernel (the row
// stored to Y), then the pre-LN LayerNorm of the stored fp16 row into y_ln with the
// statistics of the standalone LayerNorm: fp32 mean, then the mean squared deviation (a
// population variance), rsqrt(var + eps), (x - mean) * rstd * gamma + beta.  A thread keeps
// at most 8 chunks of 8 values in registers (N <= 16384).
constexpr int kLnChunks = 8;
__device__ __forceinline__ float block_sum256(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  __syncthreads();                                  // red is free (a previous sum was read)
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.0f;
#pragma unroll
  for (int w = 0; w < 8; ++w) s += red[w];
  return s;
}

__global__ void __launch_bounds__(256)
gemm_reduce_ln_kernel(const float* __restrict__ partial, int splits, int64_t M, int N, EpiArgs ea,
                      const uint16_t* __restrict__ gamma, const uint16_t* __restrict__ beta,
                      float eps, uint16_t* __restrict__ y_ln) {
  __shared__ float red[8];
  pdl_launch_dependents();
  pdl_wait();
  const int64_t row = blockIdx.x;
  const int nchunk = N / 8;
  uint4 yv[kLnChunks];
  float s = 0.0f;
#pragma unroll
  for (int c = 0; c < kLnChunks; ++c) {
    const int ci = threadIdx.x + 256 * c;
    yv[c] = make_uint4(0, 0, 0, 0);
    if (ci < nchunk) {
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int sp = 0; sp < splits; ++sp) {
        const float4* pp =
            reinterpret_cast<const float4*>(partial + ((int64_t)sp * M + row) * N + ci * 8);
        const float4 x = pp[0], y = pp[1];
        v[0] += x.x; v[1] += x.y; v[2] += x.z; v[3] += x.w;
        v[4] += y.x; v[5] += y.y; v[6] += y.z; v[7] += y.w;
      }
      yv[c] = epilogue8(ea, v, row, ci * 8, N);
      const uint32_t w[4] = {yv[c].x, yv[c].y, yv[c].z, yv[c].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack_h2(w[i]);
        s += f.x + f.y;
      }
    }
  }
  const float mean = block_sum256(s, red) / (float)N;
  float q = 0.0f;
#pragma unroll
  for (int c = 0; c < kLnChunks; ++c) {
    if (threadIdx.x + 256 * c < nchunk) {
      const uint32_t w[4] = {yv[c].x, yv[c].y, yv[c].z, yv[c].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack_h2(w[i]);
        const float d0 = f.x - mean, d1 = f.y - mean;
        q += d0 * d0 + d1 * d1;
      }
    }
  }
  const float rstd = rsqrtf(block_sum256(q, red) / (float)N + eps);
#pragma unroll
  for (int c = 0; c < kLnChunks; ++c) {
    const int ci = threadIdx.x + 256 * c;
    if (ci < nchunk) {
      const uint4 gu = ldg_nc_v4(gamma + ci * 8), bu = ldg_nc_v4(beta + ci * 8);
      const uint32_t w[4] = {yv[c].x, yv[c].y, yv[c].z, yv[c].w};
      const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w}, bw[4] = {bu.x, bu.y, bu.z, bu.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack_h2(w[i]), g2 = unpack_h2(gw[i]), b2 = unpack_h2(bw[i]);
        o[i] = pack_h2((f.x - mean) * rstd * g2.x + b2.x, (f.y - mean) * rstd * g2.y + b2.y);
      }
      reinterpret_cast<uint4*>(y_ln + row * N)[ci] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

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


cudaError_t make_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                        uint64_t mid, uint64_t outer, uint64_t mid_bytes, uint64_t outer_bytes,
                        uint32_t box_inner, uint32_t box_mid, CUtensorMapSwizzle swz) {
  const cuuint64_t dims[3] = {inner, mid, outer};
  const cuuint64_t strides[2] = {mid_bytes, outer_bytes};
  const cuuint32_t box[3] = {box_inner, box_mid, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Weight-streaming plan (M <= 128): one token tile, 128-channel tiles, K split so that the
// busiest persistent CTA (units taken round-robin) has the fewest k-blocks, counting about
// two k-blocks of pipeline ramp per unit and 24 (~6 us) for a split's partials and reduce
// launch.  Splits
// are whole code stages of kStreamStage k-blocks.  The split count is capped independently
// of the SM count, and the workspace is sized for the cap, so a workspace sized by the query
// for kMaxSms covers every device.
static void stream_plan(GemmPlan& p, int nsm) {
  p.kind = kGemmStream;
  p.tiles_t = 1;
  p.tn = (int)std::max<int64_t>(16, (p.M + 15) / 16 * 16);
  p.tiles_c = (int)(p.N / TCH);
  p.kblocks = (int)((p.K + BK - 1) / BK);
  const int cap = std::max(1, std::min({16, p.kblocks / 4,
                                        (2 * kMaxSms + p.tiles_c - 1) / p.tiles_c}));
  const int64_t cta = std::max(1, nsm);
  int best = 1;
  int64_t best_cost = -1;
  for (int s = 1; s <= cap; ++s) {
    const int kbs = ((p.kblocks + s - 1) / s + kStreamStage - 1) / kStreamStage * kStreamStage;
    if (s > 1 && (s - 1) * kbs >= p.kblocks) break;    // an empty split
    const int64_t rounds = ((int64_t)p.tiles_c * s + cta - 1) / cta;
    const int64_t cost = rounds * (kbs + 2) + (s > 1 ? 24 : 0);
    if (best_cost < 0 || cost < best_cost) {
      best = s;
      best_cost = cost;
    }
  }
  p.kb_per_split = ((p.kblocks + best - 1) / best + kStreamStage - 1) / kStreamStage * kStreamStage;
  p.splits = (p.kblocks + p.kb_per_split - 1) / p.kb_per_split;
  p.ws_bytes = (cap > 1) ? (size_t)cap * p.M * p.N * sizeof(float) : 0;
  p.units = (int64_t)p.tiles_c * p.splits;
  p.grid = (int)std::min<int64_t>(p.units, nsm);
}

// CTA-pair plan: tiles of 256 channels (a pair) x tn tokens, tn = 2 tnh the smallest multiple
// of 16 that covers M in ceil(M / 256) tiles (M = 144 -> one tile of 144).  K is split when
// the tiles leave clusters idle: the split count minimises the busiest cluster's k-blocks
// (units of equal size taken in turn: round-robin, or the next free ticket in the kernel's
// dynamic order, which deals the same counts; about two k-blocks of ramp per unit and 24 for
// a split's partials and reduce).  The count is capped independently of the SM count (at most 8, at least 8
// k-blocks per split, no more units than two rounds of the largest cluster count planned for)
// and the workspace is sized for the cap, so a workspace sized by the query covers any device.
// With several token tiles the workspace also holds the 256-byte unit counter of the
// kernel's dynamic order.
static bool pair_fits(int64_t M, int64_t N) { return M > 128 && N % 256 == 0; }

static void pair_plan(GemmPlan& p, int nsm) {
  p.kind = kGemmPair;
  p.tiles_t = (int)((p.M + 255) / 256);
  const int64_t per = (p.M + p.tiles_t - 1) / p.tiles_t;
  p.tn = (int)std::min<int64_t>(256, (per + 15) / 16 * 16);
  p.tiles_c = (int)(p.N / TCH);               // pairs = tiles_c / 2
  p.kblocks = (int)((p.K + BK - 1) / BK);
  const int64_t tiles = (int64_t)p.tiles_t * (p.tiles_c / 2);
  const int64_t ncl = std::max(1, nsm / 2);
  const int64_t cap = std::max<int64_t>(
      1, std::min<int64_t>({8, p.kblocks / 8, (2 * (kMaxSms / 2) + tiles - 1) / tiles}));
  // with one or two token tiles the weights stream from HBM in code stages of
  // kPairStageKb k-blocks, so splits are whole stages when K allows
  const int gran = (p.tiles_t <= 2 && p.kblocks % kPairStageKb == 0) ? kPairStageKb : 1;
  int best = 1;
  int64_t best_cost = -1;
  for (int s = 1; s <= cap; ++s) {
    const int kbs = ((p.kblocks + s - 1) / s + gran - 1) / gran * gran;
    if (s > 1 && (int64_t)(s - 1) * kbs >= p.kblocks) break;   // an empty split
    const int64_t rounds = (tiles * s + ncl - 1) / ncl;
    const int64_t cost = rounds * (kbs + 2) + (s > 1 ? 24 : 0);
    if (best_cost < 0 || cost < best_cost) {
      best = s;
      best_cost = cost;
    }
  }
  p.kb_per_split = ((p.kblocks + best - 1) / best + gran - 1) / gran * gran;
  p.splits = (p.kblocks + p.kb_per_split - 1) / p.kb_per_split;
  p.ws_bytes = (cap > 1) ? (size_t)cap * p.M * p.N * sizeof(float) : 0;
  // several token tiles: the units run in dynamic order from a counter after the partials
  if (p.tiles_t >= 2) {
    p.sched_off = (p.ws_bytes + 255) / 256 * 256;
    p.ws_bytes = p.sched_off + 256;
  }
  p.units = tiles * p.splits;
  p.grid = (int)(2 * std::min<int64_t>(p.units, ncl));
}

size_t gemm_ws_bytes(int64_t M, int64_t K, int64_t N) {
  if (M <= 0 || K <= 0 || N <= 0) return 0;
  return std::max(gemm_plan(M, K, N, kMaxSms, true).ws_bytes,
                  gemm_plan(M, K, N, kMaxSms, false).ws_bytes);
}

GemmPlan gemm_plan(int64_t M, int64_t K, int64_t N, int nsm, bool allow_pair) {
  GemmPlan p{};
  p.M = M; p.N = N; p.K = K;
  if (M > 0 && M <= 128) {
    stream_plan(p, nsm);
    return p;
  }
  if (allow_pair && pair_fits(M, N)) {
    pair_plan(p, nsm);
    return p;
  }
  p.kind = kGemmTiled;
  p.tiles_t = (int)std::max<int64_t>(1, (M + TN_MAX - 1) / TN_MAX);
  // tokens per tile: the smallest multiple of 16 that covers M in tiles_t tiles
  const int64_t per = (M + p.tiles_t - 1) / p.tiles_t;
  p.tn = (int)std::min<int64_t>(TN_MAX, std::max<int64_t>(16, (per + 15) / 16 * 16));
  p.tiles_c = (int)((N + TCH - 1) / TCH);
  p.kblocks = (int)((K + BK - 1) / BK);
  const int64_t tiles = (int64_t)p.tiles_t * p.tiles_c;
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

// The split-K reduce: 8 outputs per thread, or with a LayerNorm one row per CTA.
static cudaError_t launch_reduce(const GemmPlan& p, void* ws, const EpiArgs& ea, const LnOut* ln,
                                 cudaStream_t st) {
  const float* part = static_cast<const float*>(ws);
  if (ln) {
    if (p.N > 256 * 8 * kLnChunks || p.M > 0x7FFFFFFF) return cudaErrorInvalidValue;
    return launch_pdl(gemm_reduce_ln_kernel, dim3((unsigned)p.M), dim3(256), 0, st, part, p.splits,
                      p.M, (int)p.N, ea, ln->gamma, ln->beta, ln->eps, ln->y);
  }
  const int64_t chunks = p.M * (p.N / 8);
  return launch_pdl(gemm_reduce_kernel, dim3((unsigned)((chunks + 255) / 256)), dim3(256), 0, st,
                    part, p.splits, p.M, (int)p.N, ea);
}

cudaError_t launch_gemm(const GemmPlan& p, const uint16_t* X, const fg_q4mat& W,
                        const uint16_t* bias, int epi, const uint16_t* residual, uint16_t* Y,
                        void* ws, cudaStream_t st, cudaEvent_t mid_event, const KvOut* kv,
                        const LnOut* ln, const uint16_t* w16) {
  if (p.M == 0) return cudaSuccess;
  if (ln && p.splits == 1) return cudaErrorInvalidValue;     // the caller runs LayerNorm
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  static cudaError_t attr_err = [] {
    cudaError_t e0 = cudaFuncSetAttribute(gemm_q4_tc_kernel<false>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    cudaError_t e1 = cudaFuncSetAttribute(gemm_q4_tc_kernel<true>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    return e0 != cudaSuccess ? e0 : e1;
  }();
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap tmX, tmC, tmS;
  e = make_map_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X, (uint64_t)p.K, (uint64_t)p.M,
                  (uint64_t)p.K * 2, BK, (uint32_t)p.tn, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = make_map_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, W.codes, (uint64_t)(p.N / 2),
                  (uint64_t)p.K, (uint64_t)(p.N / 2), TCH / 2, BK, CU_TENSOR_MAP_SWIZZLE_64B);
  if (e != cudaSuccess) return e;
  e = make_map_2d(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT32, W.ab, (uint64_t)(p.N / 64),
                  (uint64_t)p.K, (uint64_t)(p.N / 64) * 4, 4, BK, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  const EpiArgs final_ea{bias, residual, Y, nullptr, epi, kv ? *kv : KvOut{}};
  EpiArgs ea = final_ea;
  if (p.splits > 1) ea.partial = static_cast<float*>(ws);
  if (p.kind == kGemmPair) {
    if (kv && kv->k_codes) return cudaErrorInvalidValue;   // the append lives in kind 0/1
    e = launch_gemm_pair(p, W, X, ea, st, w16, ws);
    if (e != cudaSuccess || p.splits == 1) return e;
    if (mid_event) cudaEventRecord(mid_event, st);
    return launch_reduce(p, ws, final_ea, ln, st);
  }
  if (p.kind == kGemmStream) {
    e = launch_gemm_stream(p, W, tmX, ea, st);
    if (e != cudaSuccess || p.splits == 1) return e;
    if (mid_event) cudaEventRecord(mid_event, st);
    return launch_reduce(p, ws, final_ea, ln, st);
  }
  // ring depths: large token tiles (prefill) pair each restored slot with an X slot (4 + 4,
  // 6 code stages); small ones (decode) keep 6 X slots (L2 latency of the X tile) and spend
  // the rest on restored slots (so a restore waits for the MMAs of a k-block many k-blocks
  // back) and code stages (about 12: 60 KB of codes from HBM in flight per SM)
  const int xb = p.tn * 128;
  int rx, rc_target;
  if (p.tn > 128) {
    rx = 0;
    rc_target = 6;
  } else {
    rx = 6;
    rc_target = 10;
  }
  int ra;
  if (rx == 0) {
    ra = std::min(RA_MAX, (POOL_BYTES - rc_target * CS_BYTES) / (W_BYTES + xb));
    rx = ra;
  } else {
    ra = std::min(RA_MAX, (POOL_BYTES - rc_target * CS_BYTES - rx * xb) / W_BYTES);
  }
  const int rc = std::min(RC_MAX, (POOL_BYTES - ra * W_BYTES - rx * xb) / CS_BYTES) / RG * RG;
  if (ra < RG || rx < 2 || rx > ra || rc < RG || rc % RG != 0 ||
      ra * W_BYTES + rx * xb + rc * CS_BYTES > POOL_BYTES)
    return cudaErrorInvalidConfiguration;
  // two MMA issuers when the token tile fits two accumulators per buffer and every unit
  // has at least one k-block for each
  const int last_unit_kb = p.kblocks - (p.splits - 1) * p.kb_per_split;
  const int ni = (p.tn <= 128 && p.kb_per_split >= 2 && last_unit_kb >= 2) ? 2 : 1;
  const KArgs ka{(int)p.M, (int)p.N, (int)p.K, p.tn, make_idesc(p.tn), p.tiles_t, p.tiles_c,
                 p.kblocks, p.kb_per_split, (int)p.units, ra, rx, ni, rc};
  const bool with_kv = ea.kv.k_codes != nullptr && p.splits == 1;
  e = launch_pdl(with_kv ? gemm_q4_tc_kernel<true> : gemm_q4_tc_kernel<false>,
                 dim3((unsigned)p.grid), dim3(THREADS), SMEM_BYTES, st, tmX, tmC,
                 tmS, ka, ea);
  if (e != cudaSuccess || p.splits == 1) return e;
  if (mid_event) cudaEventRecord(mid_event, st);
  return launch_reduce(p, ws, final_ea, ln, st);
}

cudaError_t gemm_read_error(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_gemm_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(unsigned int));
}

}  // namespace fg
