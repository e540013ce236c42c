// Weight-streaming dequant-fused GEMM for few tokens (sm_103a):
//   Y[M][N] = epi( X[M][K] * W^[K][N] + bias ),   M <= 128 (decode: M = B)
// W^ restored to fp16 from 4-bit codes grouped 64 along the output channel N with
// per-group (a, b) [FlexGen review (jaehun.me), "4-bit 압축은 정수 연산 가속과 같은가":
// weights grouped along the output channel, restored to FP16 before compute].
//
// With few tokens the weights are the traffic: each 4-bit code is read once from HBM and
// used by M tokens.  The tiled kernel restores weights into shared memory as the MMA's A
// operand; with N = M <= 128 tokens per MMA the tensor core then spends its shared-memory
// bandwidth reading 4 KB of A per K = 16 step while the restorers write the next tile.
// Here the restored weights go to tensor memory: tcgen05.mma reads A from TMEM (lane =
// output channel, one 32-bit column = two consecutive k) and only the X tile (B) from
// shared memory.
//
// Restore.  A code word holds 8 consecutive output channels at one k.  A warp owns the 32
// channels of one TMEM lane quarter.  For each 8 k-rows a lane loads one word and one
// movmatrix transposes the 8 x 8 matrix of 16-bit elements (4 channels each): lane (g, t)
// then holds channels 4g..4g+3 at k = 2t and 2t+1, i.e. one TMEM column (a k pair) of four
// channels.  Each pair is restored with one HFMA2: the nibble OR-ed into mantissa bits
// 6..9 of 1.0h is 1 + q/16, and (1 + q/16) * 16s + (a - 16s) = a + q*s with the (s, a) of
// the two k-rows.  tcgen05.st.16x128b writes register 0 to lane g and register 1 to lane
// 8 + g (lanes 16 + g and 24 + g with the 16-lane offset), column t: TMEM lane 8j + g of a
// quarter holds channel 4g + j of the quarter's 32, which the epilogue maps back.
//
// Loads.  A thread that issues a TMA copy waits several hundred cycles before it can issue
// the next, whatever the copy's size (measured: ~600 cycles for 1 KB to 16 KB), so the copy
// count per weight byte sets the pace.  Codes and statistics move in stages of four k-blocks
// (one 256-row box each: 16 KB + 4 KB) from two producer threads taking alternate stages, and
// the X tiles (one per k-block) from four producer threads.
//
// Persistent kernel, one CTA per SM over (split, 128-channel tile) units, K step 64:
//   warps 0, 2, 16, 17  X producers (RPAR = 2): thread p loads the X tiles (tn x 64, 128B swizzle,
//               K-major) of k-blocks == p (mod 4) into an X ring; a tile completes on its
//               k-block's A barrier.  Warp 0 owns TMEM: 512 columns = accumulators (two
//               buffers of two issuers' tn columns when tn <= 64, else one buffer) and an
//               8-stage A ring of 32 columns
//   warps 1, 3  one thread each issues tcgen05.mma (kind::f16, M = 128, N = tn, K = 16, A
//               in TMEM) for alternate k-blocks into its own accumulator, and commits every
//               k-block, which frees its A stage and X slot
//   warps 18, 19  code producers: code and statistics boxes of alternate stages into a code
//               ring of up to 8 stages (the HBM stream: ~120 KB in flight per SM)
//   warps 4-11  restore: warp 4 + 4r + q restores lane quarter q of the k-blocks of every
//               stage whose position in the stage is == r (mod 2)
//   warps 12-15 epilogue of the previous unit (tcgen05.ld, lane = channel): bias / ReLU /
//               residual in fp32 and fp16 stores, or fp32 split-K partials
//
// Every mbarrier wait is bounded (about 2 s); on timeout the CTA raises an abort flag,
// sets the device error word, drains its outstanding copies and exits.
#include <cuda.h>

#include <algorithm>

#include "fg_common.cuh"
#include "fg_internal.h"
#include "gemm_tc.cuh"

namespace fg {

__device__ unsigned int g_gemm_stream_error = 0;

namespace {

constexpr int TCH = 128;                    // output channels per tile (MMA M, TMEM lanes)
constexpr int TN_MAX = 128;                 // tokens (MMA N)
constexpr int NI = 2;                       // MMA issuing threads (warps 1 and 3)
constexpr uint32_t ACC_COLS = 256;          // accumulators: nbuf buffers x NI issuers x tn
constexpr int BK = 64;
constexpr int RA = 8;                       // A stages in TMEM (32 columns each)
constexpr int SK = kStreamStage;            // k-blocks per code stage
constexpr int RC_MAX = 8;                   // code stages
constexpr int NXP = 4;                      // X producer threads
constexpr int RPAR = 2;                     // restore warps per lane quarter
constexpr int RW0 = 4;                      // first restore warp
constexpr int RW = 4 * RPAR;                // restore warps
constexpr int EW0 = RW0 + RW;               // first epilogue warp (4 warps)
constexpr int XW2 = EW0 + 4;                // X producer warps 0, 2, XW2, XW2 + 1
constexpr int CW0 = XW2 + 2;                // code producer warps CW0, CW0 + 1
constexpr int THREADS = (CW0 + 2) * 32;
constexpr int C_BYTES = BK * TCH / 2;       // 4 KB of codes per k-block (64-byte rows)
constexpr int S_BYTES = BK * 4 * 4;         // 1 KB: (a, b) words of 4 groups x 64 k-rows
constexpr int CS_BYTES = SK * (C_BYTES + S_BYTES);  // one code stage: codes, then statistics
constexpr int SMEM_BYTES = 232448;
constexpr int BAR_BYTES = 640 + 1024;      // barriers, then the epilogue's exchange words
constexpr int XCH_OFF = 640;
constexpr int POOL_BYTES = SMEM_BYTES - 1024 /*align*/ - BAR_BYTES;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_COL0 = ACC_COLS;       // A ring after the accumulators
static_assert(A_COL0 + RA * (BK / 2) == TMEM_COLS, "TMEM budget");
static_assert((2 * RC_MAX + 2 * RA + 5) * 8 + 8 <= XCH_OFF, "barrier space");
static_assert(CS_BYTES % 1024 == 0 && (SK * C_BYTES) % 512 == 0, "stage alignment");
static_assert(SK % RPAR == 0, "restore warps take every RPAR-th position of a stage");
constexpr long long kWaitCycles = 1ll << 32;

struct SArgs {
  int M, N, K, tn;
  uint32_t idesc;
  int tiles_c, kblocks, kb_per_split, units;
  int rx, rc;
  int nbuf;                     // accumulator buffers: 2 (epilogue overlaps the next unit) or 1
  const uint8_t* codes;         // the weight (the tensor maps address the same memory)
  const uint32_t* ab;
};

struct SUnit {
  int c0, split, kb_begin, kb_end;
};
__device__ __forceinline__ SUnit stream_unit(int u, const SArgs& ka) {
  SUnit r;
  r.split = u / ka.tiles_c;
  r.c0 = (u - r.split * ka.tiles_c) * TCH;
  r.kb_begin = r.split * ka.kb_per_split;
  r.kb_end = min(ka.kblocks, r.kb_begin + ka.kb_per_split);
  return r;
}

__device__ __forceinline__ bool swait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      atomicOr(&g_gemm_stream_error, 1u);
      return false;
    }
  }
  return true;
}

// D[tmem_d] (+)= A[tmem_a] * B[bdesc]: A read from tensor memory.
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 lanes x 32 columns: register 2i -> (lane g, column 4i + t), 2i + 1 -> (lane 8 + g,
// column 4i + t) for lane (g, t) of the warp.
__device__ __forceinline__ void tmem_st_16x128b_x8(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// (16s, a - 16s) of one group's (a, b) word, s = (b - a)/15.
__device__ __forceinline__ float2 restore_consts(uint32_t ab) {
  const float2 f = unpack_h2(ab);
  const float s16 = (f.y - f.x) * (16.0f / 15.0f);
  return make_float2(s16, f.x - s16);
}

// KV: the K/V append in the epilogue (a separate instance, so that the plain GEMM carries
// none of its code: the larger kernel measured slower even when the append never ran).
template <bool KV>
__global__ void __launch_bounds__(THREADS, 1)
gemm_q4_stream_kernel(const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ CUtensorMap tmC,
                      const __grid_constant__ CUtensorMap tmS, const SArgs ka, const EpiArgs ea) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int RX = ka.rx, RC = ka.rc, tn = ka.tn;
  const int XB = tn * 128;                             // one X tile (a multiple of 2 KB)
  uint8_t* sX = smem;                                  // RX x XB
  uint8_t* sC = sX + RX * XB;                          // RC x (codes, statistics)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sC + RC * CS_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * RC_MAX + 2 * RA + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // K/V append: per-token min/max words of the four lane quarters, two buffers
  uint32_t* xch = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(bars) + XCH_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(bars);
  auto full_c = [&](int s) { return bar0 + 8u * s; };
  auto free_c = [&](int s) { return bar0 + 8u * (RC_MAX + s); };
  auto full_a = [&](int s) { return bar0 + 8u * (2 * RC_MAX + s); };
  auto mma_done = [&](int s) { return bar0 + 8u * (2 * RC_MAX + RA + s); };
  auto acc_full = [&](int s) { return bar0 + 8u * (2 * RC_MAX + 2 * RA + s); };
  auto acc_empty = [&](int s) { return bar0 + 8u * (2 * RC_MAX + 2 * RA + 2 + s); };
  const uint32_t xchg = bar0 + 8u * (2 * RC_MAX + 2 * RA + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < RC; ++s) {
      mbar_init(full_c(s), 1);
      mbar_init(free_c(s), RW * (SK / RPAR));    // each restore warp, per stage position
    }
    for (int s = 0; s < RA; ++s) {
      mbar_init(full_a(s), 4 + 1);               // four restore warps + the X producer
      mbar_init(mma_done(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(acc_full(s), NI);                // one commit per MMA issuer
      mbar_init(acc_empty(s), 4);                // one arrival per epilogue warp
    }
    mbar_init(xchg, 4);                          // one arrival per epilogue warp
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

  const int xp = (warp == 0) ? 0 : (warp == 2) ? 1 : (warp == XW2) ? 2 : (warp == XW2 + 1) ? 3 : -1;
  if (xp >= 0) {
    // ------------------------------------------------------------ X producers
    // Thread xp loads the X tiles of k-blocks == xp (mod NXP).  The X ring has as many
    // slots as the A ring: the slot of k-block it is free once the MMAs of k-block it - RA
    // are done, and that barrier cannot move a further phase before this tile lands.
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < ka.units && ok; u += gridDim.x) {
        const SUnit w = stream_unit(u, ka);
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++it) {
          if (it % NXP != xp) continue;
          if (it >= RA && !swait(mma_done(it % RA), ((it / RA) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(full_a(it % RA), (uint32_t)XB);
          tma_load_2d(smem_u32(sX + (it % RA) * XB), &tmX, kb * BK, 0, full_a(it % RA));
        }
      }
      // after an abort the k-block barriers may lack restore arrivals: short waits
      if (!ok) {
        for (int i = max(0, it - RA); i < it; ++i) {
          if (i % NXP != xp) continue;
          const long long t0 = clock64();
          while (!mbar_try(full_a(i % RA), (i / RA) & 1)) {
            if (clock64() - t0 > (1ll << 26)) {
              atomicOr(&g_gemm_stream_error, 2u);
              break;
            }
          }
        }
      }
    }
  } else if (warp >= CW0 && warp < CW0 + 2) {
    // ------------------------------------------------------------ code producers
    // Thread cp loads stages == cp (mod 2): the codes and the statistics of SK k-blocks
    // (256 k-rows; rows past K read as zeros).
    const int cp = warp - CW0;
    if (lane == 0) {
      int st = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < ka.units && ok; u += gridDim.x) {
        const SUnit w = stream_unit(u, ka);
        const int nst = (w.kb_end - w.kb_begin + SK - 1) / SK;
        for (int g = 0; g < nst; ++g, ++st) {
          if (st % 2 != cp) continue;
          const int c = st % RC;
          if (st >= RC && !swait(free_c(c), ((st / RC) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          // the stage was last read through the generic proxy
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          uint8_t* cs = sC + c * CS_BYTES;
          const int k0 = (w.kb_begin + g * SK) * BK;
          mbar_expect_tx(full_c(c), (uint32_t)CS_BYTES);
          tma_load_2d(smem_u32(cs), &tmC, w.c0 / 2, k0, full_c(c));
          tma_load_2d(smem_u32(cs + SK * C_BYTES), &tmS, (w.c0 / 256) * 4, k0, full_c(c));
        }
      }
      // every issued load lands before the CTA exits
      for (int i = max(0, st - RC); i < st; ++i) {
        if (i % 2 != cp) continue;
        const long long t0 = clock64();
        while (!mbar_try(full_c(i % RC), (i / RC) & 1)) {
          if (clock64() - t0 > kWaitCycles) {
            atomicOr(&g_gemm_stream_error, 2u);
            break;
          }
        }
      }
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    // One thread issuing every tcgen05 op of the CTA spends tens of cycles per op, more
    // than the tensor pipe needs for an N <= 128 MMA; issuer mi takes the k-blocks with
    // index == mi (mod NI) into its own accumulator, and the epilogue adds them.
    const int mi = warp >> 1;
    if (lane == 0) {
      // X slot offsets and the K16 step add (bytes >> 4) to the start-address field
      const uint64_t bdesc0 = smem_desc(smem_u32(sX), 16, 1024);
      const uint64_t b_step = (uint64_t)(XB >> 4);
      int tl = 0, it = 0, r = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < ka.units && ok; u += gridDim.x, ++tl) {
        const SUnit w = stream_unit(u, ka);
        const int b = tl % ka.nbuf, use = tl / ka.nbuf;
        if (tl >= ka.nbuf && !swait(acc_empty(b), (use & 1) ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t tacc = tmem + (uint32_t)((b * NI + mi) * tn);
        uint32_t accumulate = 0u;
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++it) {
          const int cr = r;                          // A stage and X slot of k-block it
          const uint32_t cph = ph;
          if (++r == RA) {
            r = 0;
            ph ^= 1;
          }
          if (it % NI != mi) continue;
          if (!swait(full_a(cr), cph, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ta = tmem + A_COL0 + cr * (BK / 2);
          const uint64_t bd = bdesc0 + (uint64_t)cr * b_step;
          umma_f16_tmem_a(tacc, ta, bd, ka.idesc, accumulate);
          umma_f16_tmem_a(tacc, ta + 8, bd + 2, ka.idesc, 1u);
          umma_f16_tmem_a(tacc, ta + 16, bd + 4, ka.idesc, 1u);
          umma_f16_tmem_a(tacc, ta + 24, bd + 6, ka.idesc, 1u);
          umma_commit(mma_done(cr));
          accumulate = 1u;
        }
        if (!ok) break;
        umma_commit(acc_full(b));
      }
    }
  } else if (warp >= RW0 && warp < EW0) {
    // ------------------------------------------------------------ restore codes -> TMEM
    const int q = warp & 3, rr = (warp - RW0) >> 2;
    const int gid = lane >> 2, tig = lane & 3;
    // word of k-row 8rb + gid, channels 32q + 8tig .. +7: the 64B swizzle puts 16-byte
    // chunk q of k-row k at chunk q ^ ((k >> 1) & 3), and (k >> 1) & 3 = (gid >> 1) & 3
    const int code_off = gid * 64 + ((q ^ ((gid >> 1) & 3)) << 4) + tig * 4;
    const uint32_t t_lo = tmem + ((uint32_t)(32 * q) << 16) + A_COL0;
    const uint32_t t_hi = t_lo + (16u << 16);
    int it0 = 0, st = 0;                              // first k-block of the unit, stage
    bool ok = true;
    for (int u = blockIdx.x; u < ka.units && ok; u += gridDim.x) {
      const SUnit w = stream_unit(u, ka);
      const int L = w.kb_end - w.kb_begin;
      const int nst = (L + SK - 1) / SK;
      const int gw = ((w.c0 >> 6) & 3) + (q >> 1);     // this quarter's group in the box
      for (int g = 0; g < nst && ok; ++g, ++st) {
        const int c = st % RC;
        if (!swait(full_c(c), (st / RC) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* cs = sC + c * CS_BYTES;
        // this warp's positions j of the stage: its k-blocks, or an arrival alone when the
        // unit ends inside the stage
#pragma unroll 1
        for (int j = rr; j < SK; j += RPAR) {
          const int jj = g * SK + j;
          if (jj >= L) {
            if (lane == 0) mbar_arrive(free_c(c));
            continue;
          }
          const int it = it0 + jj, cr = it % RA;
          const uint8_t* cj = cs + j * C_BYTES;
          const uint32_t* ss = reinterpret_cast<const uint32_t*>(cs + SK * C_BYTES + j * S_BYTES);
          uint32_t cw[8];
#pragma unroll
          for (int rb = 0; rb < 8; ++rb)
            cw[rb] = *reinterpret_cast<const uint32_t*>(cj + code_off + rb * 512);
          // restore constants of k-rows 2*lane and 2*lane + 1 as half2 pairs
          const float2 k0 = restore_consts(ss[(2 * lane) * 4 + gw]);
          const float2 k1 = restore_consts(ss[(2 * lane + 1) * 4 + gw]);
          const uint32_t sp = pack_h2(k0.x, k1.x), cp = pack_h2(k0.y, k1.y);
          // the A stage is free once the MMAs of k-block it - RA are done
          if (it >= RA && !swait(mma_done(cr), ((it / RA) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          uint32_t lo[16], hi[16];
#pragma unroll
          for (int rb = 0; rb < 8; ++rb) {
            const uint32_t xw = movtrans(cw[rb]);
            const uint32_t s16 = __shfl_sync(0xFFFFFFFFu, sp, 4 * rb + tig);
            const uint32_t c16 = __shfl_sync(0xFFFFFFFFu, cp, 4 * rb + tig);
            const uint4 e = restore8(xw, s16, c16);     // channels 4g + 0..3, k pair t
            lo[2 * rb] = e.x;
            lo[2 * rb + 1] = e.y;
            hi[2 * rb] = e.z;
            hi[2 * rb + 1] = e.w;
          }
          // this position of the stage may be refilled: every lane's words are consumed
          __syncwarp();
          if (lane == 0) mbar_arrive(free_c(c));
          tmem_st_16x128b_x8(t_lo + cr * (BK / 2), lo);
          tmem_st_16x128b_x8(t_hi + cr * (BK / 2), hi);
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(full_a(cr));
        }
      }
      it0 += L;
    }
  } else if (warp >= EW0 && warp < EW0 + 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int ch_in_tile = 32 * q + 4 * (lane & 7) + (lane >> 3);
    const int64_t N = ka.N;
    const int M = ka.M;
    int tl = 0, it = 0;
    uint32_t xph = 0;                                 // K/V exchanges so far
    bool fail = false;
    for (int u = blockIdx.x; u < ka.units; u += gridDim.x, ++tl) {
      const SUnit w = stream_unit(u, ka);
      const int b = tl % ka.nbuf, use = tl / ka.nbuf;
      // the warp-collective TMEM loads below need the whole warp: decide for all its lanes
      if (!__all_sync(0xFFFFFFFFu, swait(acc_full(b), use & 1, abort_flag))) break;
      tc_fence_after();
      // issuer mi accumulated this unit iff one of its k-blocks it .. it + L - 1 is == mi
      // (mod NI)
      const int L = w.kb_end - w.kb_begin;
      const int64_t ch = w.c0 + ch_in_tile;
      const float bias_f = (!ea.partial && ea.bias) ? h2f(ea.bias[ch]) : 0.0f;
      // a K or V tile of the QKV projection (h is a multiple of 128: no tile straddles)
      const bool kv_tile = KV && ea.kv.k_codes != nullptr && !ea.partial && w.c0 >= ea.kv.h;
      // column part of this lane's destination: its code word (lanes 0, 2, 4, 6: channels
      // 32q + 4 lane ..) and the group's statistics word (quarters 0 and 2)
      const KvCol kcol = kv_tile ? kv_col(ea.kv, w.c0 + 32 * q + 4 * (lane & 6)) : KvCol{};
      for (int cb = 0; cb < M; cb += 32) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
        for (int m = 0; m < NI; ++m) {
          if (L < NI && (m - it % NI + NI) % NI >= L) continue;
          uint32_t rv[32];
          __syncwarp();
          const uint32_t taddr =
              tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)((b * NI + m) * tn + cb);
          tmem_ld16(taddr, rv);
          tmem_ld16(taddr + 16, rv + 16);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] += __uint_as_float(rv[i]);
        }
        if (ea.partial) {
          float* pp = ea.partial + ((int64_t)w.split * M + cb) * N + ch;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (cb + i < M) pp[(int64_t)i * N] = v[i];
          continue;
        }
        uint32_t yp[16];                              // the stored fp16 outputs, in pairs
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float y = v[i] + bias_f;
          if (ea.epi == FG_EPI_RELU) y = fmaxf(y, 0.0f);
          else if (ea.epi == FG_EPI_RESIDUAL && cb + i < M) y += h2f(ea.residual[(cb + i) * N + ch]);
          const uint32_t yh = f2h(y);
          yp[i >> 1] = (i & 1) ? (yp[i >> 1] | (yh << 16)) : yh;
          if (cb + i < M) ea.Y[(int64_t)(cb + i) * N + ch] = (uint16_t)yh;
        }
        if (!kv_tile) continue;
        // ---- K/V append.  A 64-channel group is two lane quarters (q, q ^ 1): the min/max
        // of token i over this quarter's 32 channels goes to lane i, then to the partner
        // through shared memory
        uint32_t my = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t k = order_key((yp[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
          const uint32_t kmin = __reduce_min_sync(0xFFFFFFFFu, k);
          const uint32_t kmaxn = __reduce_min_sync(0xFFFFFFFFu, ~k & 0xFFFFu);
          if (lane == i) my = kmin | (kmaxn << 16);
        }
        uint32_t* xb = xch + (xph & 1) * 128;
        xb[32 * q + lane] = my;
        __syncwarp();
        if (lane == 0) mbar_arrive(xchg);
        if (!swait(xchg, xph & 1, abort_flag)) {
          fail = true;
          break;
        }
        ++xph;
        const uint32_t abw = q4_ab_word(__vminu2(my, xb[32 * (q ^ 1) + lane]));
        const Q4Group gl = q4_group(abw);             // the group of token cb + lane
        const int krow = (cb + lane < M) ? kv_row(ea.kv, cb + lane) : 0;
        if ((q & 1) == 0 && cb + lane < M) *kv_ab_at(ea.kv, kcol, krow) = abw;
        // lanes 0, 2, 4, 6 store the code words of channels 32q + 8j .. + 7 (j = lane / 2);
        // this lane's channel is nibble 4 (lane & 1) + (lane >> 3) of its word
        const int sh = 4 * (4 * (lane & 1) + (lane >> 3));
        // c15 of a constant group is not finite (b - a = 0): its codes are 0, never near
        const float c15l = (gl.bma == 0.0f) ? 0.0f : gl.c15;
        uint32_t nearbits = 0;                        // tokens with a code near a tie
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (cb + i >= M) break;
          const float af = __shfl_sync(0xFFFFFFFFu, gl.af, i);
          const float c15 = __shfl_sync(0xFFFFFFFFu, c15l, i);
          const int kr = __shfl_sync(0xFFFFFFFFu, krow, i);
          const float x = h2f((uint16_t)(yp[i >> 1] >> (16 * (i & 1))));
          bool nr = false;
          uint32_t cw = q4_code_fast(x, af, c15, nr) << sh;
          nearbits |= (uint32_t)nr << i;
          cw |= __shfl_xor_sync(0xFFFFFFFFu, cw, 1);
          cw |= __shfl_xor_sync(0xFFFFFFFFu, cw, 8);
          cw |= __shfl_xor_sync(0xFFFFFFFFu, cw, 16);
          if ((lane & 0x19) == 0) *kv_codes_at(ea.kv, kcol, kr) = cw;
        }
        // rare: tokens with a code near a tie; their words again with the exact division,
        // from the outputs this thread stored to Y
        nearbits = __reduce_or_sync(0xFFFFFFFFu, nearbits);
        while (nearbits) {
          const int i = __ffs(nearbits) - 1;
          nearbits &= nearbits - 1;
          {
            const float af = __shfl_sync(0xFFFFFFFFu, gl.af, i);
            const float bma = __shfl_sync(0xFFFFFFFFu, gl.bma, i);
            const int kr = __shfl_sync(0xFFFFFFFFu, krow, i);
            const float x = h2f(ea.Y[(int64_t)(cb + i) * N + ch]);     // stored by this thread
            uint32_t cw = q4_code(x, af, bma) << sh;
            cw |= __shfl_xor_sync(0xFFFFFFFFu, cw, 1);
            cw |= __shfl_xor_sync(0xFFFFFFFFu, cw, 8);
            cw |= __shfl_xor_sync(0xFFFFFFFFu, cw, 16);
            if ((lane & 0x19) == 0) *kv_codes_at(ea.kv, kcol, kr) = cw;
          }
        }
      }
      if (fail) break;
      it += L;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(b));
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

}  // namespace

cudaError_t launch_gemm_stream(const GemmPlan& p, const fg_q4mat& W, const CUtensorMap& tmX,
                               const EpiArgs& ea, cudaStream_t st) {
  if (p.tn > TN_MAX || p.tiles_t != 1) return cudaErrorInvalidValue;
  static cudaError_t attr_err = [] {
    cudaError_t e0 = cudaFuncSetAttribute(gemm_q4_stream_kernel<false>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    cudaError_t e1 = cudaFuncSetAttribute(gemm_q4_stream_kernel<true>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    return e0 != cudaSuccess ? e0 : e1;
  }();
  if (attr_err != cudaSuccess) return attr_err;
  // X ring: one slot per A stage; code ring: the rest of shared memory (the HBM stream)
  const int xb = p.tn * 128;
  const int rx = RA;
  const int rc = std::min(RC_MAX, (POOL_BYTES - rx * xb) / CS_BYTES);
  if (rc < 2) return cudaErrorInvalidConfiguration;
  // code and statistics boxes of a whole stage (SK k-blocks = 256 k-rows)
  CUtensorMap tmC4, tmS4;
  cudaError_t e = make_map_2d(&tmC4, CU_TENSOR_MAP_DATA_TYPE_UINT8, W.codes, (uint64_t)(p.N / 2),
                              (uint64_t)p.K, (uint64_t)(p.N / 2), TCH / 2, SK * BK,
                              CU_TENSOR_MAP_SWIZZLE_64B);
  if (e != cudaSuccess) return e;
  e = make_map_2d(&tmS4, CU_TENSOR_MAP_DATA_TYPE_UINT32, W.ab, (uint64_t)(p.N / 64),
                  (uint64_t)p.K, (uint64_t)(p.N / 64) * 4, 4, SK * BK, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  // instruction descriptor: D f32, A and B f16, both K-major, M = 128, N = tn
  const uint32_t idesc = (1u << 4) | ((uint32_t)(p.tn >> 3) << 17) | ((uint32_t)(TCH >> 4) << 24);
  const int nbuf = (2 * NI * p.tn <= (int)ACC_COLS) ? 2 : 1;
  const SArgs ka{(int)p.M, (int)p.N, (int)p.K, p.tn, idesc, p.tiles_c, p.kblocks,
                 p.kb_per_split, (int)p.units, rx, rc, nbuf, W.codes, W.ab};
  const bool with_kv = ea.kv.k_codes != nullptr && p.splits == 1;
  return launch_pdl(with_kv ? gemm_q4_stream_kernel<true> : gemm_q4_stream_kernel<false>,
                    dim3((unsigned)p.grid), dim3(THREADS), SMEM_BYTES, st,
                    tmX, tmC4, tmS4, ka, ea);
}

cudaError_t gemm_stream_read_error(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_gemm_stream_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_gemm_stream_error, &zero, sizeof(unsigned int));
}

}  // namespace fg
