// Causal prefill attention over fp16 Q/K/V on the 5th-generation tensor cores (sm_103a).
//
// The prefill step processes every prompt token at once and builds the KV cache
// [FlexGen paper explainer, "Problem Formulation", Figure 2].  Prefill attends over the
// fp16 K/V the projection just produced (the cache keeps the 4-bit copy for decoding).
// For query row i of a sequence and head: o_i = sum_{j <= i} softmax_j(scale * q_i . k_j) v_j.
//
// A CTA owns a block of 256 query rows of one (sequence, head): two Q tiles of 128 rows (A and
// B) that share every K/V tile of 128 keys.  Q, K and V are read in place from the [rows][3h]
// QKV buffer by TMA (boxes of 64 columns x 128 rows, 128B swizzle; d = 128 takes two).
//   S = Q K^T     tcgen05.mma kind::f16, M = 128 query rows, N = 128 keys, K = d: A = the Q
//                 tile and B = the K tile, both K-major in shared memory; S (fp32) in TMEM
//   softmax       two threads per query row (TMEM lane), each over one half of the 128 key
//                 columns: causal mask on the diagonal tile and past the sequence, the row
//                 maximum exchanged between the halves through shared memory, online base-2
//                 softmax with a lazily moved reference maximum (rescale only when a row's
//                 maximum grows by more than 2^8), P = 2^(s - m) rounded to fp16 and written
//                 back over the first 32 of the half's 64 S columns (two fp16 per column).
//                 Two passes over the half (the maximum, then P) keep a thread within 80
//                 registers.
//   O += P V      tcgen05.mma with A = P read from TMEM (K = 128 keys, in two blocks of 32
//                 columns), B = the V tile (MN-major: keys are its K, the head dimension its
//                 N); O (fp32) in TMEM
// The two Q tiles ping-pong: while one tile's softmax warps work on S, the tensor core runs the
// other tile's products.  TMEM: S of A and B (128 columns each), O of A and B (d columns each).
//   warp 0      TMA producer: the two Q tiles of a block, then its K/V tiles into a 2-stage ring
//   warp 1      MMA issuer: S_A(0), S_B(0); then per key tile j and Q tile t: P_t(j) V_j into
//               O_t, then S_t(j + 1) (the tensor core runs one thread's MMAs in issue order, so
//               S_t(j + 1) overwrites the columns of P_t(j) only after P_t(j) V_j has read them)
//   warps 2-9   softmax of Q tile A: warp w owns TMEM lanes 32 (w % 4) .. and key half
//               ((w - 2) / 4) & 1
//   warps 10-17 softmax of Q tile B
//   warps 18-21 output: O_t / l of a finished block from TMEM, fp16, staged in shared memory,
//               stored by TMA; a block's first P V product into O_t waits until they have
//               read the previous block's O_t, so the softmax warps go on to the next block
//               while the output is written
// A Q tile sees key tiles 0 .. (its last row) / 128; tiles wholly above its rows are skipped.
// The kernel is persistent (one CTA per SM over the blocks, heaviest first), so the next block's
// loads and first products overlap the current block's softmax and output.
//
// Every mbarrier wait is bounded; on timeout the CTA sets the device error word (read by
// fg_check_device_error), drains its copies and MMAs and frees TMEM.
#include <math.h>

#include <algorithm>
#include <mutex>

#include "fg_common.cuh"
#include "fg_internal.h"
#include "gemm_tc.cuh"

namespace fg {

__device__ unsigned int g_prefill_error = 0;

namespace {

constexpr int QT = 128;                     // query rows per Q tile (MMA M, TMEM lanes)
constexpr int KT = 128;                     // keys per K/V tile
constexpr int QB = 2 * QT;                  // query rows per CTA
constexpr int STAGES = 2;                   // K/V ring
constexpr int THREADS = 22 * 32;
constexpr int W_SM = 2;                     // softmax warps 2..17: Q tile (w - 2) / 8, key half
                                            // ((w - 2) / 4) & 1, TMEM lane quarter w % 4
constexpr int W_OUT = 18;                   // first output warp (18..21)
constexpr uint32_t TMEM_COLS = 512;
constexpr long long kWaitCycles = 1ll << 32;
constexpr int BOX = QT * 128;               // bytes of one 64-column x 128-row box

template <int D>
struct PSmem {
  static constexpr int TILE = (D / 64) * BOX;          // one Q, K or V tile
  static constexpr int Q_OFF = 0;                      // Q_A, Q_B
  static constexpr int K_OFF = 2 * TILE;               // K stages
  static constexpr int V_OFF = K_OFF + STAGES * TILE;  // V stages
  static constexpr int O_OFF = V_OFF + STAGES * TILE;  // one output box
  static constexpr int L_OFF = O_OFF + BOX;            // row sums l [tile][key half][row]
  static constexpr int MX_OFF = L_OFF + 2 * 2 * QT * 4;  // row maxima [parity][tile][half][row]
  static constexpr int BAR_OFF = MX_OFF + 2 * 2 * 2 * QT * 4;
  static constexpr int BYTES = BAR_OFF + 256 + 1024;   // barriers; 1024 for alignment
};
static_assert(PSmem<128>::BYTES <= 227 * 1024, "shared memory per CTA");

// barriers: q_full, q_free, kv_full[2], kv_free[2], s_full[2], p_full[2], o_done[2], o_free[2],
// l_full[2], o_staged, o_stage_free, drain, mx_ready[tile][quarter] (the two key halves of a
// row have written their maxima)
constexpr int B_QFULL = 0, B_QFREE = 1, B_KVFULL = 2, B_KVFREE = 4, B_SFULL = 6, B_PFULL = 8,
              B_ODONE = 10, B_OFREE = 12, B_LFULL = 14, B_OSTAGED = 16, B_OSFREE = 17,
              B_DRAIN = 18, B_MX = 19, NBARS = 27;
static_assert(NBARS * 8 + 8 <= 256, "barrier space");

__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      atomicOr(&g_prefill_error, 1u);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(&g_prefill_error, 2u);
      return;
    }
  }
}

// Tiled TMA store of a shared-memory box to global coordinates (x, y, z), tracked by the
// issuing thread's bulk async-group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* tm, uint32_t src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(tm)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the shared-memory sources of this thread's bulk stores have been read
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// this thread's bulk stores have completed
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// D[tmem_d] (+)= A[tmem_a] * B[bdesc], A read from tensor memory.
__device__ __forceinline__ void umma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
// Waits for this thread's TMEM loads and ties the 32 values of one to the wait, so that no
// use of them is scheduled before it.
__device__ __forceinline__ void tmem_wait_ld_dep(float (&v)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]),
        "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]),
        "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]), "+f"(v[18]), "+f"(v[19]),
        "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]), "+f"(v[24]), "+f"(v[25]),
        "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]), "+f"(v[30]), "+f"(v[31])
      :
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x on the special-function unit (x <= 0 here; results below 2^-126 flush to zero, far
// below the fp16 P fed to the P V product).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Blackwell's three-input maximum and packed two-lane fp32 arithmetic (one instruction for two
// elements).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// instruction descriptors: D f32, A and B f16, M = 128.  S = Q K^T: both operands K-major,
// N = 128 keys.  O += P V: A (P, in TMEM) K-major, B (V) MN-major, N = d.
constexpr uint32_t kIdescS = (1u << 4) | ((uint32_t)(KT >> 3) << 17) | ((uint32_t)(QT >> 4) << 24);
__host__ __device__ constexpr uint32_t idesc_pv(int d) {
  return (1u << 4) | (1u << 16) | ((uint32_t)(d >> 3) << 17) | ((uint32_t)(QT >> 4) << 24);
}

struct PArgsA {
  int nseq, s, H, h, qblocks;
  float scale_log2;
};

// A work item: a block of 256 query rows of one (sequence, head).  Items run heaviest first
// (the last query blocks see the most keys): item i is query block qblocks - 1 - i / (nseq H)
// of (sequence, head) i % (nseq H).
struct Item {
  int b, hd, q0, nt0, nt1, nkv;
};
__device__ __forceinline__ Item item_of(int i, const PArgsA& pa) {
  const int bhn = pa.nseq * pa.H;
  Item it;
  const int qb = pa.qblocks - 1 - i / bhn;
  const int bh = i % bhn;
  it.b = bh / pa.H;
  it.hd = bh % pa.H;
  it.q0 = qb * QB;
  // key tiles each Q tile sees (0 when the tile lies past the sequence)
  const int r1 = it.q0 + QT;
  it.nt0 = (min(pa.s, it.q0 + QT) + KT - 1) / KT;    // >= 1: the block starts below s
  it.nt1 = (r1 < pa.s) ? (min(pa.s, r1 + QT) + KT - 1) / KT : 0;
  it.nkv = max(it.nt0, it.nt1);
  return it;
}

// Persistent: CTA c takes items c, c + gridDim, ...  The producer loads the next item's Q as
// soon as the current item's last S product is done and streams K/V through the ring across
// items; the MMA issuer starts the next item's S products while the current item's last P V
// products run, and the output warps store an item's O while the softmax warps work on the next.
template <int D>
__global__ void __launch_bounds__(THREADS, 1)
prefill_attn_tc_kernel(const __grid_constant__ CUtensorMap tmQKV,
                       const __grid_constant__ CUtensorMap tmO, const PArgsA pa) {
  using L = PSmem<D>;
  constexpr int NB = D / 64;                           // 64-column boxes per tile
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* l_buf = reinterpret_cast<float*>(smem + L::L_OFF);
  float* mx_buf = reinterpret_cast<float*>(smem + L::MX_OFF);
  const uint32_t bar0 = smem_u32(bars);
  auto bar = [&](int i) { return bar0 + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nitems = pa.nseq * pa.H * pa.qblocks;
  const int s = pa.s;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QFREE), 1);
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(bar(B_KVFULL + i), 1);
      mbar_init(bar(B_KVFREE + i), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(B_SFULL + t), 1);
      mbar_init(bar(B_PFULL + t), 8);                  // one arrival per softmax warp
      mbar_init(bar(B_ODONE + t), 1);
      mbar_init(bar(B_OFREE + t), 4);                  // one arrival per output warp
      mbar_init(bar(B_LFULL + t), 8);                  // one arrival per softmax warp
      for (int q = 0; q < 4; ++q) mbar_init(bar(B_MX + 4 * t + q), 2);   // both key halves
    }
    mbar_init(bar(B_OSTAGED), 4);                      // one arrival per output warp
    mbar_init(bar(B_OSFREE), 1);
    mbar_init(bar(B_DRAIN), 1);
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
  // TMEM columns: S_A 0..127, S_B 128..255, O_A 256.., O_B 256 + D..
  auto s_col = [&](int t) { return (uint32_t)(t * KT); };
  auto o_col = [&](int t) { return (uint32_t)(2 * KT + t * D); };
  pdl_launch_dependents();
  pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int kvg = 0, qn = 0;                             // K/V tiles, Q pairs issued
      bool ok = true;
      for (int i = blockIdx.x; i < nitems && ok; i += gridDim.x) {
        const Item it = item_of(i, pa);
        const int row_base = it.b * s;
        // the previous item's S products are done with the Q tiles
        if (qn > 0 && !bwait(bar(B_QFREE), (uint32_t)((qn - 1) & 1), abort_flag)) {
          ok = false;
          break;
        }
        mbar_expect_tx(bar(B_QFULL), (uint32_t)(2 * L::TILE));
        for (int t = 0; t < 2; ++t)
          for (int c = 0; c < NB; ++c)
            tma_load_2d(smem_u32(smem + L::Q_OFF + t * L::TILE + c * BOX), &tmQKV,
                        it.hd * D + 64 * c, row_base + it.q0 + t * QT, bar(B_QFULL));
        ++qn;
        for (int j = 0; j < it.nkv; ++j, ++kvg) {
          const int st = kvg % STAGES;
          if (kvg >= STAGES &&
              !bwait(bar(B_KVFREE + st), (uint32_t)(((kvg / STAGES) & 1) ^ 1), abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar(B_KVFULL + st), (uint32_t)(2 * L::TILE));
          for (int c = 0; c < NB; ++c) {
            tma_load_2d(smem_u32(smem + L::K_OFF + st * L::TILE + c * BOX), &tmQKV,
                        pa.h + it.hd * D + 64 * c, row_base + j * KT, bar(B_KVFULL + st));
            tma_load_2d(smem_u32(smem + L::V_OFF + st * L::TILE + c * BOX), &tmQKV,
                        2 * pa.h + it.hd * D + 64 * c, row_base + j * KT, bar(B_KVFULL + st));
          }
        }
      }
      // every issued copy has landed before the CTA exits
      if (qn > 0) drain_wait(bar(B_QFULL), (uint32_t)((qn - 1) & 1));
      for (int i = max(0, kvg - STAGES); i < kvg; ++i)
        drain_wait(bar(B_KVFULL + i % STAGES), (uint32_t)((i / STAGES) & 1));
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t qbase = smem_u32(smem + L::Q_OFF), kbase = smem_u32(smem + L::K_OFF),
                     vbase = smem_u32(smem + L::V_OFF);
      const uint32_t idesc_o = idesc_pv(D);
      bool ok = true, issued = false;
      int kvg = 0, qn = 0;                             // K/V tiles, items consumed
      int pc[2] = {0, 0}, uses[2] = {0, 0};            // P V products; items, per Q tile
      // S_t = Q_t K^T of K/V tile g over K = D: k-step i reads 16 columns, 32 bytes into box
      // i / 4
      auto issue_s = [&](int t, int g) {
        const int st = g % STAGES;
        const uint64_t qd = smem_desc(qbase + t * L::TILE, 16, 1024);
        const uint64_t kd = smem_desc(kbase + st * L::TILE, 16, 1024);
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
          const uint64_t off = (uint64_t)(((i >> 2) * BOX + (i & 3) * 32) >> 4);
          umma_f16(tmem + s_col(t), qd + off, kd + off, kIdescS, i > 0 ? 1u : 0u);
        }
        umma_commit(bar(B_SFULL + t));
      };
      // O_t (+)= P_t V of K/V tile g over K = 128 keys: k-step i reads the 8 TMEM columns of
      // P of keys 16i.. (key half i / 4 keeps its P in the first 32 of its 64 S columns) and
      // rows 16i.. of V (2048 bytes per step in its MN-major 128B-swizzled layout)
      auto issue_pv = [&](int t, int g, bool first) {
        const int st = g % STAGES;
        const uint64_t vd = smem_desc(vbase + st * L::TILE, BOX, 1024);
#pragma unroll
        for (int i = 0; i < KT / 16; ++i)
          umma_ts(tmem + o_col(t), tmem + s_col(t) + 64 * (i >> 2) + 8 * (i & 3),
                  vd + (uint64_t)(i * 128), idesc_o, (!first || i > 0) ? 1u : 0u);
        umma_commit(bar(B_ODONE + t));
      };
      for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x, ++qn) {
        const Item it = item_of(item, pa);
        const int nt[2] = {it.nt0, it.nt1};
        if (!bwait(bar(B_QFULL), (uint32_t)(qn & 1), abort_flag) ||
            !bwait(bar(B_KVFULL + kvg % STAGES), (uint32_t)((kvg / STAGES) & 1), abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(0, kvg);
        if (it.nt1 > 0) issue_s(1, kvg);
        issued = true;
        if (it.nkv == 1) umma_commit(bar(B_QFREE));    // every S product of the item issued
        for (int j = 0; j < it.nkv && ok; ++j) {
          const int g = kvg + j;
          bool next_ready = false;                     // K/V of tile g + 1 waited for
          for (int t = 0; t < 2 && ok; ++t) {
            if (j >= nt[t]) continue;
            if (!bwait(bar(B_PFULL + t), (uint32_t)(pc[t] & 1), abort_flag)) {
              ok = false;
              break;
            }
            // the first product of an item overwrites O_t: the output warps have read it
            if (j == 0 && uses[t] > 0 &&
                !bwait(bar(B_OFREE + t), (uint32_t)((uses[t] - 1) & 1), abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(t, g, j == 0);
            ++pc[t];
            if (j + 1 < nt[t]) {
              if (!next_ready) {
                const int gn = g + 1;
                if (!bwait(bar(B_KVFULL + gn % STAGES), (uint32_t)((gn / STAGES) & 1),
                           abort_flag)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                next_ready = true;
              }
              issue_s(t, g + 1);
            }
          }
          if (j == it.nkv - 2) umma_commit(bar(B_QFREE));   // the item's last S products
          umma_commit(bar(B_KVFREE + g % STAGES));     // K/V tile g read by every MMA above
        }
        uses[0] += (it.nt0 > 0);
        uses[1] += (it.nt1 > 0);
        kvg += it.nkv;
      }
      // the CTA frees TMEM only after every MMA issued here has completed
      if (issued) {
        umma_commit(bar(B_DRAIN));
        drain_wait(bar(B_DRAIN), 0u);
      }
    }
  } else if (warp >= W_SM && warp < W_OUT) {
    // ------------------------------------------------------------ softmax: one key half of
    // one Q tile's rows.  Two threads per row: half c takes key columns 64c .. 64c + 63 of each
    // S tile, the row maximum is exchanged through shared memory (mx_ready barrier of the two
    // warps of a lane quarter), and half c writes its P over the first 32 of its own S columns
    // and rescales O columns c d/2 ..
    const int t = (warp - W_SM) >> 3, c = ((warp - W_SM) >> 2) & 1;
    const int quarter = warp & 3;                      // TMEM lanes 32 quarter ..
    const int m = 32 * quarter + lane;                 // row within the Q tile
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
    const uint32_t srow = lane_addr + s_col(t) + 64 * c;
    const uint32_t mxb = bar(B_MX + 4 * t + quarter);
    const float sl2 = pa.scale_log2;
    int sc = 0, uses = 0;                              // S products consumed, items finished
    bool ok = true;
    // tcgen05.ld / st are warp-collective (.sync.aligned): every branch around them is
    // decided for the whole warp, waits included (a lane that gave up takes its warp along);
    // both halves of a row take the same decisions (the same maximum)
    for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x) {
      const Item it = item_of(item, pa);
      const int nt = t ? it.nt1 : it.nt0;
      if (nt == 0) continue;
      const int qi = it.q0 + t * QT + m;               // query position in the sequence
      float m_ref = -INFINITY, l_sum = 0.0f;           // l over this half's keys
      for (int j = 0; j < nt; ++j, ++sc) {
        const bool got = bwait(bar(B_SFULL + t), (uint32_t)(sc & 1), abort_flag);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // keys past the row (diagonal tile) or past the sequence are masked: keys k0 .. k0 +
        // lim are visible
        const int k0 = j * KT;
        const bool masked = (k0 + KT - 1 > it.q0 + t * QT) || (k0 + KT > s);   // warp-uniform
        const int lim = min(qi, s - 1) - k0 - 64 * c;  // within this half's 64 columns
        // pass 1: this half's maximum, 32 columns at a time (the second load in flight)
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        auto max_chunk = [&](float (&v)[32], int c2) {
          if (masked) {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = (32 * c2 + e <= lim) ? v[e] : -INFINITY;
          }
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], v[e], v[e + 1]);
        };
        {
          float va[32], vb[32];
          tmem_ld32(srow, va);
          tmem_wait_ld_dep(va);
          tmem_ld32(srow + 32, vb);
          max_chunk(va, 0);
          tmem_wait_ld_dep(vb);
          max_chunk(vb, 1);
        }
        // the row maximum over both halves (slot of this tile's parity: the other half reads
        // it before either can write the slot again two tiles on)
        float* mx_slot = mx_buf + (((sc & 1) * 2 + t) * 2) * QT;
        mx_slot[c * QT + m] = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        __syncwarp();
        if (lane == 0) mbar_arrive(mxb);
        const bool ex = bwait(mxb, (uint32_t)(sc & 1), abort_flag);
        if (!__all_sync(0xFFFFFFFFu, ex)) {
          ok = false;
          break;
        }
        float mx = fmaxf(mx_slot[m], mx_slot[QT + m]);
        // in base 2 (scale > 0, so scaling after the maximum is the same); a row that sees no
        // key keeps a finite maximum (such rows lie past the sequence and are never stored)
        mx = (mx == -INFINITY) ? 0.0f : mx * sl2;
        if (__any_sync(0xFFFFFFFFu, mx > m_ref + 8.0f)) {
          // move the reference maximum of every row of the warp to max(m_ref, mx): O and l
          // scale by 2^(m_ref - m_new) (1 for rows whose maximum did not grow); O holds P V of
          // the item's earlier tiles once their MMAs are done; this half rescales its d/2
          // columns of O
          const float m_new = fmaxf(m_ref, mx);
          const float alpha = ex2(m_ref - m_new);
          if (j > 0) {
            const bool done = bwait(bar(B_ODONE + t), (uint32_t)((sc - 1) & 1), abort_flag);
            if (!__all_sync(0xFFFFFFFFu, done)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int c16 = 0; c16 < D / 32; ++c16) {
              uint32_t w[16];
              const uint32_t oa = lane_addr + o_col(t) + (uint32_t)(c * (D / 2) + 16 * c16);
              tmem_ld16(oa, w);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(__uint_as_float(w[e]) * alpha);
              tmem_st16(oa, w);
            }
            tmem_wait_st();
          }
          l_sum *= alpha;
          m_ref = m_new;
        }
        // pass 2: p = 2^(s * scale - m_ref), 32 columns at a time (the scaling and the row sums
        // two elements per instruction), packed to fp16 over columns 16 c2 .. of this half's S
        // (S columns that have been read)
        const uint64_t sl2x2 = f2pack(sl2, sl2), negm2 = f2pack(-m_ref, -m_ref);
        uint64_t ls2[2] = {f2pack(0.0f, 0.0f), f2pack(0.0f, 0.0f)};
        auto p_chunk = [&](float (&v)[32], int c2) {
          if (masked) {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = (32 * c2 + e <= lim) ? v[e] : -INFINITY;
          }
          uint32_t pw[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 x = f2unpack(ffma2(f2pack(v[e], v[e + 1]), sl2x2, negm2));
            const float p0 = ex2(x.x), p1 = ex2(x.y);
            ls2[(e >> 1) & 1] = fadd2(ls2[(e >> 1) & 1], f2pack(p0, p1));
            pw[e / 2] = pack_h2(p0, p1);
          }
          tmem_st16(srow + 16 * c2, pw);
        };
        {
          float va[32], vb[32];
          tmem_ld32(srow, va);
          tmem_wait_ld_dep(va);
          tmem_ld32(srow + 32, vb);
          p_chunk(va, 0);
          tmem_wait_ld_dep(vb);
          p_chunk(vb, 1);
        }
        tmem_wait_st();
        const float2 la = f2unpack(fadd2(ls2[0], ls2[1]));
        l_sum += la.x + la.y;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL + t));
      }
      if (!ok) break;
      // this half's row sums for the output warps, once they have taken the previous item's
      if (uses > 0) {
        const bool fr = bwait(bar(B_OFREE + t), (uint32_t)((uses - 1) & 1), abort_flag);
        if (!__all_sync(0xFFFFFFFFu, fr)) {
          ok = false;
          break;
        }
      }
      l_buf[(t * 2 + c) * QT + m] = l_sum;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_LFULL + t));
      ++uses;
    }
  } else if (warp >= W_OUT) {
    // ------------------------------------------------------------ output of both Q tiles
    const int quarter = warp & 3;
    const int m = 32 * quarter + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
    const bool leader = (warp == W_OUT) && lane == 0;  // issues the stores
    int cum[2] = {0, 0}, uses[2] = {0, 0}, nbox = 0;   // P V products, items, boxes stored
    bool ok = true;
    for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x) {
      const Item it = item_of(item, pa);
      for (int t = 0; t < 2 && ok; ++t) {
        const int nt = t ? it.nt1 : it.nt0;
        if (nt == 0) continue;
        cum[t] += nt;
        // the row sums, then the item's last P V product into O_t
        bool got = bwait(bar(B_LFULL + t), (uint32_t)(uses[t] & 1), abort_flag);
        got = got && bwait(bar(B_ODONE + t), (uint32_t)((cum[t] - 1) & 1), abort_flag);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        ++uses[t];
        const float inv = 1.0f / (l_buf[(t * 2) * QT + m] + l_buf[(t * 2 + 1) * QT + m]);
        // O / l in 64-column boxes, staged in shared memory (the 128B-swizzled layout of the
        // output map: 16-byte chunk k of row m at chunk k ^ (m % 8)) and stored by TMA; rows
        // past the sequence lie outside the map and are not written
#pragma unroll 1
        for (int hb = 0; hb < NB; ++hb, ++nbox) {
          const uint32_t stage = smem_u32(smem + L::O_OFF);
          if (nbox >= 1) {
            // the box is free once the previous store has read it
            if (leader) {
              bulk_wait_read();
              mbar_arrive(bar(B_OSFREE));
            }
            const bool fr = bwait(bar(B_OSFREE), (uint32_t)((nbox - 1) & 1), abort_flag);
            if (!__all_sync(0xFFFFFFFFu, fr)) {
              ok = false;
              break;
            }
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float o[32];
            tmem_ld32(lane_addr + o_col(t) + 64 * hb + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int k = 4 * c + i;
              const float* e = o + 8 * i;
              st_shared_v4(stage + 128 * m + ((k ^ (m & 7)) << 4),
                           pack_h2(e[0] * inv, e[1] * inv), pack_h2(e[2] * inv, e[3] * inv),
                           pack_h2(e[4] * inv, e[5] * inv), pack_h2(e[6] * inv, e[7] * inv));
            }
          }
          if (hb == NB - 1) {
            // O_t has been read: the next item's first P V product may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_OFREE + t));
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_OSTAGED));
          if (leader && bwait(bar(B_OSTAGED), (uint32_t)(nbox & 1), abort_flag)) {
            tma_store_3d(&tmO, stage, it.hd * D + 64 * hb, it.q0 + t * QT, it.b);
            bulk_commit();
          }
          __syncwarp();
        }
      }
    }
    // the CTA's shared memory stays valid until its stores have completed
    if (leader) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                 : "memory");
  }
}

template <int D>
cudaError_t launch_d(const uint16_t* qkv, int32_t nseq, int32_t s, int32_t H, float scale,
                     uint16_t* out, int nsm, cudaStream_t st) {
  static cudaError_t attr = cudaFuncSetAttribute(
      prefill_attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, PSmem<D>::BYTES);
  if (attr != cudaSuccess) return attr;
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  const int64_t h = (int64_t)H * D;
  CUtensorMap tm, tmo;
  e = make_map_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qkv, (uint64_t)(3 * h),
                  (uint64_t)nseq * s, (uint64_t)(3 * h) * 2, 64, QT, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  // the output as [nseq][s][h]: a box never spills into the next sequence's rows
  e = make_map_3d(&tmo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, out, (uint64_t)h, (uint64_t)s,
                  (uint64_t)nseq, (uint64_t)h * 2, (uint64_t)s * h * 2, 64, QT,
                  CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  const int qblocks = (s + QB - 1) / QB;
  const PArgsA pa{nseq, s, H, (int)h, qblocks, scale * 1.4426950408889634f};
  const int64_t items = (int64_t)nseq * H * qblocks;
  if (items > 0x7FFFFFFF || (int64_t)nseq * s > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const int64_t grid = std::min<int64_t>(items, std::max(1, nsm));   // one CTA per SM
  return launch_pdl(prefill_attn_tc_kernel<D>, dim3((unsigned)grid), dim3(THREADS),
                    PSmem<D>::BYTES, st, tm, tmo, pa);
}

}  // namespace

cudaError_t launch_prefill_attn(const uint16_t* qkv, int32_t nseq, int32_t s, int32_t H,
                                int32_t d, float scale, uint16_t* out, int nsm, cudaStream_t st) {
  if (nseq == 0 || s == 0) return cudaSuccess;
  return d == 128 ? launch_d<128>(qkv, nseq, s, H, scale, out, nsm, st)
                  : launch_d<64>(qkv, nseq, s, H, scale, out, nsm, st);
}

cudaError_t prefill_read_error(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_prefill_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(unsigned int));
}

}  // namespace fg
