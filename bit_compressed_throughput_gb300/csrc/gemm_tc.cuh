// tcgen05 / TMA / mbarrier helpers and the epilogue arguments shared by the two
// dequant-fused GEMM kernels of libfg (sm_103a): the tiled kernel for many tokens and the
// weight-streaming kernel for few (decode).
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "fg_internal.h"

namespace fg {

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
// Non-blocking probe of a phase: far cheaper than try_wait when the phase is already
// complete, which is the common case on the MMA issuer's path.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
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
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
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

// ---- CTA pairs (cluster of two CTAs on two SMs sharing one 2-CTA tensor-core MMA)
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address in the cluster's shared window of the variable at shared::cta address `addr` in
// the CTA of rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier of any CTA of the cluster (cluster-window address).  The arrive
// releases at CTA scope: a thread's prior stores to its own shared memory are performed
// before the arrival reaches the other CTA.  That is all the pair kernel needs: the data an
// arrival announces (a restored A slot, a read-out accumulator) belongs to the arriving CTA
// and is read by its own SM's tensor core, after the other CTA's thread has seen the
// barrier complete and issued the MMA.  A cluster-scope release here cost about 1900 cycles
// per k-block on a GB300 (a membar stall), which starved the tensor pipe.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cl_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cl_addr) : "memory");
}
// One MMA of the pair (issued by one thread of the even CTA): D[256][N] += A[256][16] *
// B[16][N], A rows 0..127 and TMEM lanes of D in the even CTA, rows 128..255 in the odd one;
// B columns 0..N/2-1 in the even CTA's shared memory, the rest in the odd one's, at the
// same offsets.
__device__ __forceinline__ void umma2_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the barrier at shared offset `bar` of every CTA in `cta_mask` when this
// thread's earlier pair MMAs are complete.
__device__ __forceinline__ void umma2_commit_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
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
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
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

// Epilogue of a GEMM launch: Y = epi(acc + bias), or fp32 partials for a split-K reduce.
// Destination of a K/V value: slot = (b*H + head)*cap + pos + t splits into a row part
// (b*H*cap + pos + t, from the GEMM row r = b*T + t; B*H*cap < 2^31 is checked on the host)
// and a column part (head*cap, the channel within the head), so an epilogue computes the
// row part once per token and the column part once per tile.
__device__ __forceinline__ int kv_row(const KvOut& kv, int r) {
  const int b = r / kv.T;
  return b * kv.H * kv.cap + kv.pos + (r - b * kv.T);
}
struct KvCol {
  uint8_t* codes;      // the code byte of column n at row part 0
  uint32_t* ab;        // the statistics word of column n's group at row part 0
};
__device__ __forceinline__ KvCol kv_col(const KvOut& kv, int n) {
  const bool isv = n >= 2 * kv.h;
  const int c = n - (isv ? 2 * kv.h : kv.h);
  const int head = c / kv.d, cin = c - head * kv.d;
  const int64_t hs = (int64_t)head * kv.cap;
  KvCol o;
  o.codes = (isv ? kv.v_codes : kv.k_codes) + hs * (kv.d / 2) + cin / 2;
  o.ab = (isv ? kv.v_ab : kv.k_ab) + hs * (kv.d / 64) + cin / 64;
  return o;
}
__device__ __forceinline__ uint32_t* kv_codes_at(const KvOut& kv, const KvCol& col, int row) {
  return reinterpret_cast<uint32_t*>(col.codes + (int64_t)row * (kv.d / 2));
}
__device__ __forceinline__ uint32_t* kv_ab_at(const KvOut& kv, const KvCol& col, int row) {
  return col.ab + (int64_t)row * (kv.d / 64);
}

struct EpiArgs {
  const uint16_t* bias;
  const uint16_t* residual;
  uint16_t* Y;
  float* partial;     // split-K: [splits][M][N] fp32, else null
  int epi;
  KvOut kv;
};


// Tensor maps (host): the driver's encoder, fetched once; a 2-D map over a row-major
// matrix of `outer` rows of `inner` elements, `row_bytes` apart.
cudaError_t get_encode();
cudaError_t make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                        uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                        uint32_t box_outer, CUtensorMapSwizzle swz);
// A 3-D map over [outer][mid][inner] elements (strides in bytes); boxes are one deep in the
// outer dimension.
cudaError_t make_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                        uint64_t mid, uint64_t outer, uint64_t mid_bytes, uint64_t outer_bytes,
                        uint32_t box_inner, uint32_t box_mid, CUtensorMapSwizzle swz);

// Weight-streaming GEMM for M <= 128 tokens: enqueues the main kernel on `st` (the caller
// launches the split-K reduce when p.splits > 1).  tmX is the tiled kernel's X map (64 k x
// tn tokens, 128B swizzle); the code and statistics maps of whole stages are built here.
cudaError_t launch_gemm_stream(const GemmPlan& p, const fg_q4mat& W, const CUtensorMap& tmX,
                               const EpiArgs& ea, cudaStream_t st);

// The CTA-pair kernel (p.kind == kGemmPair): enqueues the main kernel on `st` (the caller
// launches the split-K reduce when p.splits > 1); builds its own tensor maps.  w16 (nullable):
// the weight already restored to fp16 [K][N]; the kernel then loads its A slots by TMA instead
// of restoring the codes.  ws: the plan's workspace (with several token tiles it holds the
// unit counter at p.sched_off, zeroed here on `st` before the launch).
cudaError_t launch_gemm_pair(const GemmPlan& p, const fg_q4mat& W, const uint16_t* X,
                             const EpiArgs& ea, cudaStream_t st, const uint16_t* w16,
                             void* ws);

}  // namespace fg
