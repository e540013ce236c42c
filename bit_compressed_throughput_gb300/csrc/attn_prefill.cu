// Causal prefill attention over fp16 Q/K/V (sm_103a).
//
// The prefill step processes every prompt token at once and builds the KV cache
// [FlexGen paper explainer, "Problem Formulation", Figure 2].  Prefill attends over the
// fp16 K/V the projection just produced (the cache keeps the 4-bit copy for decoding).
//
// Flash-style: a CTA owns 128 query rows of one (sequence, head), 8 warps x 16 rows, so each
// K/V tile of 64 keys serves 128 rows; the tiles stream through a double-buffered cp.async
// ring; S = Q K^T and O += P V run on mma.sync m16n8k16 (fp16 in, fp32 accumulate) with an
// online base-2 softmax.  Q fragments are reloaded from shared memory for every tile rather
// than held in registers, so a thread stays within 128 registers and two CTAs (16 warps)
// share an SM.  A warp skips the key tiles that lie wholly above its rows (causal), and the
// CTAs of the last query tiles, which see the most keys, are scheduled first.  Q, K, V are
// read in place from the [rows][3h] QKV buffer.
#include <math.h>

#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {
namespace {

constexpr int kRows = 128;     // query rows per CTA
constexpr int kKeys = 64;      // keys per tile
constexpr int kWarpsA = kRows / 16;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^x on the special-function unit (inputs <= 0 here; results below 2^-126 flush to zero,
// far below the fp16 P fed to the P V product).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
struct Smem {
  static constexpr int LD = D + 8;                  // padded row (halves)
  static constexpr int QTILE = kRows * LD;          // halves of the Q tile
  static constexpr int TILE = kKeys * LD;           // halves of a K or V tile
  static constexpr int BYTES = (QTILE + 4 * TILE) * 2;   // Q, K[2], V[2]
};

template <int D>
__global__ void __launch_bounds__(kWarpsA * 32, 2)
prefill_attn_kernel(const uint16_t* __restrict__ qkv, int s, int H, float scale_log2,
                    uint16_t* __restrict__ out) {
  constexpr int LD = Smem<D>::LD;
  constexpr int TILE = Smem<D>::TILE;
  extern __shared__ __align__(16) uint16_t sm[];
  pdl_launch_dependents();
  pdl_wait();
  uint16_t* sQ = sm;
  uint16_t* sK = sm + Smem<D>::QTILE;  // 2 tiles
  uint16_t* sV = sK + 2 * TILE;        // 2 tiles

  // heaviest query tiles first
  const int qt = gridDim.x - 1 - blockIdx.x, hd = blockIdx.y, seq = blockIdx.z;
  const int h = H * D;
  const int64_t row0 = (int64_t)seq * s;       // first row of this sequence
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int q0 = qt * kRows;

  // ---- async loads: a tile is `rows` rows x D halves = rows * D/8 16-byte chunks
  auto load_tile = [&](uint16_t* dst, int col, int r0, int rows) {
    constexpr int CPR = D / 8;
    for (int c = threadIdx.x; c < rows * CPR; c += kWarpsA * 32) {
      const int r = c / CPR, cc = c % CPR;
      const int pos = r0 + r;
      const bool valid = pos < s;
      const uint16_t* src = qkv + (row0 + (valid ? pos : 0)) * (3 * h) + col + cc * 8;
      cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(dst + r * LD + cc * 8)), src,
                 valid);
    }
  };
  load_tile(sQ, hd * D, q0, kRows);
  load_tile(sK, h + hd * D, 0, kKeys);
  load_tile(sV, 2 * h + hd * D, 0, kKeys);
  cp_commit();

  // causal: key tiles up to the one holding the CTA's last row
  const int nkt = min((q0 + kRows - 1) / kKeys + 1, (s + kKeys - 1) / kKeys);
  const int wrow_last = q0 + warp * 16 + 15;              // this warp's last row
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[i][c] = 0.0f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};

  for (int kt = 0; kt < nkt; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < nkt) {
      load_tile(sK + (buf ^ 1) * TILE, h + hd * D, (kt + 1) * kKeys, kKeys);
      load_tile(sV + (buf ^ 1) * TILE, 2 * h + hd * D, (kt + 1) * kKeys, kKeys);
    }
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    // a tile whose first key lies past this warp's last row is fully masked for it
    if (kt * kKeys > wrow_last) {
      __syncthreads();   // the buffer is refilled by the next iteration's loads
      continue;
    }
    const uint16_t* kb = sK + buf * TILE;
    const uint16_t* vb = sV + buf * TILE;

    // ---- S = Q K^T for 16 rows x 64 keys (Q fragments from shared memory)
    float sc[kKeys / 8][4];
#pragma unroll
    for (int nb = 0; nb < kKeys / 8; ++nb)
#pragma unroll
      for (int c = 0; c < 4; ++c) sc[nb][c] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t qf[4];
      {
        const int r = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int c = ks * 16 + 8 * (lane >> 4);
        ldsm_x4(static_cast<uint32_t>(__cvta_generic_to_shared(sQ + r * LD + c)), qf[0], qf[1],
                qf[2], qf[3]);
      }
#pragma unroll
      for (int nb = 0; nb < kKeys / 8; nb += 2) {
        const int i = lane >> 3;
        const int key = nb * 8 + (lane & 7) + 8 * (i >> 1);
        const int c = ks * 16 + 8 * (i & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(static_cast<uint32_t>(__cvta_generic_to_shared(kb + key * LD + c)), b0, b1, b2,
                b3);
        mma16816(sc[nb], qf[0], qf[1], qf[2], qf[3], b0, b1);
        mma16816(sc[nb + 1], qf[0], qf[1], qf[2], qf[3], b2, b3);
      }
    }
    // ---- mask (causal and sequence tail), online softmax in base 2
    const int qrow[2] = {q0 + warp * 16 + gid, q0 + warp * 16 + gid + 8};
    float mx[2] = {-INFINITY, -INFINITY};
    // only a tile reaching past this warp's first row, or past the sequence, needs the mask
    if (kt * kKeys + kKeys - 1 > q0 + warp * 16 || kt * kKeys + kKeys > s) {
#pragma unroll
      for (int nb = 0; nb < kKeys / 8; ++nb) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int key = kt * kKeys + nb * 8 + 2 * tig + (c & 1);
          const int r = c >> 1;
          float v = sc[nb][c] * scale_log2;
          if (key > qrow[r] || key >= s) v = -INFINITY;
          sc[nb][c] = v;
          mx[r] = fmaxf(mx[r], v);
        }
      }
    } else {
#pragma unroll
      for (int nb = 0; nb < kKeys / 8; ++nb) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float v = sc[nb][c] * scale_log2;
          sc[nb][c] = v;
          mx[c >> 1] = fmaxf(mx[c >> 1], v);
        }
      }
    }
    float corr[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xFFFFFFFFu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xFFFFFFFFu, mx[r], 2));
      const float m_new = fmaxf(m_run[r], mx[r]);
      corr[r] = (m_run[r] == -INFINITY) ? 0.0f : ex2(m_run[r] - m_new);
      m_run[r] = m_new;
    }
    float ls[2] = {0.0f, 0.0f};
#pragma unroll
    for (int nb = 0; nb < kKeys / 8; ++nb) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int r = c >> 1;
        const float p = (m_run[r] == -INFINITY) ? 0.0f : ex2(sc[nb][c] - m_run[r]);
        sc[nb][c] = p;
        ls[r] += p;
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      ls[r] += __shfl_xor_sync(0xFFFFFFFFu, ls[r], 1);
      ls[r] += __shfl_xor_sync(0xFFFFFFFFu, ls[r], 2);
      l_run[r] = l_run[r] * corr[r] + ls[r];
    }
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o[i][0] *= corr[0]; o[i][1] *= corr[0];
      o[i][2] *= corr[1]; o[i][3] *= corr[1];
    }
    // ---- O += P V
#pragma unroll
    for (int kk = 0; kk < kKeys / 16; ++kk) {
      const uint32_t a0 = pack_h2(sc[2 * kk][0], sc[2 * kk][1]);
      const uint32_t a1 = pack_h2(sc[2 * kk][2], sc[2 * kk][3]);
      const uint32_t a2 = pack_h2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      const uint32_t a3 = pack_h2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
      for (int nb = 0; nb < D / 8; nb += 2) {
        const int i = lane >> 3;
        const int key = kk * 16 + (lane & 7) + 8 * (i & 1);
        const int c = nb * 8 + 8 * (i >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(static_cast<uint32_t>(__cvta_generic_to_shared(vb + key * LD + c)), b0, b1, b2,
                  b3);
        mma16816(o[nb], a0, a1, a2, a3, b0, b1);
        mma16816(o[nb + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();     // the buffer is refilled by the next iteration's loads
  }

  // ---- normalise and store
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int qr = q0 + warp * 16 + gid + 8 * r;
    if (qr >= s) continue;
    const float inv = (l_run[r] > 0.0f) ? 1.0f / l_run[r] : 0.0f;
    uint16_t* op = out + (row0 + qr) * h + hd * D;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      *reinterpret_cast<uint32_t*>(op + i * 8 + 2 * tig) =
          pack_h2(o[i][2 * r] * inv, o[i][2 * r + 1] * inv);
    }
  }
}

}  // namespace

cudaError_t launch_prefill_attn(const uint16_t* qkv, int32_t nseq, int32_t s, int32_t H,
                                int32_t d, float scale, uint16_t* out, cudaStream_t st) {
  if (nseq == 0 || s == 0) return cudaSuccess;
  dim3 grid((unsigned)((s + kRows - 1) / kRows), (unsigned)H, (unsigned)nseq);
  const float sl2 = scale * 1.4426950408889634f;
  if (d == 128) {
    static cudaError_t attr = cudaFuncSetAttribute(
        prefill_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<128>::BYTES);
    if (attr != cudaSuccess) return attr;
    return launch_pdl(prefill_attn_kernel<128>, grid, dim3(kWarpsA * 32), Smem<128>::BYTES, st,
                      qkv, s, H, sl2, out);
  } else {
    static cudaError_t attr = cudaFuncSetAttribute(
        prefill_attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<64>::BYTES);
    if (attr != cudaSuccess) return attr;
    return launch_pdl(prefill_attn_kernel<64>, grid, dim3(kWarpsA * 32), Smem<64>::BYTES, st, qkv,
                      s, H, sl2, out);
  }
}

}  // namespace fg
