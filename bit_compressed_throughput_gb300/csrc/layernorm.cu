// Pre-LN LayerNorm of the OPT decoder layer (sm_103a): y = (x - mean)/sqrt(var + eps)
// * gamma + beta over rows of h fp16 values, fp32 statistics, population variance.
//
// One CTA per row.  The row is held in registers (h <= 16384: at most 8 16-byte chunks
// per thread at 256 threads), so the mean and the variance of the deviations are two
// reductions over registers and the row is read from HBM once: 2 bytes in, 2 bytes out
// per element.
#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxChunks = 8;   // 8 x 8 values x 256 threads = 16384

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();                    // red[] reuse across calls
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = (l < kThreads / 32) ? red[l] : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
  return t;                           // every lane of every warp holds the total
}

__global__ void __launch_bounds__(kThreads)
layernorm_kernel(const uint16_t* __restrict__ x, int h, const uint16_t* __restrict__ gamma,
                 const uint16_t* __restrict__ beta, float eps, uint16_t* __restrict__ y) {
  __shared__ float red[kThreads / 32];
  const int64_t row = blockIdx.x;
  const uint16_t* xr = x + row * h;
  const int nchunk = h / 8;          // 16-byte chunks in the row
  float v[kMaxChunks][8];
  float s = 0.0f;
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int ci = c * kThreads + threadIdx.x;
    if (ci < nchunk) {
      const uint4 u = ldg_nc_v4(xr + ci * 8);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack_h2(w[i]);
        v[c][2 * i] = f.x;
        v[c][2 * i + 1] = f.y;
        s += f.x + f.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[c][i] = 0.0f;
    }
  }
  const float mean = block_sum(s, red) / (float)h;
  float q = 0.0f;
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int ci = c * kThreads + threadIdx.x;
    if (ci < nchunk) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float dv = v[c][i] - mean;
        q += dv * dv;
      }
    }
  }
  const float var = block_sum(q, red) / (float)h;
  const float rstd = rsqrtf(var + eps);
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int ci = c * kThreads + threadIdx.x;
    if (ci < nchunk) {
      const uint4 gu = ldg_nc_v4(gamma + ci * 8), bu = ldg_nc_v4(beta + ci * 8);
      const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w}, bw[4] = {bu.x, bu.y, bu.z, bu.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 g2 = unpack_h2(gw[i]), b2 = unpack_h2(bw[i]);
        o[i] = pack_h2((v[c][2 * i] - mean) * rstd * g2.x + b2.x,
                       (v[c][2 * i + 1] - mean) * rstd * g2.y + b2.y);
      }
      reinterpret_cast<uint4*>(y + row * h)[ci] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

cudaError_t launch_layernorm(const uint16_t* x, int64_t rows, int32_t h, const uint16_t* g,
                             const uint16_t* b, float eps, uint16_t* y, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  layernorm_kernel<<<(unsigned)rows, kThreads, 0, st>>>(x, h, g, b, eps, y);
  return cudaGetLastError();
}

}  // namespace fg
