// Pre-LN LayerNorm of the OPT decoder layer (sm_103a): y = (x - mean)/sqrt(var + eps)
// * gamma + beta over rows of h fp16 values, fp32 statistics, population variance.
//
// WPR warps per row (1 for h <= 2048, 2 for h = 4096, up to 8 for h = 16384), 8 warps per
// CTA: each lane holds at most 8 16-byte chunks of its row in registers, so the mean and the variance of
// the deviations are reductions over registers (warp shuffles, then WPR partials through
// shared memory) and the row is read from HBM once: 2 bytes in, 2 bytes out per element.
// A warp per row keeps short rows (decode) and long batches (prefill) free of block-wide
// synchronisation on the row's critical path.
#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxChunks = 8;   // 16-byte chunks per lane

template <int WPR>
__global__ void __launch_bounds__(kThreads, 3)
layernorm_kernel(const uint16_t* __restrict__ x, int64_t rows, int h,
                 const uint16_t* __restrict__ gamma, const uint16_t* __restrict__ beta,
                 float eps, uint16_t* __restrict__ y) {
  __shared__ float red[2][kWarps];
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (kWarps / WPR) + warp / WPR;
  const bool live = row < rows;
  const int sub = warp % WPR;
  const int nchunk = h / 8;                 // 16-byte chunks in the row
  const int stride = 32 * WPR;              // chunk stride between a lane's chunks
  const int c0 = sub * 32 + lane;
  const uint16_t* xr = x + (live ? row : 0) * h;
  uint4 v[kMaxChunks];
  float s = 0.0f;
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int ci = c0 + c * stride;
    v[c] = (live && ci < nchunk) ? ldg_nc_v4(xr + ci * 8) : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = unpack_h2(w[i]);
      s += f.x + f.y;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  if (WPR > 1) {
    if (lane == 0) red[0][warp] = s;
    __syncthreads();
    s = 0.0f;
#pragma unroll
    for (int i = 0; i < WPR; ++i) s += red[0][(warp / WPR) * WPR + i];
  }
  const float mean = s / (float)h;
  float q = 0.0f;
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int ci = c0 + c * stride;
    if (ci < nchunk) {
      const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack_h2(w[i]);
        const float d0 = f.x - mean, d1 = f.y - mean;
        q += d0 * d0 + d1 * d1;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xFFFFFFFFu, q, o);
  if (WPR > 1) {
    if (lane == 0) red[1][warp] = q;
    __syncthreads();
    q = 0.0f;
#pragma unroll
    for (int i = 0; i < WPR; ++i) q += red[1][(warp / WPR) * WPR + i];
  }
  const float var = q / (float)h;
  const float rstd = rsqrtf(var + eps);
  if (!live) return;
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int ci = c0 + c * stride;
    if (ci < nchunk) {
      const uint4 gu = ldg_nc_v4(gamma + ci * 8), bu = ldg_nc_v4(beta + ci * 8);
      const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
      const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w}, bw[4] = {bu.x, bu.y, bu.z, bu.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack_h2(w[i]), g2 = unpack_h2(gw[i]), b2 = unpack_h2(bw[i]);
        o[i] = pack_h2((f.x - mean) * rstd * g2.x + b2.x, (f.y - mean) * rstd * g2.y + b2.y);
      }
      reinterpret_cast<uint4*>(y + row * h)[ci] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

cudaError_t launch_layernorm(const uint16_t* x, int64_t rows, int32_t h, const uint16_t* g,
                             const uint16_t* b, float eps, uint16_t* y, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  // warps per row: the fewest that keep a lane's share of the row within kMaxChunks
  const int nchunk = h / 8;
  int wpr = 1;
  while (nchunk > 32 * kMaxChunks * wpr) wpr *= 2;     // h <= 16384: at most 8
  const int64_t rows_per_cta = kWarps / wpr;
  const unsigned grid = (unsigned)((rows + rows_per_cta - 1) / rows_per_cta);
  if (wpr == 1)
    return launch_pdl(layernorm_kernel<1>, dim3(grid), dim3(kThreads), 0, st, x, rows, h, g, b, eps, y);
  else if (wpr == 2)
    return launch_pdl(layernorm_kernel<2>, dim3(grid), dim3(kThreads), 0, st, x, rows, h, g, b, eps, y);
  else if (wpr == 4)
    return launch_pdl(layernorm_kernel<4>, dim3(grid), dim3(kThreads), 0, st, x, rows, h, g, b, eps, y);
  else
    return launch_pdl(layernorm_kernel<8>, dim3(grid), dim3(kThreads), 0, st, x, rows, h, g, b, eps, y);
}

}  // namespace fg
