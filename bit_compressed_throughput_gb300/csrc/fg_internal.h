// Host-side declarations shared by the translation units of libfg.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>
#include <utility>

#include "../../include/fg.h"

namespace fg {

// Largest SM count the workspace queries plan for (GB300 has 152).
constexpr int kMaxSms = 192;

// Launchers: enqueue one kernel on `st`; return cudaGetLastError().
cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* codes,
                            uint32_t* ab, cudaStream_t st);
cudaError_t launch_dequant(const uint8_t* codes, const uint32_t* ab, int64_t rows, int64_t cols,
                           uint16_t* y, cudaStream_t st);
// The same values with each run of 8 channels stored as 0,4,1,5,2,6,3,7: the A-tile order of
// the CTA-pair GEMM, whose fp16-weight mode loads these instead of restoring.
cudaError_t launch_dequant_pairperm(const uint8_t* codes, const uint32_t* ab, int64_t rows,
                                    int64_t cols, uint16_t* y, cudaStream_t st);
cudaError_t launch_kv_append(const uint16_t* k_new, const uint16_t* v_new, int64_t row_stride,
                             int32_t T, int32_t pos, const fg_kvcache& kv, cudaStream_t st);
cudaError_t launch_layernorm(const uint16_t* x, int64_t rows, int32_t h, const uint16_t* g,
                             const uint16_t* b, float eps, uint16_t* y, cudaStream_t st);
cudaError_t launch_prefill_attn(const uint16_t* qkv, int32_t nseq, int32_t s, int32_t H,
                                int32_t d, float scale, uint16_t* out, int nsm, cudaStream_t st);

// Launch with programmatic stream serialisation (see pdl_wait in fg_common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Message returned by fg_last_error() on this thread.
void set_last_error(const std::string& msg);

// Host validation shared by the entry points (FG_OK or a negative fg_status; no CUDA call
// except in check_device).  check_device: the current device is sm_103; *sms_out receives
// its SM count capped at kMaxSms.  check_decode_attn: the arguments of a decode-attention
// call; *nothing_to_do is set when the cache holds no sequences.
int check_device(int* sms_out);
int check_kv(const fg_kvcache* kv);
int check_decode_attn(const uint16_t* q, int64_t q_stride, const fg_kvcache* kv, int32_t len,
                      float scale, const uint16_t* out, bool* nothing_to_do);
// Decode attention with per-kernel event timing (when profiling is on); ws holds at least
// decode_attn_ws_bytes(kv, len, sms) bytes.  Returns FG_OK or FG_ERR_CUDA.
int run_decode_attn(const uint16_t* q, int64_t q_stride, const fg_kvcache& kv, int len,
                    float scale, uint16_t* out, void* ws, int sms, cudaStream_t st);

// Decode attention: number of sequence splits used for (kv, len); workspace bytes.
int decode_attn_splits(const fg_kvcache& kv, int32_t len, int num_sms);
size_t decode_attn_ws_bytes(const fg_kvcache& kv, int32_t len, int num_sms);
// Launches the split kernel and, when splits > 1, the combine kernel (recording
// `mid_event`, when given, between the two).  `kernels_out` receives 1 or 2.
cudaError_t launch_decode_attn(const uint16_t* q, int64_t q_stride, const fg_kvcache& kv,
                               int32_t len, float scale, uint16_t* out, void* ws,
                               int num_sms, cudaStream_t st, int* kernels_out,
                               cudaEvent_t mid_event);

// Scores-only decode attention (top-K): the dense kernel's K stream and scores, each score
// as an order key into keys [B*H][len], each work item's softmax state (m, l) into ml
// [B*H][splits]; *splits_out receives the split count.
cudaError_t launch_decode_attn_scores(const uint16_t* q, int64_t q_stride, const fg_kvcache& kv,
                                      int32_t len, float scale, uint32_t* keys, float2* ml,
                                      int nsm, cudaStream_t st, int* splits_out);
// Top-K sparse decode attention: workspace bytes; launches the score and the
// select-and-attend kernels.
size_t decode_attn_topk_ws_bytes(const fg_kvcache& kv, int32_t len);
cudaError_t launch_decode_attn_topk(const uint16_t* q, int64_t q_stride, const fg_kvcache& kv,
                                    int32_t len, int32_t k, float scale, uint16_t* out,
                                    int32_t* sel, void* ws, int nsm, cudaStream_t st);

// Dequant-fused GEMM plan: tn tokens x 128 channels per tile, split-K factor and
// workspace.  kind 0: the tiled kernel (restored weights in shared memory); kind 1: the
// weight-streaming kernel for M <= 128 (restored weights in tensor memory); kind 2: the
// tiled product on CTA pairs (256 channels x 256 tokens per 2-CTA tile) for M >= 256 with
// little token padding.
constexpr int kGemmTiled = 0;
constexpr int kGemmStream = 1;
constexpr int kGemmPair = 2;
constexpr int kStreamStage = 4;          // k-blocks of 64 per code stage of the streaming kernel
constexpr int kPairStageKb = 4;          // k-blocks per code stage of the CTA-pair GEMM (decode)
struct GemmPlan {
  int kind;
  int64_t M, N, K;
  int tn;                  // tokens per tile: a multiple of 16 in [16, 256]
  int tiles_t, tiles_c, kblocks, splits, kb_per_split;
  int64_t units;   // (split, tile) work units
  int grid;        // persistent CTAs: min(units, SMs)
  size_t ws_bytes;
  size_t sched_off;  // kind 2 with tiles_t >= 2: offset in the workspace of the unit counter
};
// K/V append of the QKV projection: columns [h, 2h) of Y are K and [2h, 3h) are V; row
// r = b*T + t of the GEMM is position pos + t of sequence b.  Each 64-channel group of a
// K or V row is quantised from its fp16 output values (the values Y holds) and written to
// the head-major cache: codes at ((b*H + head)*cap + pos + t)*(d/2) + c/2, the (a, b) word
// at that slot times d/64 plus c/64 (c = the channel within the head).  k_codes == null:
// no append.
struct KvOut {
  uint8_t* k_codes;
  uint8_t* v_codes;
  uint32_t* k_ab;
  uint32_t* v_ab;
  int h, H, d, cap, T, pos;
};

// allow_pair = false keeps to the one-CTA kernels (the K/V-append epilogue exists there only).
GemmPlan gemm_plan(int64_t M, int64_t K, int64_t N, int num_sms, bool allow_pair = true);
// Workspace bytes that cover every plan of an M x K x N product on up to kMaxSms SMs.
size_t gemm_ws_bytes(int64_t M, int64_t K, int64_t N);
// LayerNorm of the GEMM's output rows, fused into the split-K reduce: y = LN(Y) with
// (gamma, beta, eps), N <= 16384.
struct LnOut {
  const uint16_t* gamma;
  const uint16_t* beta;
  float eps;
  uint16_t* y;
};
// kv: K/V append in the epilogue (null or k_codes == null: none).  ln: LayerNorm in the
// split-K reduce (only for a split plan; null: none).  w16: W already restored to fp16
// [K][N] (only the CTA-pair plan uses it; null: restore in the GEMM).
cudaError_t launch_gemm(const GemmPlan& p, const uint16_t* X, const fg_q4mat& W,
                        const uint16_t* bias, int epi, const uint16_t* residual, uint16_t* Y,
                        void* ws, cudaStream_t st, cudaEvent_t mid_event,
                        const KvOut* kv = nullptr, const LnOut* ln = nullptr,
                        const uint16_t* w16 = nullptr);
// Device error words of the bounded waits (GEMM, decode attention): read-and-clear.
cudaError_t gemm_read_error(unsigned int* out);
cudaError_t gemm_stream_read_error(unsigned int* out);
cudaError_t gemm_pair_read_error(unsigned int* out);
cudaError_t prefill_read_error(unsigned int* out);
cudaError_t attn_read_error(unsigned int* out);

// Algorithmic work of one launch (bytes for memory-bound kernels, flops for the GEMM and
// prefill attention): 4-bit storage costs 0.5 byte per element plus one (a, b) fp16 pair
// per group of 64, i.e. 0.5625 byte.
inline double work_gemm(int64_t M, int64_t N, int64_t K) { return 2.0 * M * N * K; }
// Weight-streaming GEMM (few tokens): bound by the 4-bit weight stream, so its work is
// bytes: the weights at 0.5625 byte per element plus the fp16 activations in and out.
inline double work_gemm_stream(int64_t M, int64_t N, int64_t K) {
  return 0.5625 * K * N + 2.0 * M * K + 2.0 * M * N;
}
inline double work_gemm_reduce(int64_t M, int64_t N, int splits) {
  return (double)splits * M * N * 4.0 + 2.0 * M * N;
}
inline double work_quantize(double elems) { return elems * (2.0 + 0.5625); }
inline double work_dequant(double elems) { return elems * (0.5625 + 2.0); }
inline double work_decode_attn(int64_t B, int64_t len, int64_t h) {
  return 2.0 * B * len * h * 0.5625 + 4.0 * B * h;
}
// Top-K attention: the whole 4-bit K, the 4-bit V of k positions, the fp32 scores written
// and read back, q in and out.
inline double work_decode_attn_topk(int64_t B, int64_t H, int64_t len, int64_t k, int64_t h) {
  return B * len * h * 0.5625 + B * k * h * 0.5625 + 8.0 * B * H * len + 4.0 * B * h;
}
inline double work_prefill_attn(int64_t nseq, int64_t s, int64_t h) {
  return 2.0 * nseq * h * s * (s + 1);
}
inline double work_layernorm(int64_t rows, int64_t h) { return 4.0 * rows * h; }

}  // namespace fg
