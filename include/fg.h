/*
 * fg.h -- C ABI of libfg, the GB300 (sm_103a) engine for one OPT-style decoder layer
 * over 4-bit group-compressed weights and KV cache, run over a block of sequences.
 *
 * The method (FlexGen):
 *  - Weights and the KV cache are stored as 4-bit codes, grouped 64 elements at a
 *    time -- along the output channel for weights, along the hidden dimension for
 *    K/V -- with the group minimum a and maximum b kept per group, and are restored
 *    to FP16 before any compute; INT4 is a storage format, not an INT4 matmul.
 *    [FlexGen review (jaehun.me), section "4-bit 압축은 정수 연산 가속과 같은가",
 *     restating paper §5; "论文阅读：FlexGen" (blog.gzher.com) §3.4]
 *  - One layer is applied to every GPU batch of a block (B = g*m sequences) before the
 *    next layer's weights are used; generation is a prefill over the prompt that builds
 *    the KV cache, then decode steps that add one token per sequence.
 *    [FlexGen paper explainer, "Compute Schedule" and Algorithm 1; Figure 2]
 *
 * Storage formats (the pages leave them open; these are this library's):
 *  - fp16 values are IEEE binary16 bit patterns (uint16_t).
 *  - codes: element 2i in the low nibble, element 2i+1 in the high nibble of byte i,
 *    along the grouped (contiguous) dimension.
 *  - group statistics: one uint32_t per group of 64, the fp16 bits of a in the low
 *    half and of b in the high half.
 *  - code q = rint((x - a) * 15 / (b - a)) in IEEE binary32 with one rounding per
 *    operation (subtract, multiply by 15, divide), round half to even, clamped to
 *    [0, 15]; a and b are the group min and max (-0 ordered below +0); a constant
 *    group (b - a == 0) stores all-zero codes.  Restoring: fp16(a + q * ((b - a) / 15)).
 *  - weight W[K][N] (K = input channel, N = output channel): codes [K][N/2] bytes,
 *    ab [K][N/64] words, row-major, groups of 64 consecutive n at fixed k.
 *  - KV cache of one layer: codes [B][H][cap][d/2] bytes and ab [B][H][cap][d/64]
 *    words for K and for V, groups of 64 consecutive hidden channels (a group never
 *    straddles two heads since d is 64 or 128).
 *
 * Conventions for every call:
 *  - Pointers marked "device" are device memory owned by the caller; the library
 *    never allocates, frees or keeps them.  Work is enqueued asynchronously on
 *    `stream` (a cudaStream_t passed as void*; NULL = the legacy default stream).
 *  - Arguments are validated on the host before any launch; a bad argument returns a
 *    negative fg_status and launches nothing.  Validation touches no CUDA API, so it
 *    can be exercised on a machine without a GPU.
 *  - Device pointers must be 16-byte aligned.
 *  - A failed launch returns FG_ERR_CUDA; fg_last_error() gives the CUDA message
 *    (thread-local).  FG_ERR_ARCH: the current device is not sm_103.
 *  - Every device wait inside a kernel is bounded; a wait that runs out sets a device
 *    error word that fg_check_device_error() reads (FG_ERR_TIMEOUT).
 */
#ifndef FG_H_
#define FG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FG_OK = 0,
  FG_ERR_ARG = -1,        /* null pointer, misaligned pointer, bad enum */
  FG_ERR_SHAPE = -2,      /* a dimension outside the supported set */
  FG_ERR_WORKSPACE = -3,  /* workspace smaller than the matching *_workspace_bytes() */
  FG_ERR_CUDA = -4,       /* a CUDA call or launch failed (see fg_last_error) */
  FG_ERR_ARCH = -5,       /* current device is not compute capability 10.3 */
  FG_ERR_CAPACITY = -6,   /* KV cache position out of range */
  FG_ERR_TIMEOUT = -7     /* a bounded device wait ran out (kernel result invalid) */
} fg_status;

/* A 4-bit group-compressed weight W[K][N]. codes: device [K][N/2]; ab: device [K][N/64]. */
typedef struct {
  const uint8_t* codes;
  const uint32_t* ab;
  int64_t K;
  int64_t N;
} fg_q4mat;

/* The INT4 KV cache of one layer (device buffers, layout above). */
typedef struct {
  uint8_t* k_codes;
  uint8_t* v_codes;
  uint32_t* k_ab;
  uint32_t* v_ab;
  int32_t B;    /* sequences */
  int32_t cap;  /* positions per sequence, a multiple of 16 (whole 16-position tiles) */
  int32_t h;    /* hidden size */
  int32_t H;    /* heads; d = h / H must be 64 or 128 */
} fg_kvcache;

typedef struct {
  int32_t h;      /* hidden size, multiple of 256, at most 16384 */
  int32_t H;      /* heads */
  int32_t d;      /* head dim, 64 or 128, h == H*d */
  int32_t f;      /* FFN width, multiple of 256; 0 = attention block without the MLP */
  float ln_eps;   /* LayerNorm epsilon */
} fg_dims;

/* One pre-LN decoder layer: h1 = x + Attn(LN1(x)) Wo + bo; y = h1 + ReLU(LN2(h1) W1 + b1) W2 + b2
 * with [Q|K|V] = LN1(x) Wqkv + bqkv. Weights K-major (W[in][out]); wqkv is [h][3h] with
 * columns q | k | v. All vectors fp16, device; biases may be NULL (zero).
 * w1/w2/b1/b2/ln2_* unused when f == 0. */
typedef struct {
  fg_q4mat wqkv, wo, w1, w2;
  const uint16_t *bqkv, *bo, *b1, *b2;
  const uint16_t *ln1_g, *ln1_b, *ln2_g, *ln2_b;
} fg_layer;

/* Epilogues of fg_dequant_gemm_q4. */
enum { FG_EPI_NONE = 0, FG_EPI_RELU = 1, FG_EPI_RESIDUAL = 2 };

/* ---------------------------------------------------------------------- quantise */

/* Group-wise 4-bit quantisation of fp16 x[rows][cols] (groups of 64 along cols), as
 * defined above.  x, codes [rows][cols/2], ab [rows][cols/64]: device.
 * cols % 64 == 0, rows >= 0 (rows == 0 is a no-op).  Bit-exact with the definition.
 * [FlexGen review (jaehun.me), "4-bit 압축은 정수 연산 가속과 같은가"] */
int fg_quantize_g64(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* codes,
                    uint32_t* ab, void* stream);

/* Restore fp16 y[rows][cols] = fp16(a + q * ((b - a) / 15)) (binary32, one rounding per
 * operation).  The standalone restore; the GEMM and attention restore in registers.
 * [same passage: values are restored to FP16 before compute] */
int fg_dequant_g64(const uint8_t* codes, const uint32_t* ab, int64_t rows, int64_t cols,
                   uint16_t* y, void* stream);

/* ---------------------------------------------------------------------- GEMM */

/* Y[M][N] = epi(X[M][K] * W^ + bias) with W^ the fp16 restoration of W, fp32 accumulate.
 * epi: FG_EPI_NONE; FG_EPI_RELU (max(.,0)); FG_EPI_RESIDUAL (+ residual[M][N]).
 * X, bias (nullable, [N]), residual (FG_EPI_RESIDUAL only), Y: device fp16, row-major,
 * leading dimensions K (X) and N (Y, residual).  K % 16 == 0, N % 256 == 0 (one output tile
 * of group statistics is one 16-byte row), M >= 0.
 * Y may alias residual.  ws: device scratch of at least fg_gemm_workspace_bytes(M,K,N)
 * bytes (split-K partial sums when M is small; with M > 256 a 4-byte unit counter that the
 * call zeroes on `stream` before its kernel); NULL allowed when that is 0.  Two calls in
 * flight at once on different streams need workspaces of their own.
 * [FlexGen review (jaehun.me), "4-bit 압축은 정수 연산 가속과 같은가": restore to FP16
 *  before compute, not an INT4 matmul; FlexGen paper explainer, "Cost Model and Policy
 *  Search": the four h x h and two h x h2 weight matrices of a layer] */
int fg_dequant_gemm_q4(const uint16_t* X, int64_t M, const fg_q4mat* W, const uint16_t* bias,
                       int epilogue, const uint16_t* residual, uint16_t* Y, void* ws,
                       size_t ws_bytes, void* stream);
/* Scratch bytes fg_dequant_gemm_q4 needs for an M x K by K x N product (split-K fp32
 * partials when M is small, and 256 bytes for the unit counter of the many-token plans;
 * 0 when neither applies).  Host computation only; the pages have no counterpart (their
 * GEMMs run in PyTorch). */
size_t fg_gemm_workspace_bytes(int64_t M, int64_t K, int64_t N);

/* The QKV projection with the KV quantise-and-append in its epilogue:
 *   Y[M][3h] = X[M][K] * W^[K][3h] + bias   (columns: Q, then K, then V),
 * and for every row r = b*T + t (sequence b of the cache, t < T) the K and V columns of
 * row r, rounded to fp16 as Y holds them, are quantised in groups of 64 (the same codes
 * and (a, b) as fg_kv_append_q4 gives for those rows) and written at position pos + t.
 * One launch (two when M is small enough for a split-K sum): the fp16 K/V are not read
 * back from memory.  h = kv->h, a multiple of 128; W->N == 3h; M == kv->B * T; T >= 1;
 * pos + T <= kv->cap; kv->B * kv->H * kv->cap < 2^31.  Y is still written in full (prefill attention reads the fp16 K/V).
 * ws as for fg_dequant_gemm_q4.  Errors as fg_dequant_gemm_q4, plus FG_ERR_CAPACITY.
 * [FlexGen review (jaehun.me), "4-bit 압축은 정수 연산 가속과 같은가": K/V grouped 64
 *  along the hidden dimension] */
int fg_dequant_gemm_q4_kv(const uint16_t* X, int64_t M, const fg_q4mat* W, const uint16_t* bias,
                          uint16_t* Y, const fg_kvcache* kv, int32_t T, int32_t pos, void* ws,
                          size_t ws_bytes, void* stream);

/* A GEMM whose output rows also pass through the pre-LN LayerNorm of the next sub-layer:
 *   Y = epilogue(X * W^ + bias)   (as fg_dequant_gemm_q4),
 *   Y_ln[r] = (Y[r] - mean) / sqrt(var + ln_eps) * ln_gamma + ln_beta   over the N values of
 *   row r of Y as stored (fp16), fp32 mean and population variance (as fg_layernorm).
 * When the plan splits K (few rows) the split-K reduce sums the partials, applies the
 * epilogue, stores Y and normalises the row in the same kernel (one CTA per row); otherwise
 * the GEMM is followed by the LayerNorm kernel.  N <= 16384; Y_ln must not alias Y (it
 * may alias nothing the GEMM reads).  ws as for fg_dequant_gemm_q4.  Errors as
 * fg_dequant_gemm_q4.  [OPT decoder layer as a pre-LN block; FlexGen paper explainer,
 *  "Computation Delegation": the layer's GEMMs and attention on the GPU] */
int fg_dequant_gemm_q4_ln(const uint16_t* X, int64_t M, const fg_q4mat* W, const uint16_t* bias,
                          int epilogue, const uint16_t* residual, uint16_t* Y,
                          const uint16_t* ln_gamma, const uint16_t* ln_beta, float ln_eps,
                          uint16_t* Y_ln, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------- KV cache */

/* Quantise new keys and values into the cache at positions pos .. pos+T-1 of every
 * sequence.  k_new, v_new: device fp16, row (b, t) at (b*T + t) * row_stride elements,
 * h contiguous values per row (row_stride >= h, a multiple of 8; lets K/V be read in
 * place from a [rows][3h] QKV buffer).  T >= 0; pos >= 0; pos + T <= cap.
 * Codes and statistics are bit-exact with fg_quantize_g64 on the same rows.
 * [FlexGen review (jaehun.me), "4-bit 압축은 정수 연산 가속과 같은가": KV grouped
 *  along the hidden dimension; FlexGen paper explainer, Figure 2: each decode step
 *  extends the cache] */
int fg_kv_append_q4(const uint16_t* k_new, const uint16_t* v_new, int64_t row_stride,
                    int32_t T, int32_t pos, const fg_kvcache* kv, void* stream);

/* ---------------------------------------------------------------------- attention */

/* Decode attention of one new token per sequence over cache positions 0 .. len-1:
 * out[b][hd*d + j] = sum_t softmax_t(scale * q_b,hd . K^_b,hd,t) V^_b,hd,t,j with K^, V^
 * the fp16 restorations of the cached codes.  q: device fp16, row b at b*q_stride
 * elements; out: device fp16 [B][h].  1 <= len <= cap.  ws: device scratch of at least
 * fg_decode_attn_workspace_bytes(kv, len) bytes (split-sequence partials).
 * [FlexGen paper explainer, "Computation Delegation": decoding attention is I/O bound
 *  over the KV cache] */
int fg_decode_attn_q4kv(const uint16_t* q, int64_t q_stride, const fg_kvcache* kv, int32_t len,
                        float scale, uint16_t* out, void* ws, size_t ws_bytes, void* stream);
/* Scratch bytes fg_decode_attn_q4kv needs (split-sequence partials, planned for up to 192
 * SMs; 0 when no split is planned).  Host computation only; no counterpart on the pages. */
size_t fg_decode_attn_workspace_bytes(const fg_kvcache* kv, int32_t len);

/* Decode attention exactly as fg_decode_attn_q4kv, for callers that cannot allocate
 * device memory -- code that must not call cudaMalloc (a region that forbids allocation,
 * an external allocator that owns all device memory, a host runtime that can only pass
 * existing buffers through) and so cannot supply the split-sequence workspace.  Its
 * scratch is a fixed array of FG_DECODE_ATTN_STATIC_SCRATCH_BYTES in device global
 * memory defined by the library itself (held on every GPU that loads the library until
 * the process exits); the call allocates nothing.  The caller still passes q, the cache
 * and out.  A call whose split scratch (fg_decode_attn_workspace_bytes) would exceed the
 * array returns FG_ERR_WORKSPACE without launching, and fg_last_error() says so.
 * The first call on a device looks up the array's device address for that device; make
 * that first call before any stream capture.  All calls share the array: calls that
 * overlap on the GPU race on it.  No part of it needs to start at zero; each call writes
 * every byte it reads.  The paper has no counterpart of this entry point. */
#define FG_DECODE_ATTN_STATIC_SCRATCH_BYTES (4u << 20)
int fg_decode_attn_q4kv_static(const uint16_t* q, int64_t q_stride, const fg_kvcache* kv,
                               int32_t len, float scale, uint16_t* out, void* stream);

/* Top-K sparse decode attention over the same cache: the scores of all positions
 * 0 .. len-1 come from the 4-bit K and the softmax runs over all of them, but only the k
 * positions with the highest scores contribute their values:
 *   out[b][hd*d + j] = sum_{t in top-k(b,hd)} p_t V^_b,hd,t,j   (no renormalisation)
 * with equal scores at the k-th place going to the lower position.  1 <= k <= len <= cap,
 * d in {64, 128}, (len + k) * 4 + 1024 bytes <= 227 KB.  q, out as fg_decode_attn_q4kv.  sel
 * (nullable): device int32 [B][H][k] receiving the selected positions in increasing
 * position order.  ws: device scratch of at least fg_decode_attn_topk_workspace_bytes(kv,
 * len) bytes (the scores).
 * [论文阅读：FlexGen, §3.4: optional sparse attention that loads only the top 10% of the value
 *  cache; FlexGen paper explainer, §3.3: Top-K sparse attention cuts I/O volume] */
int fg_decode_attn_q4kv_topk(const uint16_t* q, int64_t q_stride, const fg_kvcache* kv,
                             int32_t len, int32_t k, float scale, uint16_t* out, int32_t* sel,
                             void* ws, size_t ws_bytes, void* stream);
size_t fg_decode_attn_topk_workspace_bytes(const fg_kvcache* kv, int32_t len);

/* Causal prefill attention over fp16 Q/K/V read from a QKV buffer qkv[nseq*s][3h]
 * (columns q | k | v, head hd at hd*d): out[nseq*s][h] fp16, position i attends over
 * positions 0..i of its own sequence, scores scaled by `scale`.  d in {64, 128}, scale > 0,
 * nseq <= 65535, nseq * s < 2^31; qkv and out device pointers, 16-byte aligned (FG_ERR_ARG
 * otherwise).  nseq == 0 or s == 0 is a no-op.
 * [FlexGen paper explainer, Figure 2: the prefill step processes all prompt tokens] */
int fg_prefill_attn(const uint16_t* qkv, int32_t nseq, int32_t s, int32_t H, int32_t d,
                    float scale, uint16_t* out, void* stream);

/* ---------------------------------------------------------------------- LayerNorm */

/* y[rows][h] = (x - mean) / sqrt(var + eps) * gamma + beta, fp32 statistics (population
 * variance), fp16 in and out.  x, gamma, beta, y: device fp16 (gamma, beta [h]); h % 64
 * == 0, h <= 16384, eps > 0; rows == 0 is a no-op.  The pages name no normalisation: this
 * is the pre-LN of the OPT decoder layer the workloads specify (LN1 before attention, LN2
 * before the MLP); the pages have no counterpart of the call itself. */
int fg_layernorm(const uint16_t* x, int64_t rows, int32_t h, const uint16_t* gamma,
                 const uint16_t* beta, float eps, uint16_t* y, void* stream);

/* ---------------------------------------------------------------------- layer */

/* Prefill of one layer over a block of m GPU batches of g sequences each, prompt length s:
 * x, y: device fp16 [m][g][s][h] (y may alias x).  GPU batch k is processed in full
 * (M = g*s rows per GEMM) before batch k+1; its K/V are quantised into `kv` positions
 * 0..s-1 of sequences k*g .. k*g+g-1.  kv->B == g*m, s <= kv->cap.  When g*s > 128 the
 * call first restores the layer's four weight matrices to fp16 in `ws` (once for the m GPU
 * batches) and its GEMMs read those instead of restoring the codes tile by tile; the results
 * are those of the 4-bit weights either way.
 * ws: device scratch of at least fg_layer_workspace_bytes(dims, g, m, s) bytes.
 * [FlexGen paper explainer, Algorithm 1 (a layer over every GPU batch of the block);
 *  Figure 2 (prefill builds the cache); FlexGen review, "4-bit 압축은 정수 연산 가속과
 *  같은가": weights restored to FP16 before compute] */
int fg_layer_prefill(const fg_dims* dims, const fg_layer* layer, fg_kvcache* kv,
                     const uint16_t* x, uint16_t* y, int32_t g, int32_t m, int32_t s,
                     void* ws, size_t ws_bytes, void* stream);

/* One decode step of one layer for the whole block: x, y: device fp16 [m][g][h] = [B][h]
 * (y may alias x), one launch per operation with M = B rows so each weight is read once
 * per step.  pos is the cache length before the step: the new K/V are appended at pos
 * and attention runs over positions 0..pos.  pos + 1 <= kv->cap.
 * [FlexGen paper explainer, Algorithm 1 and Figure 2] */
int fg_layer_decode(const fg_dims* dims, const fg_layer* layer, fg_kvcache* kv,
                    const uint16_t* x, uint16_t* y, int32_t g, int32_t m, int32_t pos,
                    void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes for fg_layer_prefill with prompts up to s_max and for fg_layer_decode
 * with caches up to s_max positions (the larger of the two uses): per GPU batch of g
 * sequences the LayerNorm output, the [g*s][3h] QKV, the attention output, h1 and the
 * [g*s][f] FFN activation, plus GEMM split-K partials, the layer's weights restored to fp16
 * for a prefill of more than 128 rows (2*(4h^2 + 2hf) bytes) and, for decode over the whole
 * block of g*m sequences, the split-sequence attention partials.  Returns 0 for invalid dims
 * or g, m, s_max <= 0.  A pure host computation (no CUDA call).
 * [FlexGen paper explainer, "Compute Schedule": a layer runs over every GPU batch of the
 *  block, so the scratch is sized by g, m and the sequence length, not by the stack] */
size_t fg_workspace_bytes(const fg_dims* dims, int32_t g, int32_t m, int32_t s_max);
/* The same value as fg_workspace_bytes, under the name of the layer calls it sizes. */
size_t fg_layer_workspace_bytes(const fg_dims* dims, int32_t g, int32_t m, int32_t s_max);

/* ---------------------------------------------------------------------- runtime */

const char* fg_status_string(int status);
const char* fg_last_error(void);
/* Synchronise `stream`, read and clear the device error word: FG_OK or FG_ERR_TIMEOUT. */
int fg_check_device_error(void* stream);

/* Per-kernel timing with CUDA events recorded around every launch on its stream.
 * kind: one of FG_K_* below.  fg_prof_query synchronises the recorded events and
 * returns the launch count, total milliseconds and the algorithmic work of those
 * launches (bytes for HBM-bound kinds, flops for the GEMM and prefill attention). */
enum {
  FG_K_QUANT = 0, FG_K_DEQUANT = 1, FG_K_GEMM = 2, FG_K_GEMM_REDUCE = 3,
  FG_K_KV_APPEND = 4, FG_K_DECODE_ATTN = 5, FG_K_DECODE_COMBINE = 6,
  FG_K_PREFILL_ATTN = 7, FG_K_LAYERNORM = 8,
  FG_K_GEMM_STREAM = 9,   /* the weight-streaming GEMM (M <= 128): work counted in bytes */
  FG_K_DECODE_ATTN_TOPK = 10,   /* both kernels of the top-K attention: bytes */
  FG_K_GEMM_PAIR = 11,   /* the tiled GEMM on CTA pairs (many tokens): flops */
  FG_K_GEMM_PAIR_F16W = 12,   /* the CTA-pair GEMM on weights restored to fp16 (layer
                                 prefill): flops */
  FG_K_COUNT = 13
};
int fg_prof_enable(int on);
int fg_prof_reset(void);
int fg_prof_query(int kind, int64_t* launches, double* ms, double* work);
const char* fg_kernel_name(int kind);

#ifdef __cplusplus
}
#endif
#endif /* FG_H_ */
