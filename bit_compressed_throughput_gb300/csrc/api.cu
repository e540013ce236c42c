// C ABI of libfg: argument validation, workspace planning, per-kernel event timing and
// the composition of one decoder layer's prefill and decode step out of the kernels.
//
// Call order inside a layer follows the block schedule: a layer runs over every GPU batch
// of the block before the caller moves to the next layer, and decode runs the whole
// block as one M = B launch per operation so each weight is read once per step
// [FlexGen paper explainer, "Compute Schedule", Algorithm 1; FlexGen review (jaehun.me),
// "Block은 여러 GPU 배치에 걸친 가중치 재사용 단위다"].
#include <math.h>

#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/fg.h"
#include "fg_internal.h"

namespace fg {
namespace {

thread_local std::string t_last_error;

// Upper bound on SMs used when sizing workspaces, so workspace sizes need no device query.


int set_cuda_error(cudaError_t e) {
  t_last_error = cudaGetErrorString(e);
  return FG_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- device facts
struct DevInfo {
  bool init = false;
  bool ok = false;
  int sms = 0;
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

}  // namespace

int check_device(int* sms_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e);
  if (dev < 0 || dev >= 64) return FG_ERR_ARCH;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& di = g_dev[dev];
  if (!di.init) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return set_cuda_error(e);
    di.ok = (major == 10 && minor == 3);
    di.sms = std::min(sms, kMaxSms);
    di.init = true;
  }
  if (!di.ok) {
    t_last_error = "libfg is built for sm_103a (GB300); the current device is not compute 10.3";
    return FG_ERR_ARCH;
  }
  if (sms_out) *sms_out = di.sms;
  return FG_OK;
}

namespace {

// ---------------------------------------------------------------- profiling
struct ProfRec {
  int kind;
  cudaEvent_t a, b;
  double work;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_pending;
std::vector<cudaEvent_t> g_pool;
int64_t g_launches[FG_K_COUNT];
double g_ms[FG_K_COUNT];
double g_work[FG_K_COUNT];

cudaEvent_t pool_get_locked() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// A timed span on `st`: the constructor records the start event, close() ends one kernel
// at an event the launcher recorded between two kernels, stop() records the end event.
struct Span {
  cudaStream_t st;
  bool on = false;
  cudaEvent_t cur = nullptr;
  explicit Span(cudaStream_t s) : st(s) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    on = g_prof_on;
    if (on) {
      cur = pool_get_locked();
      cudaEventRecord(cur, st);
    }
  }
  cudaEvent_t mid_event() {
    if (!on) return nullptr;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    return pool_get_locked();
  }
  void close(int kind, double work, cudaEvent_t end_recorded) {
    if (!on) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_pending.push_back({kind, cur, end_recorded, work});
    cur = end_recorded;
  }
  void stop(int kind, double work) {
    if (!on) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    cudaEvent_t e = pool_get_locked();
    cudaEventRecord(e, st);
    g_pending.push_back({kind, cur, e, work});
    cur = nullptr;
  }
};

void prof_drain_locked() {
  std::vector<cudaEvent_t> release;
  for (auto& r : g_pending) {
    cudaEventSynchronize(r.b);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, r.a, r.b);
    g_launches[r.kind] += 1;
    g_ms[r.kind] += ms;
    g_work[r.kind] += r.work;
    release.push_back(r.a);
    release.push_back(r.b);
  }
  g_pending.clear();
  std::sort(release.begin(), release.end());
  release.erase(std::unique(release.begin(), release.end()), release.end());
  for (auto e : release) g_pool.push_back(e);
}

// ---------------------------------------------------------------- validation helpers
int check_q4mat(const fg_q4mat* W) {
  if (!W || !W->codes || !W->ab) return FG_ERR_ARG;
  if (!aligned16(W->codes) || !aligned16(W->ab)) return FG_ERR_ARG;
  // N % 256: the group statistics of one 256-column tile are one 16-byte TMA row
  if (W->K <= 0 || W->K % 16 != 0 || W->N <= 0 || W->N % 256 != 0) return FG_ERR_SHAPE;
  if (W->K > (1ll << 31) - 1 || W->N > (1ll << 31) - 1) return FG_ERR_SHAPE;
  return FG_OK;
}

}  // namespace

int check_kv(const fg_kvcache* kv) {
  if (!kv || !kv->k_codes || !kv->v_codes || !kv->k_ab || !kv->v_ab) return FG_ERR_ARG;
  if (!aligned16(kv->k_codes) || !aligned16(kv->v_codes) || !aligned16(kv->k_ab) ||
      !aligned16(kv->v_ab))
    return FG_ERR_ARG;
  // cap % 16: decode attention streams whole 16-position tiles of a head's region
  if (kv->B < 0 || kv->cap <= 0 || kv->cap % 16 != 0 || kv->h <= 0 || kv->H <= 0 ||
      kv->h % 64 != 0 || kv->h % kv->H != 0)
    return FG_ERR_SHAPE;
  const int d = kv->h / kv->H;
  if (d != 64 && d != 128) return FG_ERR_SHAPE;
  return FG_OK;
}

int check_decode_attn(const uint16_t* q, int64_t q_stride, const fg_kvcache* kv, int32_t len,
                      float scale, const uint16_t* out, bool* nothing_to_do) {
  *nothing_to_do = false;
  int rc = check_kv(kv);
  if (rc) return rc;
  if (len <= 0) return FG_ERR_SHAPE;
  if (len > kv->cap) return FG_ERR_CAPACITY;
  if (q_stride < kv->h || q_stride % 8 != 0) return FG_ERR_SHAPE;
  if (!(scale > 0.0f) || !isfinite(scale)) return FG_ERR_ARG;
  if (kv->B == 0) {
    *nothing_to_do = true;
    return FG_OK;
  }
  if (!q || !out || !aligned16(q) || !aligned16(out)) return FG_ERR_ARG;
  return FG_OK;
}

namespace {

int check_dims(const fg_dims* dm) {
  if (!dm) return FG_ERR_ARG;
  if (dm->h <= 0 || dm->h % 256 != 0 || dm->h > 16384 || dm->H <= 0 || dm->h != dm->H * dm->d ||
      (dm->d != 64 && dm->d != 128) || dm->f < 0 || dm->f % 256 != 0 || !(dm->ln_eps > 0.0f))
    return FG_ERR_SHAPE;
  return FG_OK;
}

size_t round_up(size_t x) { return (x + 255) & ~size_t(255); }

// Sub-cache of sequences [b0, b0 + nb).
fg_kvcache kv_slice(const fg_kvcache& kv, int b0, int nb) {
  const int d = kv.h / kv.H;
  const int64_t slots = (int64_t)b0 * kv.H * kv.cap;
  fg_kvcache s = kv;
  s.k_codes = kv.k_codes + slots * (d / 2);
  s.v_codes = kv.v_codes + slots * (d / 2);
  s.k_ab = kv.k_ab + slots * (d / 64);
  s.v_ab = kv.v_ab + slots * (d / 64);
  s.B = nb;
  return s;
}

// The K/V append of rows b*T + t (positions pos + t) into `kv`.
KvOut kv_out(const fg_kvcache& kv, int T, int pos) {
  KvOut o;
  o.k_codes = kv.k_codes;
  o.v_codes = kv.v_codes;
  o.k_ab = reinterpret_cast<uint32_t*>(kv.k_ab);
  o.v_ab = reinterpret_cast<uint32_t*>(kv.v_ab);
  o.h = kv.h;
  o.H = kv.H;
  o.d = kv.h / kv.H;
  o.cap = kv.cap;
  o.T = T;
  o.pos = pos;
  return o;
}

// ---------------------------------------------------------------- timed launches
// kv: the QKV projection's K/V append in the GEMM epilogue (null: none).
// Profiler kind of a plan's main kernel.
int gemm_kind(const GemmPlan& p, const uint16_t* w16) {
  if (p.kind == kGemmStream) return FG_K_GEMM_STREAM;
  if (p.kind == kGemmPair) return w16 ? FG_K_GEMM_PAIR_F16W : FG_K_GEMM_PAIR;
  return FG_K_GEMM;
}

// w16 (nullable): W restored to fp16 [K][N], used by a CTA-pair plan instead of the codes.
int run_gemm(const uint16_t* X, int64_t M, const fg_q4mat& W, const uint16_t* bias, int epi,
             const uint16_t* residual, uint16_t* Y, void* ws, int sms, cudaStream_t st,
             const KvOut* kv = nullptr, const uint16_t* w16 = nullptr) {
  const GemmPlan p = gemm_plan(M, W.K, W.N, sms, kv == nullptr);
  if (p.kind != kGemmPair) w16 = nullptr;
  Span sp(st);
  cudaEvent_t mid = (p.splits > 1) ? sp.mid_event() : nullptr;
  cudaError_t e = launch_gemm(p, X, W, bias, epi, residual, Y, ws, st, mid, kv, nullptr, w16);
  if (e != cudaSuccess) return set_cuda_error(e);
  const bool stream = (p.kind == kGemmStream);
  const int kind = gemm_kind(p, w16);
  // the streaming kernel's work is bytes: with the append, also the 4-bit K/V written
  const double w = stream ? work_gemm_stream(M, W.N, W.K) + (kv ? 2.0 * M * kv->h * 0.5625 : 0.0)
                          : work_gemm(M, W.N, W.K);
  if (p.splits > 1 && mid) {
    sp.close(kind, w, mid);
    sp.stop(FG_K_GEMM_REDUCE, work_gemm_reduce(M, W.N, p.splits));
  } else {
    sp.stop(kind, w);
  }
  return FG_OK;
}

// W restored to fp16 [K][N] for the CTA-pair GEMM's fp16-weight mode: the values of
// fg_dequant_g64, each run of 8 channels in the GEMM's A-tile order (0,4,1,5,2,6,3,7).
int run_restore(const fg_q4mat& W, uint16_t* y, cudaStream_t st) {
  Span sp(st);
  cudaError_t e = launch_dequant_pairperm(W.codes, W.ab, W.K, W.N, y, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  sp.stop(FG_K_DEQUANT, work_dequant((double)W.K * W.N));
  return FG_OK;
}

int run_layernorm(const uint16_t* x, int64_t rows, int h, const uint16_t* g, const uint16_t* b,
                  float eps, uint16_t* y, cudaStream_t st) {
  Span sp(st);
  cudaError_t e = launch_layernorm(x, rows, h, g, b, eps, y, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  sp.stop(FG_K_LAYERNORM, work_layernorm(rows, h));
  return FG_OK;
}

// GEMM whose output rows also go through LayerNorm (y_ln = LN(Y)): with a split-K plan
// the reduce kernel does both (one launch after the GEMM); otherwise the GEMM, then the
// LayerNorm kernel.
int run_gemm_ln(const uint16_t* X, int64_t M, const fg_q4mat& W, const uint16_t* bias, int epi,
                const uint16_t* residual, uint16_t* Y, const uint16_t* g, const uint16_t* b,
                float eps, uint16_t* y_ln, void* ws, int sms, cudaStream_t st,
                const uint16_t* w16 = nullptr) {
  const GemmPlan p = gemm_plan(M, W.K, W.N, sms);
  if (p.kind != kGemmPair) w16 = nullptr;
  if (p.splits == 1) {
    int rc = run_gemm(X, M, W, bias, epi, residual, Y, ws, sms, st, nullptr, w16);
    if (rc) return rc;
    return run_layernorm(Y, M, (int)W.N, g, b, eps, y_ln, st);
  }
  Span sp(st);
  cudaEvent_t mid = sp.mid_event();
  const LnOut ln{g, b, eps, y_ln};
  cudaError_t e = launch_gemm(p, X, W, bias, epi, residual, Y, ws, st, mid, nullptr, &ln, w16);
  if (e != cudaSuccess) return set_cuda_error(e);
  const bool stream = (p.kind == kGemmStream);
  const int kind = gemm_kind(p, w16);
  const double w = stream ? work_gemm_stream(M, W.N, W.K) : work_gemm(M, W.N, W.K);
  if (mid) {
    sp.close(kind, w, mid);
    // the reduce reads the partials and writes Y (its work), then writes LN(Y)
    sp.stop(FG_K_GEMM_REDUCE, work_gemm_reduce(M, W.N, p.splits) + 2.0 * M * W.N);
  } else {
    sp.stop(kind, w);
  }
  return FG_OK;
}

int run_kv_append(const uint16_t* k, const uint16_t* v, int64_t stride, int T, int pos,
                  const fg_kvcache& kv, cudaStream_t st) {
  Span sp(st);
  cudaError_t e = launch_kv_append(k, v, stride, T, pos, kv, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  sp.stop(FG_K_KV_APPEND, work_quantize(2.0 * kv.B * T * kv.h));
  return FG_OK;
}

}  // namespace

int run_decode_attn(const uint16_t* q, int64_t q_stride, const fg_kvcache& kv, int len,
                    float scale, uint16_t* out, void* ws, int sms, cudaStream_t st) {
  Span sp(st);
  const int splits = decode_attn_splits(kv, len, sms);
  cudaEvent_t mid = (splits > 1) ? sp.mid_event() : nullptr;
  int nk = 0;
  cudaError_t e = launch_decode_attn(q, q_stride, kv, len, scale, out, ws, sms, st, &nk, mid);
  if (e != cudaSuccess) return set_cuda_error(e);
  const double w = work_decode_attn(kv.B, len, kv.h);
  if (nk == 2 && mid) {
    sp.close(FG_K_DECODE_ATTN, w, mid);
    const int d = kv.h / kv.H;
    sp.stop(FG_K_DECODE_COMBINE, (double)kv.B * kv.H * splits * (d + 2) * 4.0 + 2.0 * kv.B * kv.h);
  } else {
    sp.stop(FG_K_DECODE_ATTN, w);
  }
  return FG_OK;
}

namespace {

int run_prefill_attn(const uint16_t* qkv, int nseq, int s, int H, int d, float scale,
                     uint16_t* out, int sms, cudaStream_t st) {
  Span sp(st);
  cudaError_t e = launch_prefill_attn(qkv, nseq, s, H, d, scale, out, sms, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  sp.stop(FG_K_PREFILL_ATTN, work_prefill_attn(nseq, s, (int64_t)H * d));
  return FG_OK;
}

// ---------------------------------------------------------------- layer workspace
struct LayerWs {
  size_t ln, qkv, att, h1, mid, gemm, attn, w16, total;
};

// Prefill restores a layer's weights to fp16 once per call when its GEMMs run on CTA pairs
// (M > 128): the restore is then done once for all m GPU batches, and the GEMMs load their A
// tiles by TMA instead of restoring every tile once per token tile (M / 256 times).
bool prefill_restores(int64_t M) { return M > 128; }

LayerWs layer_ws(const fg_dims& dm, int64_t M, const fg_kvcache* kv_for_decode, int len) {
  LayerWs w{};
  const int64_t h = dm.h, f = dm.f;
  w.ln = round_up((size_t)M * h * 2);
  w.qkv = round_up((size_t)M * 3 * h * 2);
  w.att = round_up((size_t)M * h * 2);
  w.h1 = round_up((size_t)M * h * 2);
  w.mid = round_up((size_t)M * f * 2);
  size_t g = gemm_ws_bytes(M, h, 3 * h);
  g = std::max(g, gemm_ws_bytes(M, h, h));
  if (f > 0) {
    g = std::max(g, gemm_ws_bytes(M, h, f));
    g = std::max(g, gemm_ws_bytes(M, f, h));
  }
  w.gemm = round_up(g);
  w.attn = kv_for_decode ? round_up(decode_attn_ws_bytes(*kv_for_decode, len, kMaxSms)) : 0;
  // the four restored matrices (QKV h x 3h, O h x h, FC1 h x f, FC2 f x h)
  w.w16 = (!kv_for_decode && prefill_restores(M))
              ? round_up((size_t)(4 * h * h) * 2) + round_up((size_t)(2 * h * f) * 2)
              : 0;
  w.total = w.ln + w.qkv + w.att + w.h1 + w.mid + w.gemm + w.attn + w.w16;
  return w;
}

}  // namespace

void set_last_error(const std::string& msg) { t_last_error = msg; }

}  // namespace fg

using namespace fg;

extern "C" {

const char* fg_status_string(int s) {
  switch (s) {
    case FG_OK: return "ok";
    case FG_ERR_ARG: return "invalid argument (null or misaligned pointer, bad enum)";
    case FG_ERR_SHAPE: return "unsupported shape";
    case FG_ERR_WORKSPACE: return "workspace too small";
    case FG_ERR_CUDA: return "CUDA error";
    case FG_ERR_ARCH: return "device is not sm_103 (GB300)";
    case FG_ERR_CAPACITY: return "KV cache position out of range";
    case FG_ERR_TIMEOUT: return "a bounded device wait ran out";
    default: return "unknown status";
  }
}

const char* fg_last_error(void) { return t_last_error.c_str(); }

int fg_check_device_error(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return set_cuda_error(e);
  unsigned int flag = 0, sflag = 0, aflag = 0;
  e = gemm_read_error(&flag);
  if (e != cudaSuccess) return set_cuda_error(e);
  e = gemm_stream_read_error(&sflag);
  if (e != cudaSuccess) return set_cuda_error(e);
  flag |= sflag;
  e = gemm_pair_read_error(&sflag);
  if (e != cudaSuccess) return set_cuda_error(e);
  flag |= sflag;
  e = prefill_read_error(&sflag);
  if (e != cudaSuccess) return set_cuda_error(e);
  flag |= sflag;
  e = attn_read_error(&aflag);
  if (e != cudaSuccess) return set_cuda_error(e);
  if (flag || aflag) {
    t_last_error = "bounded device wait timed out (GEMM flag " + std::to_string(flag) +
                   ", decode attention flag " + std::to_string(aflag) + ")";
    return FG_ERR_TIMEOUT;
  }
  return FG_OK;
}

int fg_quantize_g64(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* codes, uint32_t* ab,
                    void* stream) {
  if (rows < 0 || cols <= 0 || cols % 64 != 0) return FG_ERR_SHAPE;
  if (rows == 0) return FG_OK;
  if (!x || !codes || !ab) return FG_ERR_ARG;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(ab)) return FG_ERR_ARG;
  int rc = check_device(nullptr);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Span sp(st);
  cudaError_t e = launch_quantize(x, rows, cols, codes, ab, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  sp.stop(FG_K_QUANT, work_quantize((double)rows * cols));
  return FG_OK;
}

int fg_dequant_g64(const uint8_t* codes, const uint32_t* ab, int64_t rows, int64_t cols,
                   uint16_t* y, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 64 != 0) return FG_ERR_SHAPE;
  if (rows == 0) return FG_OK;
  if (!y || !codes || !ab) return FG_ERR_ARG;
  if (!aligned16(y) || !aligned16(codes) || !aligned16(ab)) return FG_ERR_ARG;
  int rc = check_device(nullptr);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Span sp(st);
  cudaError_t e = launch_dequant(codes, ab, rows, cols, y, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  sp.stop(FG_K_DEQUANT, (double)rows * cols * (2.0 + 0.5625));
  return FG_OK;
}

size_t fg_gemm_workspace_bytes(int64_t M, int64_t K, int64_t N) {
  return gemm_ws_bytes(M, K, N);
}

int fg_dequant_gemm_q4(const uint16_t* X, int64_t M, const fg_q4mat* W, const uint16_t* bias,
                       int epilogue, const uint16_t* residual, uint16_t* Y, void* ws,
                       size_t ws_bytes, void* stream) {
  int rc = check_q4mat(W);
  if (rc) return rc;
  if (M < 0 || M > (1ll << 31) - 1) return FG_ERR_SHAPE;
  if (epilogue < FG_EPI_NONE || epilogue > FG_EPI_RESIDUAL) return FG_ERR_ARG;
  if (M == 0) return FG_OK;
  if (!X || !Y || (epilogue == FG_EPI_RESIDUAL && !residual)) return FG_ERR_ARG;
  if (!aligned16(X) || !aligned16(Y) || (bias && !aligned16(bias)) ||
      (residual && !aligned16(residual)))
    return FG_ERR_ARG;
  const size_t need = fg_gemm_workspace_bytes(M, W->K, W->N);
  if (ws_bytes < need || (need > 0 && (!ws || !aligned16(ws)))) return FG_ERR_WORKSPACE;
  int sms = 0;
  rc = check_device(&sms);
  if (rc) return rc;
  return run_gemm(X, M, *W, bias, epilogue, residual, Y, ws, sms,
                  static_cast<cudaStream_t>(stream));
}

int fg_dequant_gemm_q4_kv(const uint16_t* X, int64_t M, const fg_q4mat* W, const uint16_t* bias,
                          uint16_t* Y, const fg_kvcache* kv, int32_t T, int32_t pos, void* ws,
                          size_t ws_bytes, void* stream) {
  int rc = check_q4mat(W);
  if (rc) return rc;
  if ((rc = check_kv(kv))) return rc;
  // Y = [Q | K | V]: three h-wide column blocks, each a whole number of 128-channel tiles
  if (W->N != 3 * (int64_t)kv->h || kv->h % 128 != 0) return FG_ERR_SHAPE;
  if (T <= 0 || pos < 0 || M != (int64_t)kv->B * T || M > (1ll << 31) - 1) return FG_ERR_SHAPE;
  // the epilogues address cache slots (b*H + head)*cap + pos + t in 32 bits
  if ((int64_t)kv->B * kv->H * kv->cap > (1ll << 31) - 1) return FG_ERR_SHAPE;
  if ((int64_t)pos + T > kv->cap) return FG_ERR_CAPACITY;
  if (M == 0) return FG_OK;
  if (!X || !Y || !aligned16(X) || !aligned16(Y) || (bias && !aligned16(bias))) return FG_ERR_ARG;
  const size_t need = fg_gemm_workspace_bytes(M, W->K, W->N);
  if (ws_bytes < need || (need > 0 && (!ws || !aligned16(ws)))) return FG_ERR_WORKSPACE;
  int sms = 0;
  if ((rc = check_device(&sms))) return rc;
  const KvOut ko = kv_out(*kv, T, pos);
  return run_gemm(X, M, *W, bias, FG_EPI_NONE, nullptr, Y, ws, sms,
                  static_cast<cudaStream_t>(stream), &ko);
}

int fg_dequant_gemm_q4_ln(const uint16_t* X, int64_t M, const fg_q4mat* W, const uint16_t* bias,
                          int epilogue, const uint16_t* residual, uint16_t* Y,
                          const uint16_t* ln_gamma, const uint16_t* ln_beta, float ln_eps,
                          uint16_t* Y_ln, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_q4mat(W);
  if (rc) return rc;
  if (M < 0 || M > (1ll << 31) - 1 || W->N > 16384) return FG_ERR_SHAPE;
  if (epilogue < FG_EPI_NONE || epilogue > FG_EPI_RESIDUAL || !(ln_eps > 0.0f)) return FG_ERR_ARG;
  if (M == 0) return FG_OK;
  if (!X || !Y || !Y_ln || !ln_gamma || !ln_beta || Y_ln == Y ||
      (epilogue == FG_EPI_RESIDUAL && !residual))
    return FG_ERR_ARG;
  if (!aligned16(X) || !aligned16(Y) || !aligned16(Y_ln) || !aligned16(ln_gamma) ||
      !aligned16(ln_beta) || (bias && !aligned16(bias)) || (residual && !aligned16(residual)))
    return FG_ERR_ARG;
  const size_t need = fg_gemm_workspace_bytes(M, W->K, W->N);
  if (ws_bytes < need || (need > 0 && (!ws || !aligned16(ws)))) return FG_ERR_WORKSPACE;
  int sms = 0;
  if ((rc = check_device(&sms))) return rc;
  return run_gemm_ln(X, M, *W, bias, epilogue, residual, Y, ln_gamma, ln_beta, ln_eps, Y_ln, ws,
                     sms, static_cast<cudaStream_t>(stream));
}

int fg_kv_append_q4(const uint16_t* k_new, const uint16_t* v_new, int64_t row_stride, int32_t T,
                    int32_t pos, const fg_kvcache* kv, void* stream) {
  int rc = check_kv(kv);
  if (rc) return rc;
  if (T < 0 || pos < 0) return FG_ERR_SHAPE;
  if ((int64_t)pos + T > kv->cap) return FG_ERR_CAPACITY;
  if (row_stride < kv->h || row_stride % 8 != 0) return FG_ERR_SHAPE;
  if (T == 0 || kv->B == 0) return FG_OK;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return FG_ERR_ARG;
  rc = check_device(nullptr);
  if (rc) return rc;
  return run_kv_append(k_new, v_new, row_stride, T, pos, *kv, static_cast<cudaStream_t>(stream));
}

size_t fg_decode_attn_workspace_bytes(const fg_kvcache* kv, int32_t len) {
  if (!kv || check_kv(kv) != FG_OK || len <= 0) return 0;
  return decode_attn_ws_bytes(*kv, len, kMaxSms);
}

int fg_decode_attn_q4kv(const uint16_t* q, int64_t q_stride, const fg_kvcache* kv, int32_t len,
                        float scale, uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  bool noop = false;
  int rc = check_decode_attn(q, q_stride, kv, len, scale, out, &noop);
  if (rc || noop) return rc;
  const size_t need = fg_decode_attn_workspace_bytes(kv, len);
  if (ws_bytes < need || (need > 0 && (!ws || !aligned16(ws)))) return FG_ERR_WORKSPACE;
  int sms = 0;
  rc = check_device(&sms);
  if (rc) return rc;
  return run_decode_attn(q, q_stride, *kv, len, scale, out, ws, sms,
                         static_cast<cudaStream_t>(stream));
}

size_t fg_decode_attn_topk_workspace_bytes(const fg_kvcache* kv, int32_t len) {
  if (!kv || check_kv(kv) != FG_OK || len <= 0) return 0;
  return decode_attn_topk_ws_bytes(*kv, len);
}

int fg_decode_attn_q4kv_topk(const uint16_t* q, int64_t q_stride, const fg_kvcache* kv,
                             int32_t len, int32_t k, float scale, uint16_t* out, int32_t* sel,
                             void* ws, size_t ws_bytes, void* stream) {
  int rc = check_kv(kv);
  if (rc) return rc;
  if (len <= 0 || k <= 0 || k > len) return FG_ERR_SHAPE;
  if (len > kv->cap) return FG_ERR_CAPACITY;
  if ((int64_t)(len + k) * 4 + 1024 > 227 * 1024) return FG_ERR_SHAPE;
  if (q_stride < kv->h || q_stride % 8 != 0) return FG_ERR_SHAPE;
  if (!(scale > 0.0f) || !isfinite(scale)) return FG_ERR_ARG;
  if (kv->B == 0) return FG_OK;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return FG_ERR_ARG;
  const size_t need = fg_decode_attn_topk_workspace_bytes(kv, len);
  if (ws_bytes < need || !ws || !aligned16(ws)) return FG_ERR_WORKSPACE;
  int sms = 0;
  rc = check_device(&sms);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Span sp(st);
  cudaError_t e = launch_decode_attn_topk(q, q_stride, *kv, len, k, scale, out, sel, ws, sms, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  sp.stop(FG_K_DECODE_ATTN_TOPK,
          work_decode_attn_topk(kv->B, kv->H, len, k, kv->h));
  return FG_OK;
}

int fg_prefill_attn(const uint16_t* qkv, int32_t nseq, int32_t s, int32_t H, int32_t d,
                    float scale, uint16_t* out, void* stream) {
  if (nseq < 0 || s < 0 || H <= 0 || (d != 64 && d != 128) || nseq > 65535) return FG_ERR_SHAPE;
  if (!(scale > 0.0f) || !isfinite(scale)) return FG_ERR_ARG;
  if (nseq == 0 || s == 0) return FG_OK;
  if (!qkv || !out || !aligned16(qkv) || !aligned16(out)) return FG_ERR_ARG;
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  return run_prefill_attn(qkv, nseq, s, H, d, scale, out, sms, static_cast<cudaStream_t>(stream));
}

int fg_layernorm(const uint16_t* x, int64_t rows, int32_t h, const uint16_t* gamma,
                 const uint16_t* beta, float eps, uint16_t* y, void* stream) {
  if (rows < 0 || h <= 0 || h % 64 != 0 || h > 16384) return FG_ERR_SHAPE;
  if (!(eps > 0.0f)) return FG_ERR_ARG;
  if (rows == 0) return FG_OK;
  if (!x || !y || !gamma || !beta) return FG_ERR_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(gamma) || !aligned16(beta)) return FG_ERR_ARG;
  int rc = check_device(nullptr);
  if (rc) return rc;
  return run_layernorm(x, rows, h, gamma, beta, eps, y, static_cast<cudaStream_t>(stream));
}

static int check_layer(const fg_dims* dm, const fg_layer* L) {
  if (!L) return FG_ERR_ARG;
  int rc;
  if ((rc = check_q4mat(&L->wqkv)) || (rc = check_q4mat(&L->wo))) return rc;
  if (L->wqkv.K != dm->h || L->wqkv.N != 3 * dm->h || L->wo.K != dm->h || L->wo.N != dm->h)
    return FG_ERR_SHAPE;
  if (!L->ln1_g || !L->ln1_b || !aligned16(L->ln1_g) || !aligned16(L->ln1_b)) return FG_ERR_ARG;
  if ((L->bqkv && !aligned16(L->bqkv)) || (L->bo && !aligned16(L->bo))) return FG_ERR_ARG;
  if (dm->f > 0) {
    if ((rc = check_q4mat(&L->w1)) || (rc = check_q4mat(&L->w2))) return rc;
    if (L->w1.K != dm->h || L->w1.N != dm->f || L->w2.K != dm->f || L->w2.N != dm->h)
      return FG_ERR_SHAPE;
    if (!L->ln2_g || !L->ln2_b || !aligned16(L->ln2_g) || !aligned16(L->ln2_b)) return FG_ERR_ARG;
    if ((L->b1 && !aligned16(L->b1)) || (L->b2 && !aligned16(L->b2))) return FG_ERR_ARG;
  }
  return FG_OK;
}

size_t fg_workspace_bytes(const fg_dims* dm, int32_t g, int32_t m, int32_t s_max) {
  if (!dm || check_dims(dm) != FG_OK || g <= 0 || m <= 0 || s_max <= 0) return 0;
  const int64_t Mp = (int64_t)g * s_max;       // prefill rows per GPU batch
  const int64_t Md = (int64_t)g * m;           // decode rows (whole block)
  fg_kvcache kv{};
  kv.B = g * m; kv.cap = s_max; kv.h = dm->h; kv.H = dm->H;
  const LayerWs a = layer_ws(*dm, Mp, nullptr, 0);
  size_t best = a.total;
  // decode splits (and so its workspace) depend on the cache length: take the maximum
  for (int len = 1; len <= s_max; len = (len < 64) ? len + 1 : len + 16)
    best = std::max(best, layer_ws(*dm, Md, &kv, len).total);
  best = std::max(best, layer_ws(*dm, Md, &kv, s_max).total);
  return best;
}

size_t fg_layer_workspace_bytes(const fg_dims* dm, int32_t g, int32_t m, int32_t s_max) {
  return fg_workspace_bytes(dm, g, m, s_max);
}

int fg_layer_prefill(const fg_dims* dm, const fg_layer* L, fg_kvcache* kv, const uint16_t* x,
                     uint16_t* y, int32_t g, int32_t m, int32_t s, void* ws, size_t ws_bytes,
                     void* stream) {
  int rc;
  if ((rc = check_dims(dm)) || (rc = check_layer(dm, L)) || (rc = check_kv(kv))) return rc;
  if (g <= 0 || m <= 0 || s <= 0 || g > 65535) return FG_ERR_SHAPE;
  if (kv->B != g * m || kv->h != dm->h || kv->H != dm->H) return FG_ERR_SHAPE;
  if (s > kv->cap) return FG_ERR_CAPACITY;
  if (!x || !y || !aligned16(x) || !aligned16(y)) return FG_ERR_ARG;
  const int64_t M = (int64_t)g * s;
  const LayerWs w = layer_ws(*dm, M, nullptr, 0);
  if (!ws || !aligned16(ws) || ws_bytes < w.total) return FG_ERR_WORKSPACE;
  int sms = 0;
  if ((rc = check_device(&sms))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* p = static_cast<uint8_t*>(ws);
  uint16_t* ln = reinterpret_cast<uint16_t*>(p); p += w.ln;
  uint16_t* qkv = reinterpret_cast<uint16_t*>(p); p += w.qkv;
  uint16_t* att = reinterpret_cast<uint16_t*>(p); p += w.att;
  uint16_t* h1 = reinterpret_cast<uint16_t*>(p); p += w.h1;
  uint16_t* mid = reinterpret_cast<uint16_t*>(p); p += w.mid;
  void* gws = p; p += w.gemm;
  const int h = dm->h;
  const float scale = 1.0f / sqrtf((float)dm->d);
  // weights restored to fp16 once for the m GPU batches (CTA-pair GEMMs only)
  const uint16_t *wqkv16 = nullptr, *wo16 = nullptr, *w116 = nullptr, *w216 = nullptr;
  if (w.w16) {
    uint16_t* q16 = reinterpret_cast<uint16_t*>(p);
    uint16_t* o16 = q16 + (int64_t)3 * h * h;
    uint16_t* f16a = o16 + (int64_t)h * h;
    uint16_t* f16b = f16a + (int64_t)h * dm->f;
    if ((rc = run_restore(L->wqkv, q16, st)) || (rc = run_restore(L->wo, o16, st))) return rc;
    wqkv16 = q16;
    wo16 = o16;
    if (dm->f > 0) {
      if ((rc = run_restore(L->w1, f16a, st)) || (rc = run_restore(L->w2, f16b, st))) return rc;
      w116 = f16a;
      w216 = f16b;
    }
  }
  for (int k = 0; k < m; ++k) {
    const uint16_t* xk = x + (int64_t)k * M * h;
    uint16_t* yk = y + (int64_t)k * M * h;
    const fg_kvcache kvk = kv_slice(*kv, k * g, g);
    if ((rc = run_layernorm(xk, M, h, L->ln1_g, L->ln1_b, dm->ln_eps, ln, st))) return rc;
    // QKV projection, then the 4-bit K/V of positions 0 .. s-1.  The append stays a kernel
    // of its own: quantising in the GEMM epilogue (fg_dequant_gemm_q4_kv) measured slower,
    // the epilogue warps becoming the bottleneck of the K/V tiles
    if ((rc = run_gemm(ln, M, L->wqkv, L->bqkv, FG_EPI_NONE, nullptr, qkv, gws, sms, st,
                       nullptr, wqkv16)))
      return rc;
    if ((rc = run_kv_append(qkv + h, qkv + 2 * h, 3 * h, s, 0, kvk, st))) return rc;
    if ((rc = run_prefill_attn(qkv, g, s, dm->H, dm->d, scale, att, sms, st))) return rc;
    if (dm->f > 0) {
      // O projection + residual into h1, then LN2(h1) (fused into a split-K reduce)
      if ((rc = run_gemm_ln(att, M, L->wo, L->bo, FG_EPI_RESIDUAL, xk, h1, L->ln2_g, L->ln2_b,
                            dm->ln_eps, ln, gws, sms, st, wo16)))
        return rc;
      if ((rc = run_gemm(ln, M, L->w1, L->b1, FG_EPI_RELU, nullptr, mid, gws, sms, st, nullptr,
                         w116)))
        return rc;
      if ((rc = run_gemm(mid, M, L->w2, L->b2, FG_EPI_RESIDUAL, h1, yk, gws, sms, st, nullptr,
                         w216)))
        return rc;
    } else if ((rc = run_gemm(att, M, L->wo, L->bo, FG_EPI_RESIDUAL, xk, yk, gws, sms, st,
                              nullptr, wo16))) {
      return rc;
    }
  }
  return FG_OK;
}

int fg_layer_decode(const fg_dims* dm, const fg_layer* L, fg_kvcache* kv, const uint16_t* x,
                    uint16_t* y, int32_t g, int32_t m, int32_t pos, void* ws, size_t ws_bytes,
                    void* stream) {
  int rc;
  if ((rc = check_dims(dm)) || (rc = check_layer(dm, L)) || (rc = check_kv(kv))) return rc;
  if (g <= 0 || m <= 0 || pos < 0) return FG_ERR_SHAPE;
  if (kv->B != g * m || kv->h != dm->h || kv->H != dm->H) return FG_ERR_SHAPE;
  if (pos + 1 > kv->cap) return FG_ERR_CAPACITY;
  if (!x || !y || !aligned16(x) || !aligned16(y)) return FG_ERR_ARG;
  const int64_t M = (int64_t)g * m;
  const LayerWs w = layer_ws(*dm, M, kv, pos + 1);
  if (!ws || !aligned16(ws) || ws_bytes < w.total) return FG_ERR_WORKSPACE;
  int sms = 0;
  if ((rc = check_device(&sms))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* p = static_cast<uint8_t*>(ws);
  uint16_t* ln = reinterpret_cast<uint16_t*>(p); p += w.ln;
  uint16_t* qkv = reinterpret_cast<uint16_t*>(p); p += w.qkv;
  uint16_t* att = reinterpret_cast<uint16_t*>(p); p += w.att;
  uint16_t* h1 = reinterpret_cast<uint16_t*>(p); p += w.h1;
  uint16_t* mid = reinterpret_cast<uint16_t*>(p); p += w.mid;
  void* gws = p; p += w.gemm;
  void* aws = p;
  const int h = dm->h;
  const float scale = 1.0f / sqrtf((float)dm->d);
  if ((rc = run_layernorm(x, M, h, L->ln1_g, L->ln1_b, dm->ln_eps, ln, st))) return rc;
  // QKV projection, then the new token's 4-bit K/V at position pos (a kernel of its own:
  // measured faster than the append in the streaming GEMM's epilogue)
  if ((rc = run_gemm(ln, M, L->wqkv, L->bqkv, FG_EPI_NONE, nullptr, qkv, gws, sms, st))) return rc;
  if ((rc = run_kv_append(qkv + h, qkv + 2 * h, 3 * h, 1, pos, *kv, st))) return rc;
  if ((rc = run_decode_attn(qkv, 3 * h, *kv, pos + 1, scale, att, aws, sms, st))) return rc;
  if (dm->f == 0) return run_gemm(att, M, L->wo, L->bo, FG_EPI_RESIDUAL, x, y, gws, sms, st);
  // O projection + residual into h1, then LN2(h1) (fused into the split-K reduce)
  if ((rc = run_gemm_ln(att, M, L->wo, L->bo, FG_EPI_RESIDUAL, x, h1, L->ln2_g, L->ln2_b,
                        dm->ln_eps, ln, gws, sms, st)))
    return rc;
  if ((rc = run_gemm(ln, M, L->w1, L->b1, FG_EPI_RELU, nullptr, mid, gws, sms, st))) return rc;
  return run_gemm(mid, M, L->w2, L->b2, FG_EPI_RESIDUAL, h1, y, gws, sms, st);
}

// ---------------------------------------------------------------- profiling ABI
int fg_prof_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = on != 0;
  return FG_OK;
}

int fg_prof_reset(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  prof_drain_locked();
  for (int i = 0; i < FG_K_COUNT; ++i) {
    g_launches[i] = 0;
    g_ms[i] = 0.0;
    g_work[i] = 0.0;
  }
  return FG_OK;
}

int fg_prof_query(int kind, int64_t* launches, double* ms, double* work) {
  if (kind < 0 || kind >= FG_K_COUNT) return FG_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  prof_drain_locked();
  if (launches) *launches = g_launches[kind];
  if (ms) *ms = g_ms[kind];
  if (work) *work = g_work[kind];
  return FG_OK;
}

const char* fg_kernel_name(int kind) {
  static const char* names[FG_K_COUNT] = {
      "q4g64_quantize", "q4g64_dequant", "q4_dequant_gemm_tc", "gemm_splitk_reduce",
      "q4kv_append", "q4kv_decode_attn", "decode_attn_combine", "prefill_attn",
      "layernorm", "q4_dequant_gemm_stream", "q4kv_decode_attn_topk", "q4_dequant_gemm_pair",
      "gemm_f16w_pair"};
  return (kind >= 0 && kind < FG_K_COUNT) ? names[kind] : "unknown";
}

}  // extern "C"
