// C-ABI entry points of libsd: argument checks, then one launcher per operation.
// Nothing is enqueued when a check fails.
#include <stdarg.h>
#include <string.h>

#include <atomic>
#include <chrono>
#include <map>
#include <mutex>
#include <thread>
#include <utility>

#include "sd_internal.cuh"
#include "sd_planes.cuh"

namespace sd {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
}

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

static std::atomic<int> g_fallback{0};
bool fallback_forced() { return g_fallback.load(std::memory_order_relaxed) != 0; }

static std::atomic<long long> g_launches{0};
void note_launches(int k) { g_launches.fetch_add(k, std::memory_order_relaxed); }
static long long launch_total() { return g_launches.load(std::memory_order_relaxed); }

int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return SD_OK;
}

int set_smem_limit(const void* kernel, size_t bytes, const char* what) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return check_launch(what);
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_pair(dev, kernel);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return SD_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
      cudaSuccess)
    return check_launch(what);
  done[key] = bytes;
  return SD_OK;
}

int device_sm_count() {
  static std::atomic<int> cnt[kMaxDev];
  const int c = per_device_cached(cnt, [] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
      cudaGetLastError();
      return 0;
    }
    return v;
  });
  return c > 0 ? c : 152;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Validates a shape and fills Dims.  need_n64: n and n_cap multiples of 64 (the
// bulk-copy and cp.async bit-plane kernels); need_cap64: n_cap a multiple of 64
// (the planes layout), any n.
static int check_shape(const sd_shape* sh, Dims* out, bool need_n64 = false,
                       bool need_cap64 = false) {
  if (!sh) return fail(SD_ERR_INVALID_ARG, "shape is NULL");
  if (sh->batch < 1 || sh->hq < 1 || sh->hkv < 1 || sh->n < 1)
    return fail(SD_ERR_INVALID_ARG, "shape: batch, hq, hkv and n must be positive");
  if (sh->hq % sh->hkv)
    return fail(SD_ERR_INVALID_ARG, "shape: hq (%d) is not a multiple of hkv (%d)", sh->hq,
                sh->hkv);
  int G = sh->hq / sh->hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(SD_ERR_UNSUPPORTED, "shape: group size %d (supported: 1, 2, 4, 8)", G);
  if (sh->d != kD) return fail(SD_ERR_UNSUPPORTED, "shape: d = %d (supported: 128)", sh->d);
  int64_t ncap = sh->n_cap ? sh->n_cap : sh->n;
  if (ncap < sh->n) return fail(SD_ERR_INVALID_ARG, "shape: n_cap < n");
  if (sh->n >= (int64_t)1 << 31 || ncap >= (int64_t)1 << 31)
    return fail(SD_ERR_UNSUPPORTED, "shape: n >= 2^31");
  if ((int64_t)sh->batch * sh->hkv > 65535)
    return fail(SD_ERR_UNSUPPORTED, "shape: batch * hkv > 65535");
  if (need_n64 && (sh->n % 64 || ncap % 64))
    return fail(SD_ERR_UNSUPPORTED, "bit planes need n and n_cap to be multiples of 64");
  if (need_cap64 && ncap % 64)
    return fail(SD_ERR_UNSUPPORTED, "bit planes need n_cap to be a multiple of 64");
  *out = Dims{sh->batch, sh->hq, sh->hkv, G, sh->n, ncap};
  return SD_OK;
}

static int check_encoder(const sd_encoder* enc) {
  if (!enc || !enc->W1) return fail(SD_ERR_INVALID_ARG, "encoder: W1 is NULL");
  if (enc->hidden != 0 && enc->hidden != 32 && enc->hidden != 64 && enc->hidden != 128)
    return fail(SD_ERR_UNSUPPORTED, "encoder: hidden = %d (supported: 0, 32, 64, 128)",
                enc->hidden);
  if (enc->hidden && !enc->W2) return fail(SD_ERR_INVALID_ARG, "encoder: W2 is NULL");
  return SD_OK;
}

}  // namespace sd

using namespace sd;

extern "C" {

int sd_version(void) { return 104; }

int64_t sd_launch_count(void) { return (int64_t)launch_total(); }

const char* sd_last_error(void) { return g_err; }

// sd_build_index and sd_append_index: tokens [t0, n) of K are (re)indexed.
static int index_tokens(const char* fn, int kind, const sd_shape* shape, int64_t t0,
                        const void* K, const sd_encoder* enc, void* out0, void* out1,
                        void* stream) {
  Dims s;
  int rc = check_shape(shape, &s);
  if (rc) return rc;
  if (t0 < 0 || t0 > s.n)
    return fail(SD_ERR_INVALID_ARG, "%s: n_old = %lld outside [0, n = %lld]", fn, (long long)t0,
                (long long)s.n);
  if (!K || !out0) return fail(SD_ERR_INVALID_ARG, "%s: K or out0 is NULL", fn);
  if (!aligned16(K) || !aligned16(out0))
    return fail(SD_ERR_INVALID_ARG, "%s: K and out0 must be 16-byte aligned", fn);
  if (kind == SD_IDX_SIG && (rc = check_encoder(enc))) return rc;
  if (kind == SD_IDX_PLANES && s.ncap % 64)
    return fail(SD_ERR_UNSUPPORTED, "%s: bit planes need n_cap to be a multiple of 64", fn);
  if (kind == SD_IDX_PLANES && !out1)
    return fail(SD_ERR_INVALID_ARG, "%s: scales (out1) is NULL", fn);
  if (kind != SD_IDX_SIG && kind != SD_IDX_PLANES && kind != SD_IDX_MINMAX &&
      kind != SD_IDX_LANDMARK)
    return fail(SD_ERR_INVALID_ARG, "%s: unknown kind %d", fn, kind);
  if (t0 == s.n) return SD_OK;  // nothing appended
  cudaStream_t st = (cudaStream_t)stream;
  switch (kind) {
    case SD_IDX_SIG:
      return launch_sig_build(s, (const uint16_t*)K, *enc, (uint32_t*)out0, st, t0);
    case SD_IDX_PLANES:
      return launch_plane_build(s, (const uint16_t*)K, (uint32_t*)out0, (uint16_t*)out1, st, t0);
    case SD_IDX_LANDMARK:
      return launch_landmark_build(s, (const uint16_t*)K, (uint16_t*)out0, st, t0);
    default:
      return launch_minmax_build(s, (const uint16_t*)K, (uint16_t*)out0, st, t0);
  }
}

int sd_build_index(int kind, const sd_shape* shape, const void* K, const sd_encoder* enc,
                   void* out0, void* out1, void* stream) {
  return index_tokens("sd_build_index", kind, shape, 0, K, enc, out0, out1, stream);
}

int sd_append_index(int kind, const sd_shape* shape, int64_t n_old, const void* K,
                    const sd_encoder* enc, void* out0, void* out1, void* stream) {
  return index_tokens("sd_append_index", kind, shape, n_old, K, enc, out0, out1, stream);
}

int sd_encode_query(const sd_shape* shape, const void* q, const sd_encoder* enc, uint32_t* qsig,
                    void* stream) {
  Dims s;
  int rc = check_shape(shape, &s);
  if (rc) return rc;
  if ((rc = check_encoder(enc))) return rc;
  if (!q || !qsig) return fail(SD_ERR_INVALID_ARG, "sd_encode_query: q or qsig is NULL");
  return launch_encode_query(s, (const uint16_t*)q, *enc, qsig, (cudaStream_t)stream);
}

// Pointers and budget range of a read plan (modes as sd_plan_mode).
static int check_plan_args(const char* fn, const void* q, const float* sigma2, int mode,
                           int budget) {
  const bool split = mode == SD_PLAN_SPLIT;
  if ((mode == SD_PLAN_WATERFILL || mode == SD_PLAN_TOPQ || split) && !q)
    return fail(SD_ERR_INVALID_ARG, "%s: q is NULL", fn);
  if ((mode == SD_PLAN_WATERFILL || mode == SD_PLAN_FIXED || split) && !sigma2)
    return fail(SD_ERR_INVALID_ARG, "%s: sigma2 is NULL", fn);
  if ((mode == SD_PLAN_WATERFILL || split) && (budget < 0 || budget > 4 * kD))
    return fail(SD_ERR_INVALID_ARG, "%s: budget %d outside [0, %d]", fn, budget, 4 * kD);
  if ((mode == SD_PLAN_FIXED || mode == SD_PLAN_TOPQ) && (budget < 0 || budget > kD))
    return fail(SD_ERR_INVALID_ARG, "%s: channel count %d outside [0, %d]", fn, budget, kD);
  return SD_OK;
}

int sd_plan(const sd_shape* shape, const void* q, const float* sigma2, int mode, int budget,
            uint8_t* plan, void* stream) {
  Dims s;
  int rc = check_shape(shape, &s);
  if (rc) return rc;
  if (mode < 0 || mode > 4) return fail(SD_ERR_INVALID_ARG, "sd_plan: unknown mode %d", mode);
  if (mode == SD_PLAN_SPLIT && s.Hkv > kSplitMaxHeads)
    return fail(SD_ERR_UNSUPPORTED, "sd_plan: SD_PLAN_SPLIT with hkv = %d > %d", s.Hkv,
                kSplitMaxHeads);
  if ((rc = check_plan_args("sd_plan", q, sigma2, mode, budget))) return rc;
  if (!plan) return fail(SD_ERR_INVALID_ARG, "sd_plan: plan is NULL");
  return launch_plan(s, (const uint16_t*)q, sigma2, mode, budget, plan, (cudaStream_t)stream);
}

int sd_score(int kind, const sd_shape* shape, const void* index0, const void* index1,
             const void* q_or_qsig, const uint8_t* plan, void* scores, void* stream) {
  Dims s;
  int rc = check_shape(shape, &s, false, kind == SD_IDX_PLANES);
  if (rc) return rc;
  if (!index0 || !q_or_qsig || !scores) return fail(SD_ERR_INVALID_ARG, "sd_score: NULL input");
  if (!aligned16(index0) || !aligned16(scores))
    return fail(SD_ERR_INVALID_ARG, "sd_score: index0 and scores must be 16-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  switch (kind) {
    case SD_IDX_SIG:
      return launch_score_hamming(s, (const uint32_t*)index0, (const uint32_t*)q_or_qsig,
                                  (int32_t*)scores, st);
    case SD_IDX_PLANES:
      if (!index1 || !plan) return fail(SD_ERR_INVALID_ARG, "sd_score: scales or plan NULL");
      return launch_score_planes(s, (const uint32_t*)index0, (const uint16_t*)index1, plan,
                                 (const uint16_t*)q_or_qsig, (float*)scores, st);
    case SD_IDX_MINMAX:
      return launch_score_quest(s, (const uint16_t*)index0, (const uint16_t*)q_or_qsig,
                                (float*)scores, st);
    case SD_IDX_LANDMARK:
      return launch_score_landmark(s, (const uint16_t*)index0, (const uint16_t*)q_or_qsig,
                                   (float*)scores, st);
    default:
      return fail(SD_ERR_INVALID_ARG, "sd_score: unknown kind %d", kind);
  }
}

size_t sd_topk_workspace_size(int64_t rows, int64_t n_units, const sd_select* sel) {
  if (!sel || rows < 1 || n_units < 1) return 0;
  return topk_workspace_bytes(rows, n_units, *sel);
}

int sd_topk(int score_type, const void* scores, int64_t rows, int64_t n_units,
            int64_t n_tokens, const sd_select* sel, int32_t* idx, int64_t idx_stride,
            int32_t* count, void* workspace, size_t ws_bytes, void* stream) {
  if (!sel || !scores || !idx || !count) return fail(SD_ERR_INVALID_ARG, "sd_topk: NULL input");
  if (score_type != SD_SCORE_I32 && score_type != SD_SCORE_F32)
    return fail(SD_ERR_INVALID_ARG, "sd_topk: unknown score type %d", score_type);
  if (rows < 1 || n_units < 1 || n_units >= ((int64_t)1 << 31) || rows >= ((int64_t)1 << 31))
    return fail(SD_ERR_INVALID_ARG, "sd_topk: bad rows / n_units");
  if (sel->k < 1 || sel->k > kMaxTopK)
    return fail(SD_ERR_UNSUPPORTED, "sd_topk: k = %d outside [1, %d]", sel->k, kMaxTopK);
  if (sel->sink < 0 || sel->local < 0 || sel->block < 1)
    return fail(SD_ERR_INVALID_ARG, "sd_topk: negative window or block < 1");
  if (n_tokens < 1 || n_tokens > n_units * (int64_t)sel->block ||
      n_tokens <= (n_units - 1) * (int64_t)sel->block)
    return fail(SD_ERR_INVALID_ARG, "sd_topk: n_tokens does not match n_units * block");
  int64_t max_units = n_units < (int64_t)sel->sink + sel->local + sel->k
                          ? n_units : (int64_t)sel->sink + sel->local + sel->k;
  if (n_tokens >= ((int64_t)1 << 31) || max_units * sel->block >= ((int64_t)1 << 31))
    return fail(SD_ERR_UNSUPPORTED, "sd_topk: %lld tokens or %lld output entries per row (limit 2^31 - 1)",
                (long long)n_tokens, (long long)(max_units * sel->block));
  if (idx_stride < max_units * sel->block)
    return fail(SD_ERR_INVALID_ARG, "sd_topk: idx_stride %lld < %lld", (long long)idx_stride,
                (long long)(max_units * sel->block));
  if (n_units > kSmallRow && rows > 65535)
    return fail(SD_ERR_UNSUPPORTED, "sd_topk: more than 65535 rows of over %d units", kSmallRow);
  size_t need = topk_workspace_bytes(rows, n_units, *sel);
  if (need && (!workspace || ws_bytes < need))
    return fail(SD_ERR_WORKSPACE, "sd_topk: workspace %zu < %zu bytes", ws_bytes, need);
  return launch_topk(score_type, scores, rows, n_units, n_tokens, *sel, idx, idx_stride, count,
                     workspace, ws_bytes, (cudaStream_t)stream);
}

int sd_plan_score(const sd_shape* shape, const void* planes, const void* scales, const void* q,
                  const float* sigma2, int mode, int budget, uint8_t* plan, float* scores,
                  float* wmax, void* stream) {
  Dims s;
  int rc = check_shape(shape, &s, false, true);
  if (rc) return rc;
  if (!planes || !scales || !q || !scores)
    return fail(SD_ERR_INVALID_ARG, "sd_plan_score: NULL input");
  if (!aligned16(planes) || !aligned16(scores))
    return fail(SD_ERR_INVALID_ARG, "sd_plan_score: planes and scores must be 16-byte aligned");
  if ((uintptr_t)wmax % 4)
    return fail(SD_ERR_INVALID_ARG, "sd_plan_score: wmax must be 4-byte aligned");
  if (mode < 0 || mode > 4)
    return fail(SD_ERR_INVALID_ARG, "sd_plan_score: unknown plan mode %d", mode);
  if ((rc = check_plan_args("sd_plan_score", q, sigma2, mode, budget))) return rc;
  if (mode == SD_PLAN_SPLIT) {  // the heads of a sequence are coupled: plan kernel, then scan
    if (!plan) return fail(SD_ERR_INVALID_ARG, "sd_plan_score: SD_PLAN_SPLIT needs the plan buffer");
    if (s.Hkv > kSplitMaxHeads)
      return fail(SD_ERR_UNSUPPORTED, "sd_plan_score: SD_PLAN_SPLIT with hkv = %d > %d", s.Hkv,
                  kSplitMaxHeads);
    if ((rc = launch_plan(s, (const uint16_t*)q, sigma2, mode, budget, plan, (cudaStream_t)stream)))
      return rc;
    return launch_score_planes(s, (const uint32_t*)planes, (const uint16_t*)scales, plan,
                               (const uint16_t*)q, scores, (cudaStream_t)stream, nullptr, nullptr,
                               wmax);
  }
  const PsPlanIn pl{true, sigma2, mode, budget, plan};
  return launch_score_planes(s, (const uint32_t*)planes, (const uint16_t*)scales, nullptr,
                             (const uint16_t*)q, scores, (cudaStream_t)stream, nullptr, &pl, wmax);
}

int sd_topk_wmax(const float* scores, const float* wmax, int64_t rows, int64_t n,
                 const sd_select* sel, int32_t* idx, int64_t idx_stride, int32_t* count,
                 void* workspace, size_t ws_bytes, void* stream) {
  if (!scores || !wmax)
    return fail(SD_ERR_INVALID_ARG, "sd_topk_wmax: NULL input");
  if (!sel || sel->block != 1)
    return fail(SD_ERR_INVALID_ARG, "sd_topk_wmax: sel is NULL or sel.block != 1");
  if (n < 1) return fail(SD_ERR_INVALID_ARG, "sd_topk_wmax: n = %lld < 1", (long long)n);
  if (!aligned16(scores) || (uintptr_t)wmax % 4)
    return fail(SD_ERR_INVALID_ARG, "sd_topk_wmax: scores must be 16-byte, wmax 4-byte aligned");
  // the remaining checks are sd_topk's
  if (!idx || !count) return fail(SD_ERR_INVALID_ARG, "sd_topk_wmax: NULL input");
  if (rows < 1 || n >= ((int64_t)1 << 31) || rows >= ((int64_t)1 << 31))
    return fail(SD_ERR_INVALID_ARG, "sd_topk_wmax: bad rows / n");
  if (sel->k < 1 || sel->k > kMaxTopK)
    return fail(SD_ERR_UNSUPPORTED, "sd_topk_wmax: k = %d outside [1, %d]", sel->k, kMaxTopK);
  if (sel->sink < 0 || sel->local < 0)
    return fail(SD_ERR_INVALID_ARG, "sd_topk_wmax: negative window");
  const int64_t max_units = n < (int64_t)sel->sink + sel->local + sel->k
                                ? n : (int64_t)sel->sink + sel->local + sel->k;
  if (idx_stride < max_units)
    return fail(SD_ERR_INVALID_ARG, "sd_topk_wmax: idx_stride %lld < %lld",
                (long long)idx_stride, (long long)max_units);
  if (n > kSmallRow && rows > 65535)
    return fail(SD_ERR_UNSUPPORTED, "sd_topk_wmax: more than 65535 rows of over %d units",
                kSmallRow);
  const size_t need = topk_workspace_bytes(rows, n, *sel);
  if (need && (!workspace || ws_bytes < need))
    return fail(SD_ERR_WORKSPACE, "sd_topk_wmax: workspace %zu < %zu bytes", ws_bytes, need);
  return launch_topk_wmax(scores, wmax, rows, n, *sel, idx, idx_stride, count, workspace,
                          ws_bytes, (cudaStream_t)stream);
}

size_t sd_score_topk_workspace_size(const sd_shape* shape, const sd_select* sel) {
  Dims s;
  if (!sel || check_shape(shape, &s, true)) return 0;
  return score_topk_workspace_bytes((int64_t)s.B * s.Hkv, s.n, *sel);
}

int sd_score_topk(const sd_shape* shape, const void* planes, const void* scales, const void* q,
                  const uint8_t* plan, const sd_select* sel, float* scores, int32_t* idx,
                  int64_t idx_stride, int32_t* count, void* workspace, size_t ws_bytes,
                  void* stream) {
  Dims s;
  int rc = check_shape(shape, &s, true);
  if (rc) return rc;
  if (!planes || !scales || !q || !plan || !sel || !scores || !idx || !count)
    return fail(SD_ERR_INVALID_ARG, "sd_score_topk: NULL input");
  if (!aligned16(planes) || !aligned16(scores))
    return fail(SD_ERR_INVALID_ARG, "sd_score_topk: planes and scores must be 16-byte aligned");
  if (sel->k < 1 || sel->k > kMaxTopK)
    return fail(SD_ERR_UNSUPPORTED, "sd_score_topk: k = %d outside [1, %d]", sel->k, kMaxTopK);
  if (sel->sink < 0 || sel->local < 0 || sel->block != 1)
    return fail(SD_ERR_INVALID_ARG, "sd_score_topk: negative window or block != 1");
  const int64_t rows = (int64_t)s.B * s.Hkv;
  const int64_t max_units = s.n < (int64_t)sel->sink + sel->local + sel->k
                                ? s.n : (int64_t)sel->sink + sel->local + sel->k;
  if (idx_stride < max_units)
    return fail(SD_ERR_INVALID_ARG, "sd_score_topk: idx_stride %lld < %lld",
                (long long)idx_stride, (long long)max_units);
  const size_t need = score_topk_workspace_bytes(rows, s.n, *sel);
  if (!workspace || ws_bytes < need)
    return fail(SD_ERR_WORKSPACE, "sd_score_topk: workspace %zu < %zu bytes", ws_bytes, need);
  if ((uintptr_t)workspace % 256)
    return fail(SD_ERR_INVALID_ARG, "sd_score_topk: workspace must be 256-byte aligned");
  return launch_score_topk(s, (const uint32_t*)planes, (const uint16_t*)scales, plan,
                           (const uint16_t*)q, *sel, scores, idx, idx_stride, count, workspace,
                           (cudaStream_t)stream);
}

size_t sd_gather_attend_workspace_size(const sd_shape* shape, int64_t max_count) {
  Dims s;
  if (check_shape(shape, &s) || max_count < 0) return 0;
  return attend_workspace_bytes(s, max_count);
}

int sd_gather_attend(const sd_shape* shape, const void* q, const void* K, const void* V,
                     const int32_t* idx, int64_t idx_stride, const int32_t* count,
                     int64_t max_count, float scale, float* out, float* lse, void* workspace,
                     size_t ws_bytes, void* stream) {
  Dims s;
  int rc = check_shape(shape, &s);
  if (rc) return rc;
  if (!q || !K || !V || !idx || !count || !out)
    return fail(SD_ERR_INVALID_ARG, "sd_gather_attend: NULL input");
  if (!aligned16(K) || !aligned16(V))
    return fail(SD_ERR_INVALID_ARG, "sd_gather_attend: K and V must be 16-byte aligned");
  if (max_count < 0 || idx_stride < max_count)
    return fail(SD_ERR_INVALID_ARG, "sd_gather_attend: bad max_count / idx_stride");

  size_t need = attend_workspace_bytes(s, max_count);
  if (need && (!workspace || ws_bytes < need))
    return fail(SD_ERR_WORKSPACE, "sd_gather_attend: workspace %zu < %zu bytes", ws_bytes,
                need);
  return launch_gather_attend(s, (const uint16_t*)q, (const uint16_t*)K, (const uint16_t*)V, idx,
                              idx_stride, count, max_count, scale, out, lse, workspace, ws_bytes,
                              (cudaStream_t)stream);
}

size_t sd_hamming_topk_workspace_size(const sd_shape* shape, const sd_select* sel) {
  Dims s;
  if (check_shape(shape, &s) || !sel) return 0;
  return hamming_topk_workspace_bytes(s, *sel);
}

int sd_hamming_topk(const sd_shape* shape, const uint32_t* sig, const uint32_t* qsig,
                    const sd_select* sel, int32_t* idx, int64_t idx_stride, int32_t* count,
                    void* workspace, size_t ws_bytes, void* stream) {
  Dims s;
  int rc = check_shape(shape, &s);
  if (rc) return rc;
  if (!sig || !qsig || !sel || !idx || !count)
    return fail(SD_ERR_INVALID_ARG, "sd_hamming_topk: NULL input");
  if (sel->block != 1)
    return fail(SD_ERR_INVALID_ARG, "sd_hamming_topk: sel.block must be 1 (token mode)");
  if (sel->k < 1 || sel->k > kMaxTopK)
    return fail(SD_ERR_UNSUPPORTED, "sd_hamming_topk: k = %d outside [1, %d]", sel->k, kMaxTopK);
  if (sel->sink < 0 || sel->local < 0)
    return fail(SD_ERR_INVALID_ARG, "sd_hamming_topk: negative window");
  const int64_t max_units = s.n < (int64_t)sel->sink + sel->local + sel->k
                                ? s.n : (int64_t)sel->sink + sel->local + sel->k;
  if (idx_stride < max_units)
    return fail(SD_ERR_INVALID_ARG, "sd_hamming_topk: idx_stride %lld < %lld",
                (long long)idx_stride, (long long)max_units);
  if (!hamming_topk_supported(s, *sel))
    return fail(SD_ERR_UNSUPPORTED,
                "sd_hamming_topk: more than 2,097,152 competing tokens or 65535 rows");
  const size_t need = hamming_topk_workspace_bytes(s, *sel);
  if (!workspace || ws_bytes < need)
    return fail(SD_ERR_WORKSPACE, "sd_hamming_topk: workspace %zu < %zu bytes", ws_bytes, need);
  return launch_hamming_topk(s, sig, qsig, *sel, idx, idx_stride, count, workspace,
                             (cudaStream_t)stream);
}

size_t sd_select_attend_workspace_size(const sd_shape* shape, const sd_select* sel,
                                       int64_t max_count) {
  Dims s;
  if (check_shape(shape, &s) || !sel || max_count < 0) return 0;
  return select_attend_workspace_bytes(s, *sel, max_count);
}

int sd_select_attend(const sd_shape* shape, const float* scores, const float* wmax,
                     const sd_select* sel, const void* q, const void* K, const void* V,
                     float scale, int32_t* idx, int64_t idx_stride, int32_t* count,
                     int64_t max_count, float* out, float* lse, void* workspace,
                     size_t ws_bytes, void* stream) {
  Dims s;
  int rc = check_shape(shape, &s);
  if (rc) return rc;
  if (!scores || !wmax || !q || !K || !V || !idx || !count || !out)
    return fail(SD_ERR_INVALID_ARG, "sd_select_attend: NULL input");
  if (!sel || sel->block != 1)
    return fail(SD_ERR_INVALID_ARG, "sd_select_attend: sel is NULL or sel.block != 1");
  const int64_t n = s.n, rows = (int64_t)s.B * s.Hkv;
  if (n < 1) return fail(SD_ERR_INVALID_ARG, "sd_select_attend: n = %lld < 1", (long long)n);
  if (!aligned16(scores) || (uintptr_t)wmax % 4)
    return fail(SD_ERR_INVALID_ARG,
                "sd_select_attend: scores must be 16-byte, wmax 4-byte aligned");
  if (!aligned16(K) || !aligned16(V))
    return fail(SD_ERR_INVALID_ARG, "sd_select_attend: K and V must be 16-byte aligned");
  if (sel->k < 1 || sel->k > kMaxTopK)
    return fail(SD_ERR_UNSUPPORTED, "sd_select_attend: k = %d outside [1, %d]", sel->k, kMaxTopK);
  if (sel->sink < 0 || sel->local < 0)
    return fail(SD_ERR_INVALID_ARG, "sd_select_attend: negative window");
  const int64_t max_units = n < (int64_t)sel->sink + sel->local + sel->k
                                ? n : (int64_t)sel->sink + sel->local + sel->k;
  if (idx_stride < max_units || max_count < max_units || idx_stride < max_count)
    return fail(SD_ERR_INVALID_ARG,
                "sd_select_attend: need idx_stride >= max_count >= %lld (got %lld, %lld)",
                (long long)max_units, (long long)idx_stride, (long long)max_count);
  if (n > kSmallRow && rows > 65535)
    return fail(SD_ERR_UNSUPPORTED, "sd_select_attend: more than 65535 rows of over %d units",
                kSmallRow);
  const size_t need = select_attend_workspace_bytes(s, *sel, max_count);
  if (need && (!workspace || ws_bytes < need))
    return fail(SD_ERR_WORKSPACE, "sd_select_attend: workspace %zu < %zu bytes", ws_bytes, need);
  return launch_select_attend(s, scores, wmax, *sel, (const uint16_t*)q, (const uint16_t*)K,
                              (const uint16_t*)V, scale, idx, idx_stride, count, max_count, out,
                              lse, workspace, ws_bytes, (cudaStream_t)stream);
}

int sd_offload_gather(const sd_shape* shape, const uint32_t* host_planes,
                      const uint16_t* host_scales, const uint8_t* plan, uint32_t* dev_planes,
                      uint16_t* dev_scales, void* stream) {
  Dims s;
  int rc = check_shape(shape, &s, true);
  if (rc) return rc;
  if (!host_planes || !host_scales || !plan || !dev_planes || !dev_scales)
    return fail(SD_ERR_INVALID_ARG, "sd_offload_gather: NULL input");
  if (!aligned16(host_planes) || !aligned16(dev_planes))
    return fail(SD_ERR_INVALID_ARG, "sd_offload_gather: planes must be 16-byte aligned");
  // the host buffers must be pinned and mapped into the device address space
  const void* hp[2] = {host_planes, host_scales};
  const void* dp[2] = {nullptr, nullptr};
  for (int i = 0; i < 2; ++i) {
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, hp[i]);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(SD_ERR_INVALID_ARG, "sd_offload_gather: cannot query host pointer: %s",
                  cudaGetErrorString(e));
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer)
      return fail(SD_ERR_INVALID_ARG,
                  "sd_offload_gather: host buffers must be pinned (cudaHostAlloc/Register)");
    dp[i] = a.devicePointer;
  }
  return launch_offload_gather(s, (const uint32_t*)dp[0], (const uint16_t*)dp[1], plan,
                               dev_planes, dev_scales, (cudaStream_t)stream);
}

int sd_delta_select(const sd_shape* shape, const sd_select* sel, const float* scores,
                    const int32_t* idx, int64_t idx_stride, const int32_t* count,
                    int32_t admit_cap, int32_t step, const sd_resident* res,
                    int32_t* plan_slot, int32_t* plan_unit, int32_t* plan_evict,
                    int32_t* plan_count, int32_t* pool_idx, int64_t pool_stride,
                    int32_t* pool_count, void* stream) {
  Dims s;
  int rc = check_shape(shape, &s);
  if (rc) return rc;
  if (!sel || sel->block < 1 || sel->block > 4096)
    return fail(SD_ERR_INVALID_ARG, "sd_delta_select: sel is NULL or sel.block outside [1, 4096]");
  if (sel->k < 1 || sel->sink < 0 || sel->local < 0)
    return fail(SD_ERR_INVALID_ARG, "sd_delta_select: bad k, sink or local");
  if (!scores || !idx || !count || !res || !plan_count || !pool_idx || !pool_count)
    return fail(SD_ERR_INVALID_ARG, "sd_delta_select: NULL input");
  if (!res->slot_unit || !res->slot_last || !res->unit_slot)
    return fail(SD_ERR_INVALID_ARG, "sd_delta_select: NULL resident-set array");
  if (res->n_slots < 1 || res->n_slots > kDsMaxSlots)
    return fail(SD_ERR_UNSUPPORTED, "sd_delta_select: n_slots = %d outside [1, %d]",
                res->n_slots, kDsMaxSlots);
  if (admit_cap < 0 || admit_cap > kDsMaxUnits)
    return fail(SD_ERR_INVALID_ARG, "sd_delta_select: admit_cap = %d outside [0, %d]", admit_cap,
                kDsMaxUnits);
  if (admit_cap > 0 && (!plan_slot || !plan_unit || !plan_evict))
    return fail(SD_ERR_INVALID_ARG, "sd_delta_select: NULL plan array");
  if (step < 0 || step >= 0x7FFFFFFF)
    return fail(SD_ERR_INVALID_ARG, "sd_delta_select: step = %d outside [0, 2^31 - 2]", step);
  const int64_t nu = (s.n + sel->block - 1) / sel->block;
  const int64_t units = imin64(nu, (int64_t)sel->sink + sel->local + sel->k);
  if (units > kDsMaxUnits)
    return fail(SD_ERR_UNSUPPORTED, "sd_delta_select: up to %lld predicted units (limit %d)",
                (long long)units, kDsMaxUnits);
  if (idx_stride < units * sel->block || pool_stride < units * sel->block)
    return fail(SD_ERR_INVALID_ARG, "sd_delta_select: idx_stride and pool_stride must be at "
                "least %lld", (long long)(units * sel->block));
  return launch_delta_select((int64_t)s.B * s.Hkv, nu, s.n, sel->block, sel->sink, sel->local,
                             sel->k, scores, idx, idx_stride, count, admit_cap, step, res->n_slots,
                             res->slot_unit, res->slot_last, res->unit_slot, plan_slot,
                             plan_unit, plan_evict, plan_count, pool_idx, pool_stride,
                             pool_count, (cudaStream_t)stream);
}

// A device address for p: device memory as it is, pinned host memory through its
// mapping; anything else is refused.
static int device_view(const char* fn, const void* p, const void** out) {
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(SD_ERR_INVALID_ARG, "%s: cannot query pointer: %s", fn, cudaGetErrorString(e));
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *out = p;
    return SD_OK;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer) {
    *out = a.devicePointer;
    return SD_OK;
  }
  return fail(SD_ERR_INVALID_ARG, "%s: K and V must be device or pinned host memory", fn);
}

int sd_resident_gather(const sd_shape* shape, int32_t block, const void* K, const void* V,
                       const int32_t* plan_slot, const int32_t* plan_unit,
                       const int32_t* plan_count, int32_t admit_cap, int32_t n_slots,
                       void* K_pool, void* V_pool, void* stream) {
  Dims s;
  int rc = check_shape(shape, &s);
  if (rc) return rc;
  if (block < 1 || block > 4096)
    return fail(SD_ERR_INVALID_ARG, "sd_resident_gather: block = %d outside [1, 4096]", block);
  if (n_slots < 1 || n_slots > kDsMaxSlots)
    return fail(SD_ERR_UNSUPPORTED, "sd_resident_gather: n_slots = %d outside [1, %d]", n_slots,
                kDsMaxSlots);
  if (admit_cap < 0 || admit_cap > kDsMaxUnits)
    return fail(SD_ERR_INVALID_ARG, "sd_resident_gather: admit_cap = %d outside [0, %d]",
                admit_cap, kDsMaxUnits);
  if (!K || !V || !plan_count || !K_pool || !V_pool ||
      (admit_cap > 0 && (!plan_slot || !plan_unit)))
    return fail(SD_ERR_INVALID_ARG, "sd_resident_gather: NULL input");
  if (!aligned16(K) || !aligned16(V) || !aligned16(K_pool) || !aligned16(V_pool))
    return fail(SD_ERR_INVALID_ARG, "sd_resident_gather: K, V and the pools must be 16-byte "
                "aligned");
  const void *dk = nullptr, *dv = nullptr;
  if ((rc = device_view("sd_resident_gather", K, &dk))) return rc;
  if ((rc = device_view("sd_resident_gather", V, &dv))) return rc;
  return launch_resident_gather(s, block, (const uint16_t*)dk, (const uint16_t*)dv, plan_slot,
                                plan_unit, plan_count, admit_cap, n_slots, (uint16_t*)K_pool,
                                (uint16_t*)V_pool, (cudaStream_t)stream);
}

int sd_shard_candidates(const float* scores, int64_t rows, int64_t n_s, const int32_t* idx,
                        int64_t idx_stride, const int32_t* count, int32_t sink_s, int32_t local_s,
                        int64_t offset, int32_t k, float* cand_score, int32_t* cand_idx,
                        int32_t* cand_count, void* stream) {
  if (!scores || !idx || !count || !cand_score || !cand_idx || !cand_count)
    return fail(SD_ERR_INVALID_ARG, "sd_shard_candidates: NULL input");
  if (rows < 1 || rows > 65535 * 8 || n_s < 1 || n_s >= ((int64_t)1 << 31) || offset < 0 ||
      offset + n_s >= ((int64_t)1 << 31))
    return fail(SD_ERR_INVALID_ARG, "sd_shard_candidates: bad rows, n_s or offset");
  if (k < 1 || k > kMaxTopK || sink_s < 0 || local_s < 0 || idx_stride < 1)
    return fail(SD_ERR_INVALID_ARG, "sd_shard_candidates: bad k, window or stride");
  return launch_shard_candidates(scores, rows, n_s, idx, idx_stride, count, sink_s, local_s,
                                 offset, k, cand_score, cand_idx, cand_count,
                                 (cudaStream_t)stream);
}

int sd_topk_merge(int64_t rows, int32_t shards, int32_t k, const float* cand_score,
                  const int32_t* cand_idx, const int32_t* cand_count, int32_t* idx,
                  int64_t idx_stride, int32_t* count, void* stream) {
  if (!cand_score || !cand_idx || !cand_count || !idx || !count)
    return fail(SD_ERR_INVALID_ARG, "sd_topk_merge: NULL input");
  if (rows < 1 || rows > 2147483647 || shards < 1 || k < 1 || k > kMaxTopK || idx_stride < k)
    return fail(SD_ERR_INVALID_ARG, "sd_topk_merge: bad rows, shards, k or stride");
  if ((int64_t)shards * k > kMergeMaxCand)
    return fail(SD_ERR_UNSUPPORTED, "sd_topk_merge: shards * k = %lld > %d",
                (long long)shards * k, kMergeMaxCand);
  return launch_topk_merge(rows, shards, k, cand_score, cand_idx, cand_count, idx, idx_stride,
                           count, (cudaStream_t)stream);
}

int sd_shard_select(int64_t rows, const int32_t* sel_idx, int64_t sel_stride,
                    const int32_t* sel_count, int64_t offset, int64_t n_s, int32_t sink_s,
                    int32_t local_s, int32_t k, int32_t* idx, int64_t idx_stride, int32_t* count,
                    void* stream) {
  if (!sel_idx || !sel_count || !idx || !count)
    return fail(SD_ERR_INVALID_ARG, "sd_shard_select: NULL input");
  if (rows < 1 || rows > 65535 * 8 || n_s < 1 || n_s >= ((int64_t)1 << 31) || offset < 0 ||
      sink_s < 0 || local_s < 0 || (int64_t)sink_s + local_s > n_s || k < 0 || sel_stride < k)
    return fail(SD_ERR_INVALID_ARG, "sd_shard_select: bad rows, n_s, offset, window or stride");
  if (idx_stride < (int64_t)sink_s + local_s + k)
    return fail(SD_ERR_INVALID_ARG, "sd_shard_select: idx_stride %lld < %lld",
                (long long)idx_stride, (long long)sink_s + local_s + k);
  return launch_shard_select(rows, sel_idx, sel_stride, sel_count, offset, n_s, sink_s, local_s,
                             idx, idx_stride, count, (cudaStream_t)stream);
}

int sd_attend_combine(int32_t shards, int64_t batch, int32_t hq, const float* outs,
                      const float* lses, float* out, float* lse, void* stream) {
  if (!outs || !lses || !out) return fail(SD_ERR_INVALID_ARG, "sd_attend_combine: NULL input");
  if (shards < 1 || batch < 1 || hq < 1 || batch * hq * kD >= ((int64_t)1 << 40))
    return fail(SD_ERR_INVALID_ARG, "sd_attend_combine: bad shards, batch or hq");
  return launch_attend_combine(shards, batch * hq, outs, lses, out, lse, (cudaStream_t)stream);
}

int sd_set_fallback_paths(int on) {
  return g_fallback.exchange(on ? 1 : 0, std::memory_order_relaxed);
}

int sd_device_status(void* stream) {
  unsigned word = 0;
  if (int rc = scan_error_take((cudaStream_t)stream, &word)) return rc;
  if (word)
    return fail(SD_ERR_TIMEOUT,
                "sd_device_status: a bounded wait inside a bit-plane scan ran out since the last "
                "check; that scan stopped early and its scores are incomplete");
  return SD_OK;
}

int sd_debug_set_device_error(void* stream) {
  return scan_error_set(1u, (cudaStream_t)stream);
}

namespace {
// 16-byte words, grid-strided; several loads in flight per thread.
__global__ void __launch_bounds__(256) copy16_kernel(uint4* __restrict__ dst,
                                                     const uint4* __restrict__ src, int64_t n16) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n16; i += stride) dst[i] = src[i];
}
}  // namespace

int sd_copy(void* dst, const void* src, size_t bytes, void* stream) {
  if (bytes == 0) return SD_OK;
  if (!dst || !src) return fail(SD_ERR_INVALID_ARG, "sd_copy: NULL pointer");
  if (!aligned16(dst) || !aligned16(src) || bytes % 16)
    return fail(SD_ERR_INVALID_ARG, "sd_copy: pointers must be 16-byte aligned and bytes a "
                                    "multiple of 16");
  const int64_t n16 = (int64_t)(bytes / 16);
  const int64_t blocks = imin64((n16 + 255) / 256, (int64_t)device_sm_count() * 4);
  copy16_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
      static_cast<uint4*>(dst), static_cast<const uint4*>(src), n16);
  note_launches(1);
  return check_launch("sd_copy");
}

int sd_event_wait(void* event, int64_t timeout_us) {
  if (!event || timeout_us < 0) return fail(SD_ERR_INVALID_ARG, "sd_event_wait: bad argument");
  auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    cudaError_t e = cudaEventQuery((cudaEvent_t)event);
    if (e == cudaSuccess) return SD_OK;
    if (e != cudaErrorNotReady) {
      cudaGetLastError();
      return fail(SD_ERR_CUDA, "sd_event_wait: %s", cudaGetErrorString(e));
    }
    auto us = std::chrono::duration_cast<std::chrono::microseconds>(
                  std::chrono::steady_clock::now() - t0).count();
    if (us >= timeout_us)
      return fail(SD_ERR_TIMEOUT, "sd_event_wait: not complete after %lld us",
                  (long long)timeout_us);
    std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
}

}  // extern "C"
