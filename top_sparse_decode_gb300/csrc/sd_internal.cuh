// Internal declarations shared by libsd's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <atomic>

#include "sd.h"

namespace sd {

struct PsCand;    // sd_planes.cuh
struct PsPlanIn;  // sd_planes.cuh

constexpr int kD = 128;          // head dimension supported by this build
constexpr int kMaxTopK = 4096;   // largest retrieval budget of sd_topk
constexpr int kSmallRow = 8192;  // rows up to this many units are selected by one CTA

// ---- error reporting -------------------------------------------------------------
void set_error(const char* fmt, ...);
int fail(int code, const char* fmt, ...);
int check_launch(const char* what);
// counts kernel launches made by the library (sd_launch_count)
void note_launches(int k);
// Raises a kernel's dynamic shared-memory limit to `bytes`, once per (device,
// kernel): later calls, including those made while a stream is being captured
// into a CUDA graph, issue no CUDA call.
int set_smem_limit(const void* kernel, size_t bytes, const char* what);

// True while sd_set_fallback_paths(1) is in force: the gather-attend, the top-k
// kernels and the bit-plane scan take the kernels they use on GPUs where their
// thread-block clusters cannot be co-resident or bulk copies do not apply (the
// split-n attention with its workspace partials, the sample/filter/finish top-k,
// the one-CTA word-maxima top-k, the cp.async scan).  Off by default.
bool fallback_forced();

// A per-device value computed once by `compute` (for example an occupancy query)
// and cached; concurrent first calls may both compute it, and every reader sees
// either "unknown" or the whole value.  Returns 0 when the current device cannot
// be read.
constexpr int kMaxDev = 64;
template <class F>
inline int per_device_cached(std::atomic<int> (&tab)[kMaxDev], F compute) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return 0;
  }
  int v = tab[dev].load(std::memory_order_acquire);  // value + 1; 0 = not yet known
  if (v == 0) {
    v = compute() + 1;
    tab[dev].store(v, std::memory_order_release);
  }
  return v - 1;
}

// The scan's device error word (sd_scan_tma.cu): read-and-clear, and a host-side
// setter for testing the report without making a wait run out.
int scan_error_take(cudaStream_t st, unsigned* word);
int scan_error_set(unsigned word, cudaStream_t st);
// The current device's SM count (cached per device; 152 if it cannot be read).
int device_sm_count();

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t imax64(int64_t a, int64_t b) { return a > b ? a : b; }

// ---- number formats ----------------------------------------------------------------
__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}
// low / high bf16 of a packed pair
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// order-preserving 32-bit keys: larger score -> larger key
__device__ __forceinline__ uint32_t key_of_f32(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0.0 ranks with +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint32_t key_of_i32(int32_t x) { return (uint32_t)x ^ 0x80000000u; }
// max that propagates NaN (PTX max.NaN), so one compare screens several scores
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// ---- launchers (each returns SD_OK or an SD_ERR_*) ---------------------------------
struct Dims {
  int B, Hq, Hkv, G;
  int64_t n, ncap;
};

// Index builds over tokens [0, s.n); with t0 > 0 only what tokens [t0, s.n) touch is
// rewritten (their signatures, the 16- or 64-token blocks from the one holding t0).
int launch_sig_build(const Dims& s, const uint16_t* K, const sd_encoder& enc, uint32_t* sig,
                     cudaStream_t st, int64_t t0 = 0);
int launch_encode_query(const Dims& s, const uint16_t* q, const sd_encoder& enc, uint32_t* qsig,
                        cudaStream_t st);
int launch_plane_build(const Dims& s, const uint16_t* K, uint32_t* planes, uint16_t* scales,
                       cudaStream_t st, int64_t t0 = 0);
int launch_minmax_build(const Dims& s, const uint16_t* K, uint16_t* summ, cudaStream_t st,
                        int64_t t0 = 0);
constexpr int kLmBlock = 8;  // tokens per landmark block
int launch_landmark_build(const Dims& s, const uint16_t* K, uint16_t* L, cudaStream_t st,
                          int64_t t0 = 0);
int launch_score_landmark(const Dims& s, const uint16_t* L, const uint16_t* q, float* scores,
                          cudaStream_t st);
constexpr int kSplitMaxHeads = 64;  // KV heads one SD_PLAN_SPLIT plan may couple
int launch_plan(const Dims& s, const uint16_t* q, const float* sigma2, int mode, int budget,
                uint8_t* plan, cudaStream_t st);

// Delta selection against a resident set and the gather of admitted units
// (sd_resident.cu).
constexpr int kDsMaxUnits = 8192;  // predicted units per row
constexpr int kDsMaxSlots = 4096;  // resident slots per row
int launch_delta_select(int64_t rows, int64_t nu, int64_t n_tokens, int block, int sink,
                        int local, int sel_k, const float* scores, const int32_t* idx, int64_t idx_stride,
                        const int32_t* count, int C, int step, int R, int32_t* slot_unit,
                        int32_t* slot_last, int32_t* unit_slot, int32_t* plan_slot,
                        int32_t* plan_unit, int32_t* plan_evict, int32_t* plan_count,
                        int32_t* pool_idx, int64_t pool_stride, int32_t* pool_count,
                        cudaStream_t st);
int launch_resident_gather(const Dims& s, int block, const uint16_t* K, const uint16_t* V,
                           const int32_t* plan_slot, const int32_t* plan_unit,
                           const int32_t* plan_count, int C, int R, uint16_t* Kp, uint16_t* Vp,
                           cudaStream_t st);
int launch_score_hamming(const Dims& s, const uint32_t* sig, const uint32_t* qsig,
                         int32_t* scores, cudaStream_t st);
// (cand: the fused scan + top-k's candidate marks, or null; plan_in: compute the
// read plan in the scan instead of reading `plan`, or null)
bool planes_aligned(const Dims& s, const void* planes, const void* scales);
int launch_score_planes(const Dims& s, const uint32_t* planes, const uint16_t* scales,
                        const uint8_t* plan, const uint16_t* q, float* scores, cudaStream_t st,
                        const PsCand* cand = nullptr, const PsPlanIn* plan_in = nullptr,
                        float* wmax = nullptr);
int launch_score_planes_tma(const Dims& s, const uint32_t* planes, const uint16_t* scales,
                            const uint8_t* plan, const uint16_t* q, float* scores,
                            const PsCand* cand, const PsPlanIn* plan_in, float* wmax, int sms,
                            cudaStream_t st);
// Direct-streaming bit-plane scan (sd_scan_direct.cu): any n, n_cap % 64 == 0;
// returns 1 (not launched) when plane offsets exceed 32 bits.
int launch_score_planes_direct(const Dims& s, const uint32_t* planes, const uint16_t* scales,
                               const uint8_t* plan, const uint16_t* q, float* scores,
                               const PsPlanIn* plan_in, float* wmax, int sms, cudaStream_t st);
int launch_score_quest(const Dims& s, const uint16_t* summ, const uint16_t* q, float* scores,
                       cudaStream_t st);
size_t topk_workspace_bytes(int64_t rows, int64_t n_units, const sd_select& sel);
// fused bit-plane scan + top-k (sd_score_topk)
size_t score_topk_workspace_bytes(int64_t rows, int64_t n, const sd_select& sel);
int launch_score_topk(const Dims& s, const uint32_t* planes, const uint16_t* scales,
                      const uint8_t* plan, const uint16_t* q, const sd_select& sel, float* scores,
                      int32_t* idx, int64_t idx_stride, int32_t* count, void* ws,
                      cudaStream_t st);
int launch_topk(int score_type, const void* scores, int64_t rows, int64_t n_units,
                int64_t n_tokens, const sd_select& sel, int32_t* idx, int64_t idx_stride,
                int32_t* count, void* ws, size_t ws_bytes, cudaStream_t st);
int launch_topk_wmax(const float* scores, const float* wmax, int64_t rows, int64_t n,
                     const sd_select& sel, int32_t* idx, int64_t idx_stride, int32_t* count,
                     void* ws, size_t ws_bytes, cudaStream_t st);
size_t attend_workspace_bytes(const Dims& s, int64_t max_count);
// The streaming gather-attend (sd_attend_stream.cu) over the split-n workspace's
// ticket and partial slots; returns 1 (not launched) where it does not apply.
int launch_attend_stream(const Dims& s, const uint16_t* q, const uint16_t* K, const uint16_t* V,
                         const int32_t* idx, int64_t idx_stride, const int32_t* count,
                         int64_t max_count, float scale, float* out, float* lse,
                         uint32_t* ticket, float* part_o, float2* part_ml, int slots_avail,
                         cudaStream_t st);
int launch_gather_attend(const Dims& s, const uint16_t* q, const uint16_t* K, const uint16_t* V,
                         const int32_t* idx, int64_t idx_stride, const int32_t* count,
                         int64_t max_count, float scale, float* out, float* lse, void* ws,
                         size_t ws_bytes, cudaStream_t st);
size_t hamming_topk_workspace_bytes(const Dims& s, const sd_select& sel);
bool hamming_topk_supported(const Dims& s, const sd_select& sel);
int launch_hamming_topk(const Dims& s, const uint32_t* sig, const uint32_t* qsig,
                        const sd_select& sel, int32_t* idx, int64_t idx_stride, int32_t* count,
                        void* ws, cudaStream_t st);
size_t select_attend_workspace_bytes(const Dims& s, const sd_select& sel, int64_t max_count);
int launch_select_attend(const Dims& s, const float* scores, const float* wmax,
                         const sd_select& sel, const uint16_t* q, const uint16_t* K,
                         const uint16_t* V, float scale, int32_t* idx, int64_t idx_stride,
                         int32_t* count, int64_t max_count, float* out, float* lse, void* ws,
                         size_t ws_bytes, cudaStream_t st);
// One sequence split by tokens across devices (sd_shard.cu).
constexpr int kMergeMaxCand = 8192;  // shards * k one merge may hold
int launch_shard_candidates(const float* scores, int64_t rows, int64_t n_s, const int32_t* idx,
                            int64_t idx_stride, const int32_t* count, int sink_s, int local_s,
                            int64_t offset, int k, float* cs, int32_t* ci, int32_t* cc,
                            cudaStream_t st);
int launch_topk_merge(int64_t rows, int S, int k, const float* cs, const int32_t* ci,
                      const int32_t* cc, int32_t* out, int64_t out_stride, int32_t* ocount,
                      cudaStream_t st);
int launch_shard_select(int64_t rows, const int32_t* sel, int64_t sel_stride,
                        const int32_t* scount, int64_t a, int64_t n_s, int sink_s, int local_s,
                        int32_t* out, int64_t out_stride, int32_t* ocount, cudaStream_t st);
int launch_attend_combine(int S, int64_t BH, const float* outs, const float* lses, float* out,
                          float* lse, cudaStream_t st);
int launch_offload_gather(const Dims& s, const uint32_t* host_planes, const uint16_t* host_scales,
                          const uint8_t* plan, uint32_t* dev_planes, uint16_t* dev_scales,
                          cudaStream_t st);

}  // namespace sd
