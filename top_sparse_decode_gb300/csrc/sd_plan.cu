// Per-query read plan: Fathom: Per-Query Read Depth for Sparse Decoding over
// Offloaded KV Caches, paragraph "per-query reverse water-filling".
//
// The greedy (one bit at a time to the channel with the largest w_j * 4^-b_j,
// lowest j on ties) hands out exactly the first B pairs (j, b), b = 0..3, in the
// order (w_j * 4^-b descending, then 4j + b ascending): each channel's gains do
// not increase with b, so the greedy is a merge of per-channel sorted lists.
// The kernel finds the B-th largest pair value T with a 32-step bitwise search
// (one block-wide count per step), takes every pair above T and the first
// (in 4j + b order) of the pairs equal to T, and gives channel j the number of
// its pairs taken -- always a prefix b = 0, 1, ... of its four.
#include "sd_internal.cuh"

namespace sd {

// value with the largest order key such that at least `need` threads hold a
// key >= it (every thread of the block calls this)
__device__ __forceinline__ uint32_t block_kth_largest(uint32_t key, int need) {
  uint32_t T = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t cand = T | (1u << bit);
    if (__syncthreads_count(key >= cand) >= need) T = cand;
  }
  return T;
}

// exclusive count, in thread order, of threads with flag set (blockDim <= 1024)
__device__ __forceinline__ int block_rank(bool flag, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t m = __ballot_sync(0xFFFFFFFFu, flag);
  if (lane == 0) warp_tot[warp] = __popc(m);
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += warp_tot[w];
  return before + __popc(m & ((1u << lane) - 1u));
}

__global__ void __launch_bounds__(4 * kD)
plan_kernel(const uint16_t* __restrict__ q, const float* __restrict__ sigma2, int Hq, int Hkv,
            int G, int mode, int budget, uint8_t* __restrict__ plan) {
  const int bh = blockIdx.x, b = bh / Hkv, h = bh % Hkv;
  const int t = threadIdx.x;
  __shared__ float w[kD];
  __shared__ int warp_tot[32];
  uint8_t* out = plan + (int64_t)bh * kD;
  if (mode == SD_PLAN_FULL) {
    if (t < kD) out[t] = 4;
    return;
  }
  if (mode == SD_PLAN_FIXED || mode == SD_PLAN_TOPQ) {
    // the `budget` channels of largest sigma2 (FIXED) or largest query mass
    // u_j = sum_g q_gj^2 (TOPQ, fp32, g ascending, no fused multiply-add), lowest j
    // on ties, 4 bits each
    const bool live = t < kD;
    uint32_t key = 0u;
    if (live && mode == SD_PLAN_FIXED) {
      key = key_of_f32(sigma2[(int64_t)h * kD + t]);
    } else if (live) {
      float u = 0.0f;
      for (int g = 0; g < G; ++g) {
        const float x = bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + t]);
        u = __fadd_rn(u, __fmul_rn(x, x));
      }
      key = key_of_f32(u);
    }
    if (budget >= kD) {
      if (live) out[t] = 4;
      return;
    }
    if (budget == 0) {
      if (live) out[t] = 0;
      return;
    }
    // dead threads hold key 0, below every live key except key 0 itself; they sit
    // after every live thread in thread order, so ties resolve correctly
    const uint32_t T = block_kth_largest(key, budget);
    const int above = __syncthreads_count(live && key > T);
    const int r = block_rank(live && key == T, warp_tot);
    const bool take = live && (key > T || (key == T && r < budget - above));
    if (live) out[t] = take ? 4 : 0;
    return;
  }
  // gains in fp32, group sum in ascending g, no fused multiply-add
  if (t < kD) {
    float acc = 0.0f;
    for (int g = 0; g < G; ++g) {
      float x = bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + t]);
      acc = __fadd_rn(acc, __fmul_rn(x, x));
    }
    w[t] = __fmul_rn(acc, sigma2[(int64_t)h * kD + t]);
  }
  __syncthreads();
  // pair t = (j, bit): value w_j * 2^(-2 bit), one rounding like ldexpf
  const int j = t >> 2, bit = t & 3;
  const float scale4[4] = {1.0f, 0.25f, 0.0625f, 0.015625f};
  const uint32_t key = key_of_f32(__fmul_rn(w[j], scale4[bit]));
  int take;
  if (budget >= 4 * kD) {
    take = 1;
  } else if (budget == 0) {
    take = 0;
  } else {
    const uint32_t T = block_kth_largest(key, budget);
    const int above = __syncthreads_count(key > T);
    const int r = block_rank(key == T, warp_tot);
    take = key > T || (key == T && r < budget - above);
  }
  // the four pairs of channel j are adjacent lanes of one warp
  int cnt = take;
  cnt += __shfl_down_sync(0xFFFFFFFFu, cnt, 1);
  cnt += __shfl_down_sync(0xFFFFFFFFu, cnt, 2);
  if (bit == 0) out[j] = (uint8_t)cnt;
}

// SD_PLAN_SPLIT: the budget split across the KV heads of a sequence.  One CTA per
// sequence; the sequence's channels (h, j) are flattened to hj = h * kD + j and
// thread t owns channels t C .. t C + C - 1 with all four of their pairs, so the
// thread's pairs are contiguous in pair order 4 hj + b.  The (Hkv * budget)-th
// largest pair value T is found with the 32-step bitwise search (one block-wide
// count per step), every pair above T is taken and the pairs equal to T in pair
// order until the total is met; a channel's bits are its pairs taken (a prefix
// b = 0, 1, ... since its gains do not increase with b).  Same keys as plan_kernel's
// water-filling, so one head gives the same plan.
constexpr int kSplitThreads = 1024;
constexpr int kSplitChan = kSplitMaxHeads * kD / kSplitThreads;  // channels per thread, at most

// block-wide sum (every thread calls it; the result reaches every thread)
__device__ __forceinline__ int split_block_sum(int v, int* wsum, int* tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_add_sync(0xFFFFFFFFu, v);
  if (lane == 0) wsum[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int x = lane < (int)(blockDim.x >> 5) ? wsum[lane] : 0;
    x = __reduce_add_sync(0xFFFFFFFFu, x);
    if (lane == 0) *tot = x;
  }
  __syncthreads();
  const int r = *tot;
  __syncthreads();  // wsum and tot are rewritten by the next call
  return r;
}

__global__ void __launch_bounds__(kSplitThreads)
plan_split_kernel(const uint16_t* __restrict__ q, const float* __restrict__ sigma2, int Hq,
                  int Hkv, int G, int budget, uint8_t* __restrict__ plan) {
  __shared__ int wsum[32];
  __shared__ int tot;
  const int b = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int nch = Hkv * kD;
  const int C = (nch + kSplitThreads - 1) / kSplitThreads;  // <= kSplitChan
  const int c0 = t * C;
  uint8_t* out = plan + (int64_t)b * nch;
  const int64_t total = imin64((int64_t)Hkv * budget, 4 * (int64_t)nch);
  if (total == 0 || total == 4 * (int64_t)nch) {
    for (int c = 0; c < C; ++c)
      if (c0 + c < nch) out[c0 + c] = total ? 4 : 0;
    return;
  }
  uint32_t key[kSplitChan][4];
  const float scale4[4] = {1.0f, 0.25f, 0.0625f, 0.015625f};
#pragma unroll
  for (int c = 0; c < kSplitChan; ++c) {
    const int hj = c0 + c;
    float w = 0.0f;
    if (c < C && hj < nch) {
      const int h = hj / kD, j = hj % kD;
      float acc = 0.0f;  // fp32, group sum in ascending g, no fused multiply-add
      for (int g = 0; g < G; ++g) {
        const float x = bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + j]);
        acc = __fadd_rn(acc, __fmul_rn(x, x));
      }
      w = __fmul_rn(acc, sigma2[(int64_t)h * kD + j]);
    }
#pragma unroll
    for (int p = 0; p < 4; ++p)
      key[c][p] = (c < C && hj < nch) ? key_of_f32(__fmul_rn(w, scale4[p])) : 0u;
  }
  auto live = [&](int c) { return c < C && c0 + c < nch; };
  auto count = [&](auto pred) {
    int n = 0;
#pragma unroll
    for (int c = 0; c < kSplitChan; ++c)
#pragma unroll
      for (int p = 0; p < 4; ++p) n += live(c) && pred(key[c][p]);
    return split_block_sum(n, wsum, &tot);
  };
  // T: the largest value with at least `total` pairs >= it
  uint32_t T = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t cand = T | (1u << bit);
    if (count([&](uint32_t k) { return k >= cand; }) >= total) T = cand;
  }
  const int above = count([&](uint32_t k) { return k > T; });
  // pairs equal to T before this thread's, in pair order: a block exclusive scan
  int eq = 0;
#pragma unroll
  for (int c = 0; c < kSplitChan; ++c)
#pragma unroll
    for (int p = 0; p < 4; ++p) eq += live(c) && key[c][p] == T;
  int incl = eq;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int before = incl - eq;
  for (int w2 = 0; w2 < warp; ++w2) before += wsum[w2];
#pragma unroll
  for (int c = 0; c < kSplitChan; ++c) {
    if (!live(c)) continue;
    int taken = 0;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const uint32_t k = key[c][p];
      const bool e = k == T;
      if (k > T || (e && before < total - above)) ++taken;
      before += e;
    }
    out[c0 + c] = (uint8_t)taken;
  }
}

int launch_plan(const Dims& s, const uint16_t* q, const float* sigma2, int mode, int budget,
                uint8_t* plan, cudaStream_t st) {
  if (mode == SD_PLAN_SPLIT) {
    plan_split_kernel<<<s.B, kSplitThreads, 0, st>>>(q, sigma2, s.Hq, s.Hkv, s.G, budget, plan);
    note_launches(1);
    return check_launch("plan split");
  }
  plan_kernel<<<s.B * s.Hkv, 4 * kD, 0, st>>>(q, sigma2, s.Hq, s.Hkv, s.G, mode, budget, plan);
  note_launches(1);
  return check_launch("plan");
}

}  // namespace sd
