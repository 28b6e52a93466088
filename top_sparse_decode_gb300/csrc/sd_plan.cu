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

int launch_plan(const Dims& s, const uint16_t* q, const float* sigma2, int mode, int budget,
                uint8_t* plan, cudaStream_t st) {
  plan_kernel<<<s.B * s.Hkv, 4 * kD, 0, st>>>(q, sigma2, s.Hq, s.Hkv, s.G, mode, budget, plan);
  note_launches(1);
  return check_launch("plan");
}

}  // namespace sd
