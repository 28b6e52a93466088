// Per-query read plan: Fathom: Per-Query Read Depth for Sparse Decoding over
// Offloaded KV Caches, paragraph "per-query reverse water-filling".
//
// The greedy (one bit at a time to the channel with the largest w_j * 4^-b_j,
// lowest j on ties) hands out exactly the first B pairs (j, b), b = 0..3, in
// the order (w_j * 4^-b descending, j ascending, b ascending): each channel's
// gains do not increase with b, so the greedy is a merge of per-channel sorted
// lists.  The kernel therefore ranks all 4d pairs at once and gives channel j
// the number of its pairs whose rank is below B.
#include "sd_internal.cuh"

namespace sd {

__global__ void __launch_bounds__(4 * kD)
plan_kernel(const uint16_t* __restrict__ q, const float* __restrict__ sigma2, int Hq, int Hkv,
            int G, int mode, int budget, uint8_t* __restrict__ plan) {
  const int bh = blockIdx.x, b = bh / Hkv, h = bh % Hkv;
  const int t = threadIdx.x;
  __shared__ float w[kD];
  __shared__ float v[4 * kD];
  __shared__ int cnt[kD];
  if (mode == SD_PLAN_FULL) {
    if (t < kD) plan[(int64_t)bh * kD + t] = 4;
    return;
  }
  if (mode == SD_PLAN_FIXED) {
    if (t < kD) w[t] = sigma2[(int64_t)h * kD + t];
    __syncthreads();
    if (t < kD) {
      float mine = w[t];
      int rank = 0;
      for (int j = 0; j < kD; ++j) rank += (w[j] > mine) || (w[j] == mine && j < t);
      plan[(int64_t)bh * kD + t] = rank < budget ? 4 : 0;
    }
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
    cnt[t] = 0;
  }
  __syncthreads();
  // pair t = (j, bit): value w_j * 2^(-2 bit), one rounding like ldexpf
  const int j = t >> 2, bit = t & 3;
  const float scale4[4] = {1.0f, 0.25f, 0.0625f, 0.015625f};
  const float mine = __fmul_rn(w[j], scale4[bit]);
  v[t] = mine;
  __syncthreads();
  int rank = 0;
  for (int o = 0; o < 4 * kD; ++o) {
    float x = v[o];
    rank += (x > mine) || (x == mine && o < t);  // o < t  <=>  (j', b') before (j, b)
  }
  if (rank < budget) atomicAdd(&cnt[j], 1);
  __syncthreads();
  if (t < kD) plan[(int64_t)bh * kD + t] = (uint8_t)cnt[t];
}

int launch_plan(const Dims& s, const uint16_t* q, const float* sigma2, int mode, int budget,
                uint8_t* plan, cudaStream_t st) {
  plan_kernel<<<s.B * s.Hkv, 4 * kD, 0, st>>>(q, sigma2, s.Hq, s.Hkv, s.G, mode, budget, plan);
  return check_launch("plan");
}

}  // namespace sd
