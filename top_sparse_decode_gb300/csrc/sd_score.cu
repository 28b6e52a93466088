// SCORE kernels: one cheap score per cached key (or 16-token block) of every
// (sequence, KV head).
//
//  * Hamming     -- HashAttention: Semantic Sparsity for Faster Inference, 2.2:
//                   SCORE = -popcount(h_i XOR h_q), summed over the GQA group.
//  * bit planes  -- Fathom: Per-Query Read Depth ..., "bit planes per channel" and
//                   "per-query reverse water-filling": only the planned planes
//                   of each channel are read.
//  * Quest bound -- OasisKV: Scaling In-Decode KV Cache Beyond HBM ...,
//                   prerequisites: block importance from per-channel min/max.
#include <cuda_fp16.h>

#include "sd_internal.cuh"

namespace sd {

// =====================================================================================
// Hamming scan: 4 B per token per KV head, four tokens per thread (128-bit loads).
// =====================================================================================
template <int G>
__global__ void __launch_bounds__(256)
score_hamming_kernel(const uint32_t* __restrict__ sig, const uint32_t* __restrict__ qsig,
                     int Hq, int Hkv, int64_t n, int64_t ncap, bool vec,
                     int32_t* __restrict__ scores) {
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / Hkv), h = (int)(bh % Hkv);
  uint32_t qs[G];
#pragma unroll
  for (int g = 0; g < G; ++g) qs[g] = __ldg(qsig + (int64_t)b * Hq + h * G + g);
  const uint32_t* srow = sig + bh * ncap;
  int32_t* orow = scores + bh * n;
  const int64_t i0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i0 >= n) return;
  if (vec && i0 + 4 <= n) {
    uint4 s4 = __ldg(reinterpret_cast<const uint4*>(srow + i0));
    uint32_t sv[4] = {s4.x, s4.y, s4.z, s4.w};
    int r[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      int acc = 0;
#pragma unroll
      for (int g = 0; g < G; ++g) acc += __popc(sv[k] ^ qs[g]);
      r[k] = -acc;
    }
    *reinterpret_cast<int4*>(orow + i0) = make_int4(r[0], r[1], r[2], r[3]);
  } else {
    for (int64_t i = i0; i < imin64(i0 + 4, n); ++i) {
      uint32_t sv = __ldg(srow + i);
      int acc = 0;
#pragma unroll
      for (int g = 0; g < G; ++g) acc += __popc(sv ^ qs[g]);
      orow[i] = -acc;
    }
  }
}

template <int G>
static void hamming_t(const Dims& s, const uint32_t* sig, const uint32_t* qsig, int32_t* out,
                      cudaStream_t st) {
  bool vec = (s.n % 4 == 0) && (s.ncap % 4 == 0);
  dim3 grid((unsigned)((s.n + 1023) / 1024), (unsigned)(s.B * s.Hkv));
  score_hamming_kernel<G><<<grid, 256, 0, st>>>(sig, qsig, s.Hq, s.Hkv, s.n, s.ncap, vec, out);
}

int launch_score_hamming(const Dims& s, const uint32_t* sig, const uint32_t* qsig,
                         int32_t* scores, cudaStream_t st) {
  switch (s.G) {
    case 1: hamming_t<1>(s, sig, qsig, scores, st); break;
    case 2: hamming_t<2>(s, sig, qsig, scores, st); break;
    case 4: hamming_t<4>(s, sig, qsig, scores, st); break;
    default: hamming_t<8>(s, sig, qsig, scores, st); break;
  }
  return check_launch("score_hamming");
}

// =====================================================================================
// Bit-plane prefix scan.
//
// With q~_j = sum_g q_gj and W'_j = q~_j * s_j,blk, the score of token i is
//   sum_j W'_j * (prefix_ij + h(t_j) - 8)
//     = C_blk + sum over active planes (j, p < t_j) of (W'_j * 2^(3-p)) * bit_jpi,
//   C_blk = sum_j W'_j * (h(t_j) - 8),  h(t) = 2^(3-t) (t < 4), 0 (t = 4).
// So each active plane costs one bit test and one predicated add per token.
// A CTA scores 2048 tokens (64 words per plane, 32 scale blocks) of one
// (sequence, KV head); planes are staged 32 at a time in shared memory.
// Warp w owns words 8w..8w+7 and lane l owns bit l of each.
// =====================================================================================
constexpr int kPsTile = 2048;
constexpr int kPsWords = kPsTile / 32;   // 64
constexpr int kPsBlocks = kPsTile / 64;  // 32
constexpr int kPsChunk = 32;

template <int G>
__global__ void __launch_bounds__(256)
score_planes_kernel(const uint32_t* __restrict__ planes, const uint16_t* __restrict__ scales,
                    const uint8_t* __restrict__ plan, const uint16_t* __restrict__ q, int Hq,
                    int Hkv, int64_t n, int64_t ncap, float* __restrict__ scores) {
  __shared__ float qt[kD];
  __shared__ int tb[kD];
  __shared__ uint16_t act[4 * kD];
  __shared__ int nact_s;
  __shared__ float Cs[kPsBlocks];
  __shared__ __align__(16) uint32_t words[kPsChunk][kPsWords];
  __shared__ __align__(16) float Ws[kPsChunk][kPsBlocks];

  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / Hkv), h = (int)(bh % Hkv);
  const int64_t tok0 = (int64_t)blockIdx.x * kPsTile;
  const int nwv = (int)imin64(kPsWords, (n - tok0) / 32);  // valid words
  const int nbv = nwv / 2;                                        // valid blocks
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t wstride = ncap / 32, sstride = ncap / 64;
  const uint16_t* sc_bh = scales + bh * kD * sstride + tok0 / 64;

  if (threadIdx.x < kD) {
    const int j = threadIdx.x;
    float acc = 0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g)
      acc = __fadd_rn(acc, bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + j]));
    qt[j] = acc;
    tb[j] = min((int)plan[bh * kD + j], 4);  // a plan holds 0..4 bits per channel
  }
  __syncthreads();
  // active plane list (j ascending, p ascending) by a warp scan over channels
  if (warp == 0) {
    int c[4], tot = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) { c[k] = tb[lane * 4 + k]; tot += c[k]; }
    int incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += y;
    }
    int pos = incl - tot;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      for (int p = 0; p < c[k]; ++p) act[pos++] = (uint16_t)((lane * 4 + k) * 4 + p);
    if (lane == 31) nact_s = incl;
  }
  // per-block constants: warp w handles blocks 4w..4w+3
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int blk = warp * 4 + k;
    float part = 0.0f;
    if (blk < nbv) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = lane + 32 * jj;
        const int t = tb[j];
        if (t > 0) {
          float s = __half2float(__ushort_as_half(sc_bh[j * sstride + blk]));
          float wp = __fmul_rn(qt[j], s);
          float off = t < 4 ? (float)((1 << (3 - t)) - 8) : -8.0f;
          part = __fadd_rn(part, __fmul_rn(wp, off));
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part = __fadd_rn(part, __shfl_xor_sync(0xFFFFFFFFu, part, o));
    if (lane == 0) Cs[blk] = part;
  }
  __syncthreads();

  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
  const uint32_t lanemask = 1u << lane;
  const int nact = nact_s;
  const uint32_t* pl_bh = planes + bh * kD * 4 * wstride + tok0 / 32;

  for (int e0 = 0; e0 < nact; e0 += kPsChunk) {
    const int ne = min(kPsChunk, nact - e0);
    // stage the chunk's words (8-byte loads) and folded weights
    for (int x = threadIdx.x; x < ne * (kPsWords / 2); x += 256) {
      const int e = x / (kPsWords / 2), seg = x % (kPsWords / 2);
      const int ent = act[e0 + e];
      uint2 v = make_uint2(0u, 0u);
      if (seg * 2 < nwv)
        v = __ldg(reinterpret_cast<const uint2*>(pl_bh + (int64_t)ent * wstride) + seg);
      *reinterpret_cast<uint2*>(&words[e][seg * 2]) = v;
    }
    for (int x = threadIdx.x; x < ne * kPsBlocks; x += 256) {
      const int e = x / kPsBlocks, blk = x % kPsBlocks;
      const int ent = act[e0 + e];
      const int j = ent >> 2, p = ent & 3;
      float wv = 0.0f;
      if (blk < nbv) {
        float s = __half2float(__ushort_as_half(sc_bh[j * sstride + blk]));
        wv = __fmul_rn(__fmul_rn(qt[j], s), (float)(8 >> p));
      }
      Ws[e][blk] = wv;
    }
    __syncthreads();
#pragma unroll 2
    for (int e = 0; e < ne; ++e) {
      const uint4 wa = *reinterpret_cast<const uint4*>(&words[e][warp * 8]);
      const uint4 wb = *reinterpret_cast<const uint4*>(&words[e][warp * 8 + 4]);
      const float4 wt = *reinterpret_cast<const float4*>(&Ws[e][warp * 4]);
      if (wa.x & lanemask) acc[0] += wt.x;
      if (wa.y & lanemask) acc[1] += wt.x;
      if (wa.z & lanemask) acc[2] += wt.y;
      if (wa.w & lanemask) acc[3] += wt.y;
      if (wb.x & lanemask) acc[4] += wt.z;
      if (wb.y & lanemask) acc[5] += wt.z;
      if (wb.z & lanemask) acc[6] += wt.w;
      if (wb.w & lanemask) acc[7] += wt.w;
    }
    __syncthreads();
  }
  float* orow = scores + bh * n + tok0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int w = warp * 8 + k;
    if (w < nwv) orow[w * 32 + lane] = acc[k] + Cs[w >> 1];
  }
}

int launch_score_planes(const Dims& s, const uint32_t* planes, const uint16_t* scales,
                        const uint8_t* plan, const uint16_t* q, float* scores, cudaStream_t st) {
  dim3 grid((unsigned)((s.n + kPsTile - 1) / kPsTile), (unsigned)(s.B * s.Hkv));
  switch (s.G) {
    case 1: score_planes_kernel<1><<<grid, 256, 0, st>>>(planes, scales, plan, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
    case 2: score_planes_kernel<2><<<grid, 256, 0, st>>>(planes, scales, plan, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
    case 4: score_planes_kernel<4><<<grid, 256, 0, st>>>(planes, scales, plan, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
    default: score_planes_kernel<8><<<grid, 256, 0, st>>>(planes, scales, plan, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
  }
  return check_launch("score_planes");
}

// =====================================================================================
// Quest block bound.  max(q*mn, q*mx) = q*mx if q >= 0 else q*mn (mn <= mx), so
//   U = sum_j (P_j * max_j + N_j * min_j),  P_j = sum_g max(q_gj, 0),
//                                           N_j = sum_g min(q_gj, 0):
// two FMAs per channel per block instead of 4G operations.  A warp scores 4 blocks
// (512 B each), lane l owning channels 4l..4l+3; a CTA scores 32 blocks.
// =====================================================================================
template <int G>
__global__ void __launch_bounds__(256)
score_quest_kernel(const uint16_t* __restrict__ summ, const uint16_t* __restrict__ q, int Hq,
                   int Hkv, int64_t n, int64_t ncap, float* __restrict__ scores) {
  __shared__ float Ps[kD], Ns[kD];
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / Hkv), h = (int)(bh % Hkv);
  if (threadIdx.x < kD) {
    float p = 0.0f, m = 0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float x = bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + threadIdx.x]);
      p = __fadd_rn(p, fmaxf(x, 0.0f));
      m = __fadd_rn(m, fminf(x, 0.0f));
    }
    Ps[threadIdx.x] = p;
    Ns[threadIdx.x] = m;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nblk = (n + 15) / 16, nblk_cap = (ncap + 15) / 16;
  float P[4], N[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) { P[k] = Ps[lane * 4 + k]; N[k] = Ns[lane * 4 + k]; }
  const int64_t c0 = (int64_t)blockIdx.x * 32 + warp * 4;
  float acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    acc[k] = 0.0f;
    const int64_t c = c0 + k;
    if (c < nblk) {
      const uint16_t* base = summ + (bh * nblk_cap + c) * 2 * kD + lane * 4;
      uint2 lo = __ldg(reinterpret_cast<const uint2*>(base));
      uint2 hi = __ldg(reinterpret_cast<const uint2*>(base + kD));
      float a = 0.0f;
      a = __fmaf_rn(P[0], bf16_lo(hi.x), a);
      a = __fmaf_rn(N[0], bf16_lo(lo.x), a);
      a = __fmaf_rn(P[1], bf16_hi(hi.x), a);
      a = __fmaf_rn(N[1], bf16_hi(lo.x), a);
      a = __fmaf_rn(P[2], bf16_lo(hi.y), a);
      a = __fmaf_rn(N[2], bf16_lo(lo.y), a);
      a = __fmaf_rn(P[3], bf16_hi(hi.y), a);
      a = __fmaf_rn(N[3], bf16_hi(lo.y), a);
      acc[k] = a;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] += __shfl_xor_sync(0xFFFFFFFFu, acc[k], o);
  if (lane < 4 && c0 + lane < nblk) {
    float r = lane == 0 ? acc[0] : lane == 1 ? acc[1] : lane == 2 ? acc[2] : acc[3];
    scores[bh * nblk + c0 + lane] = r;
  }
}

int launch_score_quest(const Dims& s, const uint16_t* summ, const uint16_t* q, float* scores,
                       cudaStream_t st) {
  int64_t nblk = (s.n + 15) / 16;
  dim3 grid((unsigned)((nblk + 31) / 32), (unsigned)(s.B * s.Hkv));
  switch (s.G) {
    case 1: score_quest_kernel<1><<<grid, 256, 0, st>>>(summ, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
    case 2: score_quest_kernel<2><<<grid, 256, 0, st>>>(summ, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
    case 4: score_quest_kernel<4><<<grid, 256, 0, st>>>(summ, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
    default: score_quest_kernel<8><<<grid, 256, 0, st>>>(summ, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
  }
  return check_launch("score_quest");
}

}  // namespace sd
