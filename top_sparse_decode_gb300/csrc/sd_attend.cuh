// Gather-attend building blocks shared by the attend kernels (sd_attend.cu) and the
// fused selection + attention kernel (sd_topk.cu): HashAttention: Semantic Sparsity
// for Faster Inference, 2.1 (o = sum_{i in I} e^{z_i} v_i / sum_{j in I} e^{z_j},
// z_i = <q, k_i> / sqrt(d)) and 2.5 (page size 1: selected rows read in place).
#pragma once

#include <cooperative_groups.h>

#include "sd_internal.cuh"

namespace sd {

constexpr int kAtChunk = 32;
constexpr int kAtPitch = kD + 8;  // bf16 pitch of staged rows (breaks bank alignment)
constexpr int kQPitch = 36;       // fp32 pitch of a quarter of q (conflict-free LDS.128)
constexpr int kAtCS = 16;         // CTAs per row in the cluster kernel

namespace cg = cooperative_groups;

__device__ __forceinline__ void at_cp_async16(void* smem, const void* gmem) {
  unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void at_cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

// One chunk's scores and exponentials for the G heads: stages the chunk's K and V
// rows, z = scale <q, k>, then per head the chunk max m_c, p = e^{z - m_c} into zt
// and (m_c, l_c) into ml.
template <int G>
struct AtChunk {
  uint16_t Ks[kAtChunk][kAtPitch];
  uint16_t Vs[kAtChunk][kAtPitch];
  float qs[G][4][kQPitch];
  __align__(16) float zt[kAtChunk][G];  // token-major: one row holds every head's value
  float2 ml[G];
  int valid[kAtChunk];
};

// Run by 128 threads (t = threadIdx.x < 128); bar() synchronises exactly them.
template <int G, class Bar>
__device__ __forceinline__ void at_chunk(AtChunk<G>& A, const uint16_t* __restrict__ Kr,
                                         const uint16_t* __restrict__ Vr, int nt, float scale,
                                         Bar bar) {
  const int t = threadIdx.x;
  for (int e = t; e < nt * 16; e += 128) {
    const int r = e >> 4, seg = e & 15;
    const int ok = A.valid[r];
    if (ok) {
      const int64_t tok = ok - 1;
      at_cp_async16(&A.Ks[r][seg * 8], Kr + tok * kD + seg * 8);
      at_cp_async16(&A.Vs[r][seg * 8], Vr + tok * kD + seg * 8);
    } else {  // a skipped row's V is zero, so the P V fold needs no test (its p is 0)
      *reinterpret_cast<uint4*>(&A.Vs[r][seg * 8]) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  at_cp_async_wait_all();
  bar();
  {  // z for token tt, split over four threads by quarters of d
    const int tt = t >> 2, qq = t & 3;
    float dot[G];
#pragma unroll
    for (int g = 0; g < G; ++g) dot[g] = 0.0f;
    const bool ok = tt < nt && A.valid[tt];
    if (ok) {
#pragma unroll
      for (int c8 = 0; c8 < 32; c8 += 8) {
        const uint4 kv = *reinterpret_cast<const uint4*>(&A.Ks[tt][qq * 32 + c8]);
        const float kf[8] = {bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y),
                             bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w)};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 qa = *reinterpret_cast<const float4*>(&A.qs[g][qq][c8]);
          const float4 qb = *reinterpret_cast<const float4*>(&A.qs[g][qq][c8 + 4]);
          dot[g] = fmaf(qa.x, kf[0], dot[g]);
          dot[g] = fmaf(qa.y, kf[1], dot[g]);
          dot[g] = fmaf(qa.z, kf[2], dot[g]);
          dot[g] = fmaf(qa.w, kf[3], dot[g]);
          dot[g] = fmaf(qb.x, kf[4], dot[g]);
          dot[g] = fmaf(qb.y, kf[5], dot[g]);
          dot[g] = fmaf(qb.z, kf[6], dot[g]);
          dot[g] = fmaf(qb.w, kf[7], dot[g]);
        }
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      dot[g] += __shfl_xor_sync(0xFFFFFFFFu, dot[g], 1);
      dot[g] += __shfl_xor_sync(0xFFFFFFFFu, dot[g], 2);
    }
    if (qq == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) A.zt[tt][g] = ok ? dot[g] * scale : -INFINITY;
    }
  }
  bar();
  {  // per-head chunk max and exponentials: warp w handles heads w, w + 4
    const int warp = t >> 5, lane = t & 31;
    for (int g = warp; g < G; g += 4) {
      const float z = A.zt[lane][g];
      float m = z;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      const float p = z == -INFINITY ? 0.0f : expf(z - m);
      A.zt[lane][g] = p;
      float l = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
      if (lane == 0) A.ml[g] = make_float2(m, l);
    }
  }
  bar();
}

template <int G>
struct AtState {
  float o[G][kD];  // this CTA's o~ over its chunks
  float2 ml[G];    // its (m, l)
};

// One (sequence, KV head) row of a kAtCS-CTA cluster: run by threads 0..127 of every
// CTA of the cluster (bar() synchronises them); the row's other threads, if any,
// call cl.sync() twice instead (the body's two cluster barriers).
template <int G, class Bar>
__device__ __forceinline__ void at_cluster_row(AtChunk<G>& A, AtState<G>& St, int64_t row,
                                               const uint16_t* __restrict__ q,
                                               const uint16_t* __restrict__ K,
                                               const uint16_t* __restrict__ V,
                                               const int32_t* __restrict__ idx,
                                               int64_t idx_stride,
                                               const int32_t* __restrict__ count, int Hq,
                                               int Hkv, int64_t n, int64_t ncap, int max_count,
                                               float scale, float* __restrict__ out,
                                               float* __restrict__ lse, Bar bar) {
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int b = (int)(row / Hkv), h = (int)(row % Hkv);
  const int t = threadIdx.x;
  // the first chunk's indices are loaded before the count arrives (t0 < max_count
  // <= idx_stride keeps them in bounds)
  int tok_first = -1;
  if (t < kAtChunk && rank * kAtChunk + t < max_count)
    tok_first = __ldcg(idx + row * idx_stride + rank * kAtChunk + t);
  for (int e = t; e < G * kD; e += 128) {
    const int g = e / kD, j = e % kD;
    A.qs[g][j >> 5][j & 31] = bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + j]);
  }
  const int c = min(__ldcg(count + row), max_count);
  const uint16_t* Kr = K + row * ncap * kD;
  const uint16_t* Vr = V + row * ncap * kD;
  float mrun[G], lrun[G], orun[G];
#pragma unroll
  for (int g = 0; g < G; ++g) { mrun[g] = -INFINITY; lrun[g] = 0.0f; orun[g] = 0.0f; }
  for (int ch = rank; ch * kAtChunk < c; ch += kAtCS) {
    const int t0 = ch * kAtChunk, nt = min(kAtChunk, c - t0);
    if (t < kAtChunk) {
      int ok = 0;
      if (t < nt) {
        const int tok = ch == rank ? tok_first : __ldcg(idx + row * idx_stride + t0 + t);
        ok = (tok >= 0 && tok < n) ? tok + 1 : 0;  // out-of-range indices are skipped
      }
      A.valid[t] = ok;
    }
    bar();
    at_chunk<G>(A, Kr, Vr, nt, scale, bar);
    // fold the chunk into the running state; thread t owns column t (the heads'
    // sums are independent chains, so tokens go outermost)
    float pv[G];
#pragma unroll
    for (int g = 0; g < G; ++g) pv[g] = 0.0f;
#pragma unroll 8
    for (int r = 0; r < nt; ++r) {  // skipped rows hold p = 0 and V = 0
      const float v = bf16_to_f32(A.Vs[r][t]);
      if constexpr (G % 4 == 0) {
#pragma unroll
        for (int g4 = 0; g4 < G; g4 += 4) {
          const float4 z4 = *reinterpret_cast<const float4*>(&A.zt[r][g4]);
          pv[g4] = fmaf(z4.x, v, pv[g4]);
          pv[g4 + 1] = fmaf(z4.y, v, pv[g4 + 1]);
          pv[g4 + 2] = fmaf(z4.z, v, pv[g4 + 2]);
          pv[g4 + 3] = fmaf(z4.w, v, pv[g4 + 3]);
        }
      } else {
#pragma unroll
        for (int g = 0; g < G; ++g) pv[g] = fmaf(A.zt[r][g], v, pv[g]);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float2 mlc = A.ml[g];
      const float m = fmaxf(mrun[g], mlc.x);
      const float wr = mrun[g] == -INFINITY ? 0.0f : expf(mrun[g] - m);
      const float wc = mlc.x == -INFINITY ? 0.0f : expf(mlc.x - m);
      orun[g] = orun[g] * wr + pv[g] * wc;
      lrun[g] = lrun[g] * wr + mlc.y * wc;
      mrun[g] = m;
    }
    bar();  // the chunk buffers are reused
  }
#pragma unroll
  for (int g = 0; g < G; ++g) St.o[g][t] = orun[g];
  if (t == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) St.ml[g] = make_float2(mrun[g], lrun[g]);
  }
  cl.sync();
  // merge: CTA r combines outputs r * 8G .. r * 8G + 8G - 1 (head e / 128, column
  // e % 128) over every CTA's state, ranks ascending; all loads in flight together
  if (t < 8 * G) {
    const int e = rank * 8 * G + t, g = e / kD, col = e % kD;
    float2 mlr[kAtCS];
    float orr[kAtCS];
#pragma unroll
    for (int r = 0; r < kAtCS; ++r) {
      const AtState<G>* R = cl.map_shared_rank(&St, r);
      mlr[r] = R->ml[g];
      orr[r] = R->o[g][col];
    }
    float m = -INFINITY;
#pragma unroll
    for (int r = 0; r < kAtCS; ++r) m = fmaxf(m, mlr[r].x);
    float l = 0.0f, o = 0.0f;
#pragma unroll
    for (int r = 0; r < kAtCS; ++r) {
      const float w = mlr[r].x == -INFINITY ? 0.0f : expf(mlr[r].x - m);
      l = fmaf(mlr[r].y, w, l);
      o = fmaf(orr[r], w, o);
    }
    const int64_t bq = (int64_t)b * Hq + h * G + g;
    out[bq * kD + col] = l > 0.0f ? o / l : 0.0f;  // an empty set gives o = 0
    if (lse && col == 0) lse[bq] = l > 0.0f ? m + logf(l) : -INFINITY;
  }
  cl.sync();  // every CTA's state stays alive until the others have read it
}

}  // namespace sd
