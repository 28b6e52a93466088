// GATHER-ATT: HashAttention: Semantic Sparsity for Faster Inference, 2.1
// (o_hat = sum_{i in I} e^{z_i} v_i / sum_{j in I} e^{z_j}, z_i = <q, k_i> / sqrt(d),
// with the denominator index fixed as on that page) and 2.5 (page size 1: the
// selected rows are read in place, by index, 256 contiguous bytes each).
//
// Split-n: CTA (chunk, row) handles up to kAtChunk selected tokens of one
// (sequence, KV head) for all G query heads of the group, so every K/V row is
// read once per group.  It writes (m, l, o~) partials; a combine kernel merges
// them with the usual rescaling e^{m_c - m}.
#include "sd_internal.cuh"

namespace sd {

constexpr int kAtChunk = 64;
constexpr int kAtPitch = kD + 8;  // bf16 pitch of staged rows (breaks bank alignment)

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static int64_t attend_chunks(int64_t max_count) { return (max_count + kAtChunk - 1) / kAtChunk; }

size_t attend_workspace_bytes(const Dims& s, int64_t max_count) {
  int64_t nch = attend_chunks(max_count);
  int64_t rows = (int64_t)s.B * s.Hkv;
  return align256(sizeof(float) * rows * nch * s.G * kD) + align256(sizeof(float2) * rows * nch * s.G);
}

template <int G>
__global__ void __launch_bounds__(128)
attend_partial_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ K,
                      const uint16_t* __restrict__ V, const int32_t* __restrict__ idx,
                      int64_t idx_stride, const int32_t* __restrict__ count, int Hq, int Hkv,
                      int64_t n, int64_t ncap, int max_count, float scale, int nchunks,
                      float* __restrict__ part_o, float2* __restrict__ part_ml) {
  __shared__ __align__(16) uint16_t Ks[kAtChunk][kAtPitch];
  __shared__ __align__(16) uint16_t Vs[kAtChunk][kAtPitch];
  __shared__ __align__(16) float qs[G][2][68];
  __shared__ float zs[G][kAtChunk];
  __shared__ float2 ml[G];
  __shared__ int valid[kAtChunk];

  const int64_t row = blockIdx.y;
  const int b = (int)(row / Hkv), h = (int)(row % Hkv);
  const int c = min(count[row], max_count);
  const int t0 = blockIdx.x * kAtChunk;
  if (t0 >= c) return;
  const int nt = min(kAtChunk, c - t0);
  const int t = threadIdx.x;

  for (int e = t; e < G * kD; e += 128) {
    int g = e / kD, j = e % kD;
    qs[g][j >> 6][j & 63] = bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + j]);
  }
  if (t < kAtChunk) {
    int ok = 0;
    if (t < nt) {
      int tok = idx[row * idx_stride + t0 + t];
      ok = (tok >= 0 && tok < n) ? tok + 1 : 0;  // out-of-range indices are skipped
    }
    valid[t] = ok;
  }
  __syncthreads();
  const uint16_t* Kr = K + row * ncap * kD;
  const uint16_t* Vr = V + row * ncap * kD;
  for (int e = t; e < nt * 16; e += 128) {
    int r = e >> 4, seg = e & 15;
    int ok = valid[r];
    if (ok) {
      int64_t tok = ok - 1;
      cp_async16(&Ks[r][seg * 8], Kr + tok * kD + seg * 8);
      cp_async16(&Vs[r][seg * 8], Vr + tok * kD + seg * 8);
    }
  }
  cp_async_wait_all();
  __syncthreads();

  // z for token tt, split over two threads by halves of d
  {
    const int tt = t >> 1, half = t & 1;
    float dot[G];
#pragma unroll
    for (int g = 0; g < G; ++g) dot[g] = 0.0f;
    if (tt < nt && valid[tt]) {
#pragma unroll
      for (int c8 = 0; c8 < 64; c8 += 8) {
        uint4 kv = *reinterpret_cast<const uint4*>(&Ks[tt][half * 64 + c8]);
        float kf[8] = {bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y),
                       bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w)};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float4 qa = *reinterpret_cast<const float4*>(&qs[g][half][c8]);
          float4 qb = *reinterpret_cast<const float4*>(&qs[g][half][c8 + 4]);
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
    for (int g = 0; g < G; ++g) dot[g] += __shfl_xor_sync(0xFFFFFFFFu, dot[g], 1);
    if (half == 0) {
      const bool ok = tt < nt && valid[tt];
#pragma unroll
      for (int g = 0; g < G; ++g) zs[g][tt] = ok ? dot[g] * scale : -INFINITY;
    }
  }
  __syncthreads();
  // per-head chunk max and exponentials
  {
    const int warp = t >> 5, lane = t & 31;
    for (int g = warp; g < G; g += 4) {
      float z0 = zs[g][lane], z1 = zs[g][lane + 32];
      float m = fmaxf(z0, z1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      float p0 = z0 == -INFINITY ? 0.0f : expf(z0 - m);
      float p1 = z1 == -INFINITY ? 0.0f : expf(z1 - m);
      zs[g][lane] = p0;
      zs[g][lane + 32] = p1;
      float l = p0 + p1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
      if (lane == 0) ml[g] = make_float2(m, l);
    }
  }
  __syncthreads();
  // o~ = sum_t p_t v_t, thread t owns column t
  float acc[G];
#pragma unroll
  for (int g = 0; g < G; ++g) acc[g] = 0.0f;
  for (int r = 0; r < nt; ++r) {
    if (!valid[r]) continue;
    float v = bf16_to_f32(Vs[r][t]);
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = fmaf(zs[g][r], v, acc[g]);
  }
  const int64_t pbase = (row * nchunks + blockIdx.x) * G;
#pragma unroll
  for (int g = 0; g < G; ++g) part_o[(pbase + g) * kD + t] = acc[g];
  if (t < G) part_ml[pbase + t] = ml[t];
}

template <int G>
__global__ void __launch_bounds__(128)
attend_combine_kernel(const int32_t* __restrict__ count, int Hq, int Hkv, int max_count,
                      int nchunks, const float* __restrict__ part_o,
                      const float2* __restrict__ part_ml, float* __restrict__ out,
                      float* __restrict__ lse) {
  const int64_t bq = blockIdx.x;  // b * Hq + query head
  const int b = (int)(bq / Hq), hq = (int)(bq % Hq);
  const int64_t row = (int64_t)b * Hkv + hq / G;
  const int g = hq % G;
  const int c = min(count[row], max_count);
  const int nch = (c + kAtChunk - 1) / kAtChunk;
  const int t = threadIdx.x;
  if (c <= 0) {
    out[bq * kD + t] = 0.0f;
    if (lse && t == 0) lse[bq] = -INFINITY;
    return;
  }
  float m = -INFINITY;
  for (int ch = 0; ch < nch; ++ch) m = fmaxf(m, part_ml[(row * nchunks + ch) * G + g].x);
  float l = 0.0f, o = 0.0f;
  for (int ch = 0; ch < nch; ++ch) {
    float2 p = part_ml[(row * nchunks + ch) * G + g];
    float w = p.x == -INFINITY ? 0.0f : expf(p.x - m);
    l = fmaf(p.y, w, l);
    o = fmaf(part_o[((row * nchunks + ch) * G + g) * kD + t], w, o);
  }
  out[bq * kD + t] = l > 0.0f ? o / l : 0.0f;
  if (lse && t == 0) lse[bq] = l > 0.0f ? m + logf(l) : -INFINITY;
}

template <int G>
static int attend_t(const Dims& s, const uint16_t* q, const uint16_t* K, const uint16_t* V,
                    const int32_t* idx, int64_t idx_stride, const int32_t* count,
                    int64_t max_count, float scale, float* out, float* lse, void* ws,
                    cudaStream_t st) {
  const int64_t rows = (int64_t)s.B * s.Hkv;
  const int nch = (int)attend_chunks(max_count);
  float* part_o = (float*)ws;
  float2* part_ml = (float2*)((uint8_t*)ws + align256(sizeof(float) * rows * nch * G * kD));
  if (nch > 0) {
    dim3 grid((unsigned)nch, (unsigned)rows);
    attend_partial_kernel<G><<<grid, 128, 0, st>>>(q, K, V, idx, idx_stride, count, s.Hq, s.Hkv,
                                                   s.n, s.ncap, (int)max_count, scale, nch,
                                                   part_o, part_ml);
    int rc = check_launch("attend_partial");
    if (rc) return rc;
  }
  attend_combine_kernel<G><<<(unsigned)(s.B * s.Hq), 128, 0, st>>>(
      count, s.Hq, s.Hkv, (int)max_count, nch, part_o, part_ml, out, lse);
  return check_launch("attend_combine");
}

int launch_gather_attend(const Dims& s, const uint16_t* q, const uint16_t* K, const uint16_t* V,
                         const int32_t* idx, int64_t idx_stride, const int32_t* count,
                         int64_t max_count, float scale, float* out, float* lse, void* ws,
                         size_t, cudaStream_t st) {
  switch (s.G) {
    case 1: return attend_t<1>(s, q, K, V, idx, idx_stride, count, max_count, scale, out, lse, ws, st);
    case 2: return attend_t<2>(s, q, K, V, idx, idx_stride, count, max_count, scale, out, lse, ws, st);
    case 4: return attend_t<4>(s, q, K, V, idx, idx_stride, count, max_count, scale, out, lse, ws, st);
    default: return attend_t<8>(s, q, K, V, idx, idx_stride, count, max_count, scale, out, lse, ws, st);
  }
}

}  // namespace sd
