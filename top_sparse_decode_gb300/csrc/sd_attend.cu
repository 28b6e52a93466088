// GATHER-ATT: HashAttention: Semantic Sparsity for Faster Inference, 2.1
// (o_hat = sum_{i in I} e^{z_i} v_i / sum_{j in I} e^{z_j}, z_i = <q, k_i> / sqrt(d),
// with the denominator index fixed as on that page) and 2.5 (page size 1: the
// selected rows are read in place, by index, 256 contiguous bytes each).
//
// Many long rows (a batch of sequences) go to the streaming kernel
// (sd_attend_stream.cu), which keeps every SM's share of the rows in flight from HBM.
// Otherwise, split-n: a CTA handles chunks of kAtChunk selected tokens of one (sequence, KV
// head) for all G query heads of the group, so every K/V row is read once per
// group.  Each row is one thread-block cluster of kAtCS CTAs: CTA r takes chunks
// r, r + kAtCS, ... and keeps a running (m, l, o~) over them; then every CTA merges
// its sixteenth of the outputs over all CTAs' states, in rank order, through
// distributed shared memory with the usual rescaling e^{m_r - m}.  (Where that cluster cannot run, CTAs write (m, l, o~)
// partials per chunk and the last CTA of the row, by a ticket, merges them.)
#include <cooperative_groups.h>

#include "sd_attend.cuh"

namespace sd {

constexpr int kMergeMax = 256;    // chunks whose merge weights are staged at once

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static int64_t attend_chunks(int64_t max_count) { return (max_count + kAtChunk - 1) / kAtChunk; }

struct AttWs {
  uint32_t* ticket;  // [rows], zeroed at the start of every call
  float* part_o;     // [rows][nch][G][kD]
  float2* part_ml;   // [rows][nch][G]
};

static AttWs carve_att(void* ws, int64_t rows, int64_t nch, int G) {
  uint8_t* p = (uint8_t*)ws;
  AttWs w;
  w.ticket = (uint32_t*)p;
  p += align256(sizeof(uint32_t) * rows);
  w.part_o = (float*)p;
  p += align256(sizeof(float) * rows * nch * G * kD);
  w.part_ml = (float2*)p;
  return w;
}

size_t attend_workspace_bytes(const Dims& s, int64_t max_count) {
  int64_t nch = attend_chunks(max_count);
  int64_t rows = (int64_t)s.B * s.Hkv;
  return align256(sizeof(uint32_t) * rows) + align256(sizeof(float) * rows * nch * s.G * kD) +
         align256(sizeof(float2) * rows * nch * s.G);
}

template <int G>
__global__ void __launch_bounds__(128)
attend_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ K,
              const uint16_t* __restrict__ V, const int32_t* __restrict__ idx,
              int64_t idx_stride, const int32_t* __restrict__ count, int Hq, int Hkv, int64_t n,
              int64_t ncap, int max_count, float scale, int nchunks, AttWs ws,
              float* __restrict__ out, float* __restrict__ lse) {
  __shared__ __align__(16) uint16_t Ks[kAtChunk][kAtPitch];
  __shared__ __align__(16) uint16_t Vs[kAtChunk][kAtPitch];
  __shared__ __align__(16) float qs[G][4][kQPitch];
  __shared__ float zs[G][kAtChunk];
  __shared__ float2 ml[G];
  __shared__ int valid[kAtChunk];
  __shared__ bool last;

  const int64_t row = blockIdx.y;
  const int b = (int)(row / Hkv), h = (int)(row % Hkv);
  const int c = min(count[row], max_count);
  const int t = threadIdx.x;
  const int t0 = blockIdx.x * kAtChunk;
  if (c <= 0) {  // empty set: o = 0, lse = -inf, written once per row
    if (blockIdx.x == 0) {
      for (int g = 0; g < G; ++g) {
        const int64_t bq = (int64_t)b * Hq + h * G + g;
        out[bq * kD + t] = 0.0f;
        if (lse && t == 0) lse[bq] = -INFINITY;
      }
    }
    return;
  }
  if (t0 >= c) return;
  const int nt = min(kAtChunk, c - t0);
  const int nch_row = (c + kAtChunk - 1) / kAtChunk;

  for (int e = t; e < G * kD; e += 128) {
    const int g = e / kD, j = e % kD;
    qs[g][j >> 5][j & 31] = bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + j]);
  }
  if (t < kAtChunk) {
    int ok = 0;
    if (t < nt) {
      const int tok = idx[row * idx_stride + t0 + t];
      ok = (tok >= 0 && tok < n) ? tok + 1 : 0;  // out-of-range indices are skipped
    }
    valid[t] = ok;
  }
  __syncthreads();
  const uint16_t* Kr = K + row * ncap * kD;
  const uint16_t* Vr = V + row * ncap * kD;
  for (int e = t; e < nt * 16; e += 128) {
    const int r = e >> 4, seg = e & 15;
    const int ok = valid[r];
    if (ok) {
      const int64_t tok = ok - 1;
      at_cp_async16(&Ks[r][seg * 8], Kr + tok * kD + seg * 8);
      at_cp_async16(&Vs[r][seg * 8], Vr + tok * kD + seg * 8);
    }
  }
  at_cp_async_wait_all();
  __syncthreads();

  // z for token tt, split over four threads by quarters of d
  {
    const int tt = t >> 2, qq = t & 3;
    float dot[G];
#pragma unroll
    for (int g = 0; g < G; ++g) dot[g] = 0.0f;
    const bool ok = tt < nt && valid[tt];
    if (ok) {
#pragma unroll
      for (int c8 = 0; c8 < 32; c8 += 8) {
        const uint4 kv = *reinterpret_cast<const uint4*>(&Ks[tt][qq * 32 + c8]);
        const float kf[8] = {bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y),
                             bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w)};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 qa = *reinterpret_cast<const float4*>(&qs[g][qq][c8]);
          const float4 qb = *reinterpret_cast<const float4*>(&qs[g][qq][c8 + 4]);
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
      for (int g = 0; g < G; ++g) zs[g][tt] = ok ? dot[g] * scale : -INFINITY;
    }
  }
  __syncthreads();
  // per-head chunk max and exponentials: warp w handles heads w, w + 4
  {
    const int warp = t >> 5, lane = t & 31;
    for (int g = warp; g < G; g += 4) {
      const float z = zs[g][lane];
      float m = z;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      const float p = z == -INFINITY ? 0.0f : expf(z - m);
      zs[g][lane] = p;
      float l = p;
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
    if (!valid[r]) continue;  // skipped rows were not staged
    const float v = bf16_to_f32(Vs[r][t]);
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = fmaf(zs[g][r], v, acc[g]);
  }
  const int64_t pbase = (row * nchunks + blockIdx.x) * G;
#pragma unroll
  for (int g = 0; g < G; ++g) ws.part_o[(pbase + g) * kD + t] = acc[g];
  if (t < G) ws.part_ml[pbase + t] = ml[t];

  // the last CTA of the row merges the partials in chunk order
  __threadfence();
  __syncthreads();
  if (t == 0) last = atomicAdd(&ws.ticket[row], 1u) == (uint32_t)(nch_row - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  // merge: the row max m, then per window of up to kMergeMax chunks their weights
  // e^{m_c - m} staged in shared memory; o accumulates with 8 loads in flight
  __shared__ float wts[G][kMergeMax];
  __shared__ float lsum[G], mrow[G];
  const int64_t rbase = row * nchunks * G;
  const int warp = t >> 5, lane = t & 31;
  for (int g = warp; g < G; g += 4) {
    float m = -INFINITY;
    for (int ch = lane; ch < nch_row; ch += 32) m = fmaxf(m, __ldcg(&ws.part_ml[rbase + ch * G + g].x));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) { mrow[g] = m; lsum[g] = 0.0f; }
  }
  float o_acc[G];
#pragma unroll
  for (int g = 0; g < G; ++g) o_acc[g] = 0.0f;
  for (int c0 = 0; c0 < nch_row; c0 += kMergeMax) {
    const int nw = min(kMergeMax, nch_row - c0);
    __syncthreads();  // mrow ready; the previous window's weights consumed
    for (int g = warp; g < G; g += 4) {
      const float m = mrow[g];
      float l = 0.0f;
      for (int i = lane; i < nw; i += 32) {
        const float2 p = __ldcg(&ws.part_ml[rbase + (c0 + i) * G + g]);
        const float wgt = p.x == -INFINITY ? 0.0f : expf(p.x - m);
        wts[g][i] = wgt;
        l = fmaf(p.y, wgt, l);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
      if (lane == 0) lsum[g] += l;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float o = o_acc[g];
      int i = 0;
      for (; i + 8 <= nw; i += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldcg(&ws.part_o[(rbase + (c0 + i + u) * G + g) * kD + t]);
#pragma unroll
        for (int u = 0; u < 8; ++u) o = fmaf(v[u], wts[g][i + u], o);
      }
      for (; i < nw; ++i) o = fmaf(__ldcg(&ws.part_o[(rbase + (c0 + i) * G + g) * kD + t]), wts[g][i], o);
      o_acc[g] = o;
    }
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float l = lsum[g];
    const int64_t bq = (int64_t)b * Hq + h * G + g;
    out[bq * kD + t] = l > 0.0f ? o_acc[g] / l : 0.0f;
    if (lse && t == 0) lse[bq] = l > 0.0f ? mrow[g] + logf(l) : -INFINITY;
  }
}

template <int G>
__global__ void __launch_bounds__(128)
attend_cluster_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ K,
                      const uint16_t* __restrict__ V, const int32_t* __restrict__ idx,
                      int64_t idx_stride, const int32_t* __restrict__ count, int Hq, int Hkv,
                      int64_t n, int64_t ncap, int max_count, float scale,
                      float* __restrict__ out, float* __restrict__ lse) {
  __shared__ __align__(16) AtChunk<G> A;
  __shared__ AtState<G> St;
  at_cluster_row<G>(A, St, blockIdx.y, q, K, V, idx, idx_stride, count, Hq, Hkv, n, ncap,
                    max_count, scale, out, lse, [] { __syncthreads(); });
}

// Whether the cluster kernel can run on this device (cached per device).
template <int G>
static bool attend_cluster_ok() {
  if (fallback_forced()) return false;
  static std::atomic<int> ok[kMaxDev];
  return per_device_cached(ok, [] {
    auto kern = attend_cluster_kernel<G>;
    int nc = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(kAtCS, 1, 1);
      cfg.blockDim = dim3(128, 1, 1);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kAtCS;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess) nc = 0;
    }
    cudaGetLastError();
    return nc > 0 ? 1 : 0;
  }) != 0;
}

template <int G>
static int attend_t(const Dims& s, const uint16_t* q, const uint16_t* K, const uint16_t* V,
                    const int32_t* idx, int64_t idx_stride, const int32_t* count,
                    int64_t max_count, float scale, float* out, float* lse, void* ws,
                    cudaStream_t st) {
  const int64_t rows = (int64_t)s.B * s.Hkv;
  const int nch = (int)attend_chunks(max_count);
  if (!fallback_forced() && nch > 0) {  // many long rows: the streaming kernel
    AttWs w = carve_att(ws, rows, nch, G);
    int rc = launch_attend_stream(s, q, K, V, idx, idx_stride, count, max_count, scale, out, lse,
                                  w.ticket, w.part_o, w.part_ml, nch, st);
    if (rc != 1) return rc;
  }
  if (attend_cluster_ok<G>()) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kAtCS, (unsigned)rows, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kAtCS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, attend_cluster_kernel<G>, q, K, V, idx, idx_stride, count,
                           s.Hq, s.Hkv, s.n, s.ncap, (int)max_count, scale, out, lse) !=
        cudaSuccess)
      return check_launch("attend cluster");
    note_launches(1);
    return check_launch("attend cluster");
  }
  AttWs w = carve_att(ws, rows, nch, G);
  if (cudaMemsetAsync(w.ticket, 0, sizeof(uint32_t) * rows, st) != cudaSuccess)
    return check_launch("attend: ticket clear");
  dim3 grid((unsigned)(nch > 0 ? nch : 1), (unsigned)rows);
  attend_kernel<G><<<grid, 128, 0, st>>>(q, K, V, idx, idx_stride, count, s.Hq, s.Hkv, s.n,
                                         s.ncap, (int)max_count, scale, nch > 0 ? nch : 1, w,
                                         out, lse);
  note_launches(1);
  return check_launch("attend");
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
