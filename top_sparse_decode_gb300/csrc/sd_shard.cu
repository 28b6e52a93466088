// One sequence split by tokens across devices (HashAttention: Semantic Sparsity for
// Faster Inference, 2.5: contexts beyond one device need one exchange of top-k
// candidates and one of attention partials).  Shard s holds tokens [a_s, a_s + n_s)
// with its own index, K and V; the forced windows stay with the shard holding them.
//   shard_cand_kernel   -- from the shard's own top-k (idx ascending, forced tokens
//                          included): its competing tokens' scores and global indices;
//   topk_merge_kernel   -- the sequence's top-k of every shard's candidates: the first
//                          k in (score descending, global index ascending), ascending;
//   shard_select_kernel -- the shard's attention set in its own indices: its forced
//                          windows and the merged tokens it holds, ascending;
//   attend_combine_kernel -- the split-softmax combine of the shards' (out, lse).
#include "sd_internal.cuh"

namespace sd {
namespace {

constexpr int kMergeThreads = 1024;

// One warp per row: the competing entries idx in [sink_s, n_s - local_s), compacted
// in order, with their scores and global indices.
__global__ void shard_cand_kernel(const float* __restrict__ scores, int64_t rows, int64_t n_s,
                                  const int32_t* __restrict__ idx, int64_t idx_stride,
                                  const int32_t* __restrict__ count, int sink_s, int local_s,
                                  int64_t offset, int k, float* __restrict__ cs,
                                  int32_t* __restrict__ ci, int32_t* __restrict__ cc) {
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int c = count[row];
  if (c < 0) {
    if (lane == 0) cc[row] = -1;
    return;
  }
  const int64_t lo = sink_s, hi = imax64(n_s - local_s, (int64_t)sink_s);
  int w = 0;
  for (int i0 = 0; i0 < c; i0 += 32) {
    const int i = i0 + lane;
    const int t = i < c ? idx[row * idx_stride + i] : -1;
    const bool keep = i < c && t >= lo && t < hi;
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, keep);
    const int pos = w + __popc(m & ((1u << lane) - 1u));
    if (keep && pos < k) {
      cs[row * k + pos] = scores[row * n_s + t];
      ci[row * k + pos] = (int32_t)(offset + t);
    }
    w += __popc(m);
  }
  if (lane == 0) cc[row] = min(w, k);
}

// One CTA per row: S * k candidates as unique 64-bit keys (score key << 32 | ~index)
// sorted descending in shared memory (bitonic); the first k indices, re-sorted
// ascending, are the row's selection.
__global__ void __launch_bounds__(kMergeThreads)
topk_merge_kernel(int64_t rows, int S, int k, const float* __restrict__ cs,
                  const int32_t* __restrict__ ci, const int32_t* __restrict__ cc,
                  int32_t* __restrict__ out, int64_t out_stride, int32_t* __restrict__ ocount,
                  int P) {  // P: the sort size, a power of two >= S * k
  extern __shared__ __align__(16) uint64_t key[];
  __shared__ int bad, total;
  const int64_t row = blockIdx.x;
  const int t = threadIdx.x;
  if (t == 0) { bad = 0; total = 0; }
  __syncthreads();
  for (int s = t; s < S; s += blockDim.x) {
    const int c = cc[(int64_t)s * rows + row];
    if (c < 0) atomicOr(&bad, 1);
    else atomicAdd(&total, min(c, k));
  }
  __syncthreads();
  if (bad) {
    if (t == 0) ocount[row] = -1;
    return;
  }
  for (int e = t; e < P; e += blockDim.x) {
    uint64_t v = 0;  // empty slots sort last
    if (e < S * k) {
      const int s = e / k, j = e % k;
      if (j < min(cc[(int64_t)s * rows + row], k)) {
        const int64_t o = ((int64_t)s * rows + row) * k + j;
        v = ((uint64_t)key_of_f32(cs[o]) << 32) | (uint32_t)~(uint32_t)ci[o];
      }
    }
    key[e] = v;
  }
  __syncthreads();
  // bitonic sort, descending
  for (int size = 2; size <= P; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int e = t; e < P; e += blockDim.x) {
        const int p = e ^ stride;
        if (p > e) {
          const bool desc = (e & size) == 0;
          const uint64_t x = key[e], y = key[p];
          if (desc ? x < y : x > y) { key[e] = y; key[p] = x; }
        }
      }
      __syncthreads();
    }
  const int sel = min(k, total);
  // the first `sel` indices, ascending: sort them again (indices as keys)
  int Q = 1;
  while (Q < sel) Q <<= 1;
  for (int e = t; e < Q; e += blockDim.x)
    key[e] = e < sel ? (uint64_t)(uint32_t)~(uint32_t)(key[e] & 0xFFFFFFFFu) : ~0ull;
  __syncthreads();
  for (int size = 2; size <= Q; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int e = t; e < Q; e += blockDim.x) {
        const int p = e ^ stride;
        if (p > e) {
          const bool asc = (e & size) == 0;
          const uint64_t x = key[e], y = key[p];
          if (asc ? x > y : x < y) { key[e] = y; key[p] = x; }
        }
      }
      __syncthreads();
    }
  for (int e = t; e < sel; e += blockDim.x) out[row * out_stride + e] = (int32_t)key[e];
  if (t == 0) ocount[row] = sel;
}

// One warp per row: [0, sink_s), the merged tokens in [a, a + n_s) shifted to the
// shard's indices (the merge holds no forced token), [n_s - local_s, n_s).
__global__ void shard_select_kernel(int64_t rows, const int32_t* __restrict__ sel,
                                    int64_t sel_stride, const int32_t* __restrict__ scount,
                                    int64_t a, int64_t n_s, int sink_s, int local_s,
                                    int32_t* __restrict__ out, int64_t out_stride,
                                    int32_t* __restrict__ ocount) {
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int c = scount[row];
  if (c < 0) {
    if (lane == 0) ocount[row] = -1;
    return;
  }
  int32_t* o = out + row * out_stride;
  for (int i = lane; i < sink_s; i += 32) o[i] = i;
  int w = sink_s;
  for (int i0 = 0; i0 < c; i0 += 32) {
    const int i = i0 + lane;
    const int64_t t = i < c ? (int64_t)sel[row * sel_stride + i] : -1;
    const bool mine = i < c && t >= a && t < a + n_s;
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, mine);
    if (mine) o[w + __popc(m & ((1u << lane) - 1u))] = (int32_t)(t - a);
    w += __popc(m);
  }
  for (int i = lane; i < local_s; i += 32) o[w + i] = (int32_t)(n_s - local_s + i);
  if (lane == 0) ocount[row] = w + local_s;
}

// One thread per (sequence, query head, column): L = log sum_s exp(lse_s),
// o = sum_s exp(lse_s - L) o_s; shards with lse = -inf weigh 0.
__global__ void attend_combine_kernel(int S, int64_t BH, const float* __restrict__ outs,
                                      const float* __restrict__ lses, float* __restrict__ out,
                                      float* __restrict__ lse) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= BH * kD) return;
  const int64_t bh = e / kD;
  float m = -INFINITY;
  for (int s = 0; s < S; ++s) m = fmaxf(m, lses[(int64_t)s * BH + bh]);
  float l = 0.0f, o = 0.0f;
  if (m != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const float ls = lses[(int64_t)s * BH + bh];
      const float w = ls == -INFINITY ? 0.0f : expf(ls - m);
      l += w;
      o = fmaf(w, outs[(int64_t)s * BH * kD + e], o);
    }
  }
  out[e] = l > 0.0f ? o / l : 0.0f;
  if (lse && e % kD == 0) lse[bh] = l > 0.0f ? m + logf(l) : -INFINITY;
}

}  // namespace

int launch_shard_candidates(const float* scores, int64_t rows, int64_t n_s, const int32_t* idx,
                            int64_t idx_stride, const int32_t* count, int sink_s, int local_s,
                            int64_t offset, int k, float* cs, int32_t* ci, int32_t* cc,
                            cudaStream_t st) {
  const int wpb = 8;
  shard_cand_kernel<<<(unsigned)((rows + wpb - 1) / wpb), 32 * wpb, 0, st>>>(
      scores, rows, n_s, idx, idx_stride, count, sink_s, local_s, offset, k, cs, ci, cc);
  note_launches(1);
  return check_launch("shard candidates");
}

int launch_topk_merge(int64_t rows, int S, int k, const float* cs, const int32_t* ci,
                      const int32_t* cc, int32_t* out, int64_t out_stride, int32_t* ocount,
                      cudaStream_t st) {
  int P = 1;
  while (P < S * k) P <<= 1;
  const size_t smem = sizeof(uint64_t) * (size_t)P;
  if (int rc = set_smem_limit((const void*)topk_merge_kernel, smem, "topk merge: smem attribute"))
    return rc;
  topk_merge_kernel<<<(unsigned)rows, kMergeThreads, smem, st>>>(rows, S, k, cs, ci, cc, out,
                                                                 out_stride, ocount, P);
  note_launches(1);
  return check_launch("topk merge");
}

int launch_shard_select(int64_t rows, const int32_t* sel, int64_t sel_stride,
                        const int32_t* scount, int64_t a, int64_t n_s, int sink_s, int local_s,
                        int32_t* out, int64_t out_stride, int32_t* ocount, cudaStream_t st) {
  const int wpb = 8;
  shard_select_kernel<<<(unsigned)((rows + wpb - 1) / wpb), 32 * wpb, 0, st>>>(
      rows, sel, sel_stride, scount, a, n_s, sink_s, local_s, out, out_stride, ocount);
  note_launches(1);
  return check_launch("shard select");
}

int launch_attend_combine(int S, int64_t BH, const float* outs, const float* lses, float* out,
                          float* lse, cudaStream_t st) {
  const int64_t n = BH * kD;
  attend_combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(S, BH, outs, lses, out, lse);
  note_launches(1);
  return check_launch("attend combine");
}

}  // namespace sd
