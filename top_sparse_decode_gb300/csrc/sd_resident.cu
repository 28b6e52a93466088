// Delta selection against a resident set, and the gather of the admitted blocks
// (OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead Sparse Prefetching,
// method details: the KV-selection worker intersects the predicted top-K with the
// resident set, admits at most C non-resident blocks per KV head, each paired with
// a least-recently-selected eviction target; the transfer worker's UVA gather
// kernel writes those blocks from pinned host memory into the resident pages).
//
// One CTA per (sequence, KV head) row.  The predicted units are compacted from the
// top-k output into shared memory; hits are found through the unit -> slot map;
// the a = min(C, misses, targets) admissions are made one round at a time, each a
// block-wide arg-max over the misses' admission keys and arg-min over the free
// slots' (last selected, slot) keys, both cached in shared memory.  C is small in
// practice (a fetch ratio of a few percent of K), so a round per admission costs
// less than sorting either list.
#include "sd_internal.cuh"

namespace sd {

constexpr int kDsThreads = 256;
constexpr int kDsWarps = kDsThreads / 32;

// Shared memory: the reduction scratch, then per predicted unit its admission key
// mkey (0 once resident or admitted), the unit P (ascending) and its slot after the
// step pslot (-1 while not resident), then per slot the unit it holds and its target
// key (last selected + 1, slot), ~0 once it holds a predicted unit.  Sized by the
// launch's bounds (maxP = min(n_units, sink + local + k)): at OasisKV's 129 units
// and 129 slots a CTA needs under 4 KB, so every row of a large batch runs at once,
// and the admission rounds touch shared memory only.
struct DsHead {
  unsigned long long red[2][kDsWarps];
  int wtot[kDsWarps];
};

__host__ __device__ __forceinline__ size_t ds_smem_bytes(int maxP, int R) {
  return sizeof(DsHead) + 16 * (size_t)maxP + 12 * (size_t)R;
}

// Exclusive prefix of v over the CTA in thread order, and the total.
__device__ __forceinline__ int ds_scan(int v, int* wtot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kDsWarps; ++w) {
    before += w < warp ? wtot[w] : 0;
    all += wtot[w];
  }
  __syncthreads();
  *total = all;
  return before + incl - v;
}

__global__ void __launch_bounds__(kDsThreads)
delta_select_kernel(int maxP, int64_t nu, int64_t n_tokens, int block, int sink, int local,
                    const float* __restrict__ scores, const int32_t* __restrict__ idx,
                    int64_t idx_stride, const int32_t* __restrict__ count, int C, int step,
                    int R, int32_t* __restrict__ slot_unit, int32_t* __restrict__ slot_last,
                    int32_t* __restrict__ unit_slot, int32_t* __restrict__ plan_slot,
                    int32_t* __restrict__ plan_unit, int32_t* __restrict__ plan_evict,
                    int32_t* __restrict__ plan_count, int32_t* __restrict__ pool_idx,
                    int64_t pool_stride, int32_t* __restrict__ pool_count) {
  extern __shared__ __align__(16) uint8_t ds_raw[];
  DsHead& S = *reinterpret_cast<DsHead*>(ds_raw);
  unsigned long long* mkey = reinterpret_cast<unsigned long long*>(ds_raw + sizeof(DsHead));
  unsigned long long* skey = mkey + maxP;
  int32_t* P = reinterpret_cast<int32_t*>(skey + R);
  int32_t* pslot = P + maxP;
  int32_t* sunit = pslot + maxP;
  const int64_t row = blockIdx.x;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  int32_t* su = slot_unit + row * R;
  int32_t* sl = slot_last + row * R;
  int32_t* us = unit_slot + row * nu;
  const float* sc = scores + row * nu;
  const int32_t* ir = idx + row * idx_stride;
  const int c = (int)min((int64_t)count[row], idx_stride);
  if (c < 0) {  // a NaN score in the row: nothing changes
    if (t == 0) {
      plan_count[row] = -1;
      pool_count[row] = -1;
    }
    return;
  }
  // the slots' state, once
  for (int s = t; s < R; s += kDsThreads) {
    sunit[s] = su[s];
    skey[s] = ((unsigned long long)(uint32_t)(sl[s] + 1) << 32) | (uint32_t)s;
  }
  // the predicted units: the tokens that start a unit, in the top-k's (ascending)
  // order; thread t takes the contiguous segment [t * per, (t + 1) * per) of the list
  const int per = (c + kDsThreads - 1) / kDsThreads;
  const int i0 = min(t * per, c), i1 = min(i0 + per, c);
  auto unit_of = [&](int32_t tok) -> int {
    return (tok >= 0 && tok < n_tokens && tok % block == 0 && tok / block < nu) ? tok / block
                                                                                 : -1;
  };
  int mine_n = 0;
  for (int i = i0; i < i1; ++i) mine_n += unit_of(ir[i]) >= 0;
  int np;
  int pos = ds_scan(mine_n, S.wtot, &np);
  for (int i = i0; i < i1; ++i) {
    const int u = unit_of(ir[i]);
    if (u >= 0) {
      if (pos < maxP) P[pos] = u;
      ++pos;
    }
  }
  np = min(np, maxP);
  __syncthreads();
  // hits: resident predicted units (a map entry that disagrees with its slot counts
  // as not resident) refresh their slot's last-selected step; misses get their
  // admission key: forced units first, then score descending, unit ascending (the
  // unit sits in the low bits, so keys are unique and never 0)
  int my_hits = 0, my_miss = 0;
  for (int i = t; i < np; i += kDsThreads) {
    const int u = P[i];
    const int s = us[u];
    const bool hit = s >= 0 && s < R && sunit[s] == u;
    unsigned long long key = 0ull;
    if (hit) {
      skey[s] = ~0ull;
      sl[s] = step;
      ++my_hits;
    } else {
      const bool forced = u < sink || (int64_t)u >= nu - local;
      key = forced ? (1ull << 63) | (0x7FFFFFFFull - (unsigned)u)
                   : ((unsigned long long)key_of_f32(sc[u]) << 31) | (0x7FFFFFFFull - (unsigned)u);
      ++my_miss;
    }
    mkey[i] = key;
    pslot[i] = hit ? s : -1;
  }
  int hits, misses;
  ds_scan(my_hits, S.wtot, &hits);
  ds_scan(my_miss, S.wtot, &misses);
  const int a = min(C, min(misses, R - hits));
  int made = 0;
  for (int i = 0; i < a; ++i) {
    // the best remaining miss and the oldest free slot (empty slots hold key 0 in
    // their high half, so they come first)
    unsigned long long bm = 0ull, bt = ~0ull;
    int bj = -1;
    for (int j = t; j < np; j += kDsThreads) {
      const unsigned long long k = mkey[j];
      if (k > bm) {
        bm = k;
        bj = j;
      }
    }
    for (int s = t; s < R; s += kDsThreads) bt = min(bt, skey[s]);
    const unsigned long long mine = bm;  // this thread's own best miss
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      bm = max(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, o));
      bt = min(bt, __shfl_xor_sync(0xFFFFFFFFu, bt, o));
    }
    if (lane == 0) {
      S.red[0][warp] = bm;
      S.red[1][warp] = bt;
    }
    __syncthreads();
    unsigned long long wm = 0ull, wt = ~0ull;
#pragma unroll
    for (int w = 0; w < kDsWarps; ++w) {
      wm = max(wm, S.red[0][w]);
      wt = min(wt, S.red[1][w]);
    }
    if (wm == 0ull || wt == ~0ull) break;  // no miss or no free slot left (uniform)
    const int s = (int)(uint32_t)wt;
    if (bj >= 0 && mine == wm) {  // the winning miss's owner
      mkey[bj] = 0ull;
      pslot[bj] = s;
    }
    if (t == 0) {
      const int u = (int)(0x7FFFFFFFull - (wm & 0x7FFFFFFFull));
      const int old = sunit[s];
      const bool had = old >= 0 && old < nu;
      if (had) us[old] = -1;  // evicted: no longer resident
      su[s] = u;
      sl[s] = step;
      us[u] = s;
      sunit[s] = u;
      skey[s] = ~0ull;
      plan_slot[row * C + i] = s;
      plan_unit[row * C + i] = u;
      plan_evict[row * C + i] = had ? old : -1;
    }
    ++made;
    __syncthreads();
  }
  if (t == 0) plan_count[row] = made;
  // pool rows of the resident predicted units, in unit order
  int64_t base_rows = 0;
  for (int base = 0; base < np; base += kDsThreads) {
    const int i = base + t;
    int len = 0, s = -1, u = 0;
    if (i < np && pslot[i] >= 0) {
      s = pslot[i];
      u = P[i];
      len = (int)min((int64_t)block, n_tokens - (int64_t)u * block);
    }
    int tot;
    const int64_t pos = base_rows + ds_scan(len, S.wtot, &tot);
    for (int r = 0; r < len; ++r)
      if (pos + r < pool_stride) pool_idx[row * pool_stride + pos + r] = s * block + r;
    base_rows += tot;
  }
  if (t == 0) pool_count[row] = (int32_t)min(base_rows, pool_stride);
}

int launch_delta_select(int64_t rows, int64_t nu, int64_t n_tokens, int block, int sink,
                        int local, int sel_k, const float* scores, const int32_t* idx, int64_t idx_stride,
                        const int32_t* count, int C, int step, int R, int32_t* slot_unit,
                        int32_t* slot_last, int32_t* unit_slot, int32_t* plan_slot,
                        int32_t* plan_unit, int32_t* plan_evict, int32_t* plan_count,
                        int32_t* pool_idx, int64_t pool_stride, int32_t* pool_count,
                        cudaStream_t st) {
  const int maxP = (int)imin64(nu, (int64_t)sink + local + sel_k);
  const size_t smem = ds_smem_bytes(maxP, R);
  if (int rc = set_smem_limit((const void*)delta_select_kernel, smem, "delta_select: smem attribute"))
    return rc;
  delta_select_kernel<<<(unsigned)rows, kDsThreads, smem, st>>>(
      maxP, nu, n_tokens, block, sink, local, scores, idx, idx_stride, count, C, step, R, slot_unit,
      slot_last, unit_slot, plan_slot, plan_unit, plan_evict, plan_count, pool_idx, pool_stride,
      pool_count);
  note_launches(1);
  return check_launch("delta_select");
}

// The transfer: CTA (i, row) copies admitted unit plan_unit[row][i] (tokens
// [u*block, min((u+1)*block, n))) of K and V into pool rows slot*block.. of the
// row's pool; rows of a short last unit past n are zero-filled.  Sources may be
// device memory or pinned host memory mapped into the device's address space.
constexpr int kRgThreads = 128;

__global__ void __launch_bounds__(kRgThreads)
resident_gather_kernel(int64_t n, int64_t ncap, int block, const uint16_t* __restrict__ K,
                       const uint16_t* __restrict__ V, const int32_t* __restrict__ plan_slot,
                       const int32_t* __restrict__ plan_unit,
                       const int32_t* __restrict__ plan_count, int C, int R,
                       uint16_t* __restrict__ Kp, uint16_t* __restrict__ Vp) {
  const int i = blockIdx.x;
  const int64_t row = blockIdx.y;
  if (i >= min(plan_count[row], C)) return;
  const int s = plan_slot[row * C + i], u = plan_unit[row * C + i];
  const int64_t nu = (n + block - 1) / block;
  if (s < 0 || s >= R || u < 0 || u >= nu) return;  // not a plan entry
  const int64_t t0 = (int64_t)u * block;
  const uint4* ks = reinterpret_cast<const uint4*>(K + (row * ncap + t0) * kD);
  const uint4* vs = reinterpret_cast<const uint4*>(V + (row * ncap + t0) * kD);
  uint4* kd = reinterpret_cast<uint4*>(Kp + (row * R + s) * (int64_t)block * kD);
  uint4* vd = reinterpret_cast<uint4*>(Vp + (row * R + s) * (int64_t)block * kD);
  const int segs = block * (kD / 8);  // 16-byte segments per unit
  // all loads of a thread in flight before its stores (the host link's latency)
  constexpr int kPer = 4;
  for (int e0 = threadIdx.x; e0 < segs; e0 += kRgThreads * kPer) {
    uint4 kv[kPer], vv[kPer];
#pragma unroll
    for (int p = 0; p < kPer; ++p) {
      const int e = e0 + p * kRgThreads;
      kv[p] = vv[p] = make_uint4(0u, 0u, 0u, 0u);
      if (e < segs && t0 + e / (kD / 8) < n) {
        kv[p] = ks[e];
        vv[p] = vs[e];
      }
    }
#pragma unroll
    for (int p = 0; p < kPer; ++p) {
      const int e = e0 + p * kRgThreads;
      if (e < segs) {
        kd[e] = kv[p];
        vd[e] = vv[p];
      }
    }
  }
}

int launch_resident_gather(const Dims& s, int block, const uint16_t* K, const uint16_t* V,
                           const int32_t* plan_slot, const int32_t* plan_unit,
                           const int32_t* plan_count, int C, int R, uint16_t* Kp, uint16_t* Vp,
                           cudaStream_t st) {
  if (C == 0) return SD_OK;
  dim3 grid((unsigned)C, (unsigned)(s.B * s.Hkv));
  resident_gather_kernel<<<grid, kRgThreads, 0, st>>>(s.n, s.ncap, block, K, V, plan_slot,
                                                      plan_unit, plan_count, C, R, Kp, Vp);
  note_launches(1);
  return check_launch("resident_gather");
}

}  // namespace sd
