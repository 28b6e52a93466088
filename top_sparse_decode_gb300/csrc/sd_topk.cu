// TOPK: exact top-k per row with forced windows.
//   HashAttention: Semantic Sparsity for Faster Inference, 2.1 (TOPK stage) and
//   3.1 (first and last tokens always kept, budget counted apart);
//   OasisKV: ..., method details (top-K blocks plus the active local block).
//
// Order: score descending, unit ascending.  Each candidate u in [lead, tail)
// gets a unique 64-bit composite key
//     C(u) = (key(u) - kmin) << bI  |  (M - 1 - (u - lead))
// (key = order-preserving 32-bit image of the score, kmin its row minimum,
// M = tail - lead candidates, bI = bits of M - 1), so "top-k by C" is exactly
// the required order with no ties left.  Rows of up to kSmallRow units are
// selected by one CTA in shared memory.  Longer rows:
//   1. row min/max of the keys (multi-CTA);
//   2. one 11-bit histogram pass over the top digit of C (multi-CTA; the
//      last CTA of a row picks the digit holding the k-th largest);
//   3. compaction: units with a larger digit go to an "above" list (< k of
//      them), units with that digit to a candidate list;
//   4. one CTA per row finishes the radix select among the candidates in
//      shared memory, merges with the above list, sorts ascending and writes
//      the forced and selected units expanded to tokens.
// If the chosen digit holds more than kCap candidates (only for rows with
// enormous runs of near-equal scores), step 4 resolves the remaining digits
// by passes over the row in global memory: slower, same result.
#include "sd_internal.cuh"

namespace sd {

constexpr int kCap = 8192;          // candidates a finishing CTA holds in shared memory
constexpr int kFinThreads = 1024;
constexpr int kChunk = 8192;        // units per CTA in the multi-CTA steps
constexpr int kDigit = 11;
constexpr int kBins = 1 << kDigit;

struct RowState {
  uint32_t inv_min;  // ~(row min key), via atomicMax (zero-initialised)
  uint32_t max_key;  // row max key, via atomicMax
  uint32_t nan;      // a NaN was seen
  uint32_t ticket;   // CTAs done with the histogram pass
  uint32_t digit;    // chosen top digit
  uint32_t need;     // how many of the digit's units to take
  uint32_t bucket;   // units with that digit
  uint32_t nabove;   // units with a larger digit (compaction counter)
  uint32_t ncand;    // compaction counter of the candidate list
  uint32_t pad[7];
  uint32_t hist[kBins];
};

struct Ws {
  RowState* st;      // [rows]
  uint32_t* above;   // [rows][kMaxTopK]
  uint64_t* cand;    // [rows][kCap]
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static Ws carve(void* base, int64_t rows) {
  uint8_t* p = (uint8_t*)base;
  Ws w;
  w.st = (RowState*)p;
  p += align256(sizeof(RowState) * rows);
  w.above = (uint32_t*)p;
  p += align256(sizeof(uint32_t) * kMaxTopK * rows);
  w.cand = (uint64_t*)p;
  return w;
}

size_t topk_workspace_bytes(int64_t rows, int64_t n_units, const sd_select&) {
  if (n_units <= kSmallRow) return 0;
  return align256(sizeof(RowState) * rows) + align256(sizeof(uint32_t) * kMaxTopK * rows) +
         align256(sizeof(uint64_t) * kCap * rows);
}

struct Geo {  // per-row candidate geometry
  int64_t n_units, n_tokens;
  int lead, tail, M, k, block;
};

__host__ __device__ inline Geo make_geo(int64_t n_units, int64_t n_tokens, const sd_select& s) {
  Geo g;
  g.n_units = n_units;
  g.n_tokens = n_tokens;
  g.lead = (int)imin64(s.sink, n_units);
  g.tail = (int)imax64(n_units - s.local, g.lead);
  g.M = g.tail - g.lead;
  g.k = s.k;
  g.block = s.block;
  return g;
}

template <bool F32>
__device__ __forceinline__ uint32_t load_key(const void* scores, int64_t off, bool& nan) {
  if (F32) {
    float f = __ldg(reinterpret_cast<const float*>(scores) + off);
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) nan = true;
    return key_of_f32(f);
  } else {
    return key_of_i32(__ldg(reinterpret_cast<const int32_t*>(scores) + off));
  }
}

__device__ __forceinline__ int bits_of(uint32_t x) { return x ? 32 - __clz(x) : 0; }

// --------------------------------------------------------------------------------------
// Block-wide helpers (blockDim.x = NT, a multiple of 32)
// --------------------------------------------------------------------------------------
// Given hist[0..kBins) and r >= 1 (r <= total), find digit d with
// above(d) < r <= above(d) + hist[d], above(d) = sum of hist[b] for b > d.
// Result in out[0] = d, out[1] = above(d).  Uses scratch[32].
template <int NT>
__device__ void pick_digit(const uint32_t* hist, uint32_t r, uint32_t* scratch, uint32_t* out) {
  constexpr int PER = kBins / NT;  // bins per thread, contiguous
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  uint32_t loc = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) loc += hist[t * PER + i];
  // inclusive suffix sum over threads >= t
  uint32_t suf = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_down_sync(0xFFFFFFFFu, suf, o);
    if (lane + o < 32) suf += y;
  }
  if (lane == 0) scratch[warp] = suf;  // warp total
  __syncthreads();
  uint32_t later = 0;  // totals of warps after this one
  for (int w = warp + 1; w < NT / 32; ++w) later += scratch[w];
  uint32_t above = suf - loc + later;  // sum over bins of threads > t
#pragma unroll
  for (int i = PER - 1; i >= 0; --i) {
    uint32_t h = hist[t * PER + i];
    if (above < r && r <= above + h) {
      out[0] = t * PER + i;
      out[1] = above;
    }
    above += h;
  }
  __syncthreads();
}

// Bitonic sort ascending of a[0..n2) (n2 a power of two) in shared memory.
template <int NT>
__device__ void bitonic_sort_u32(uint32_t* a, int n2) {
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n2 / 2; i += NT) {
        int lo = 2 * i - (i & (stride - 1));
        int hi = lo + stride;
        bool up = ((lo & size) == 0);
        uint32_t x = a[lo], y = a[hi];
        if ((x > y) == up) { a[lo] = y; a[hi] = x; }
      }
      __syncthreads();
    }
  }
}

// Finds T such that exactly `need` of the c unique values C[0..c) are >= T,
// given that all of them equal `prefix` in the bits above `pos`.
template <int NT>
__device__ uint64_t radix_threshold(const uint64_t* C, int c, uint32_t need, uint64_t prefix,
                                    int pos, uint32_t* hist, uint32_t* scratch, uint32_t* out) {
  uint32_t r = need;
  while (pos > 0) {
    const int w = min(kDigit, pos);
    const int npos = pos - w;
    for (int b = threadIdx.x; b < kBins; b += NT) hist[b] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < c; i += NT) {
      uint64_t x = C[i];
      if ((x >> pos) == prefix) atomicAdd(&hist[(uint32_t)(x >> npos) & ((1u << w) - 1)], 1u);
    }
    __syncthreads();
    pick_digit<NT>(hist, r, scratch, out);
    const uint32_t d = out[0], above = out[1], inb = hist[d];
    __syncthreads();
    r -= above;
    prefix = (prefix << w) | d;
    pos = npos;
    if (inb == r) break;
  }
  return prefix << pos;
}

// Writes the final ascending unit list (lead units, the sorted selected units,
// tail units) expanded to tokens, and the count.
template <int NT>
__device__ void write_units(const Geo& g, const uint32_t* sel, int nsel, int32_t* idx_row,
                            int32_t* count_row) {
  const int ntail = (int)(g.n_units - g.tail);
  const int nunits = g.lead + nsel + ntail;
  const int64_t total = (int64_t)nunits * g.block;
  for (int64_t p = threadIdx.x; p < total; p += NT) {
    int ui = (int)(p / g.block), off = (int)(p % g.block);
    int64_t u = ui < g.lead ? ui : (ui < g.lead + nsel ? (int64_t)sel[ui - g.lead]
                                                      : (int64_t)g.tail + (ui - g.lead - nsel));
    int64_t tok = u * g.block + off;
    if (tok < g.n_tokens) idx_row[p] = (int32_t)tok;
  }
  if (threadIdx.x == 0) {
    bool last_in = ntail > 0 || (nsel > 0 && (int64_t)sel[nsel - 1] == g.n_units - 1) ||
                   (nsel == 0 && ntail == 0 && g.lead == g.n_units);
    int64_t cnt = total;
    if (last_in) cnt -= (g.n_units * g.block - g.n_tokens);
    *count_row = (int32_t)cnt;
  }
}

// Shared memory of a finishing CTA.
struct FinSmem {
  uint64_t C[kCap];
  uint32_t sel[kMaxTopK];
  uint32_t hist[kBins];
  uint32_t scratch[32];
  uint32_t out[4];
  uint32_t nsel;
  uint32_t flag;
  uint32_t kmin, kmax;
};

// --------------------------------------------------------------------------------------
// Rows of at most kSmallRow units: everything in one CTA.
// --------------------------------------------------------------------------------------
template <bool F32>
__global__ void __launch_bounds__(kFinThreads)
topk_small_kernel(const void* __restrict__ scores, Geo g, int32_t* __restrict__ idx,
                  int64_t idx_stride, int32_t* __restrict__ count) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  FinSmem& S = *reinterpret_cast<FinSmem*>(smem_raw);
  const int64_t row = blockIdx.x;
  int32_t* idx_row = idx + row * idx_stride;
  const int64_t base = row * g.n_units;
  uint32_t* keys = reinterpret_cast<uint32_t*>(S.C);  // keys first, composite later (in place)
  if (threadIdx.x == 0) { S.flag = 0; S.kmin = 0xFFFFFFFFu; S.kmax = 0; S.nsel = 0; }
  __syncthreads();
  bool nan = false;
  uint32_t mn = 0xFFFFFFFFu, mx = 0;
  for (int i = threadIdx.x; i < g.M; i += kFinThreads) {
    uint32_t kk = load_key<F32>(scores, base + g.lead + i, nan);
    keys[2 * i] = kk;  // stash in the low word of C[i]
    mn = min(mn, kk);
    mx = max(mx, kk);
  }
  if (nan) atomicOr(&S.flag, 1u);
  atomicMin(&S.kmin, mn);
  atomicMax(&S.kmax, mx);
  __syncthreads();
  if (S.flag) {
    if (threadIdx.x == 0) count[row] = -1;
    return;
  }
  if (g.M <= g.k) {  // every candidate is taken: the output is already in order
    for (int i = threadIdx.x; i < g.M; i += kFinThreads) S.sel[i] = g.lead + i;
    __syncthreads();
    write_units<kFinThreads>(g, S.sel, g.M, idx_row, count + row);
    return;
  }
  const uint32_t kmin = S.kmin;
  const int bI = bits_of((uint32_t)(g.M - 1));
  const int nb = bits_of(S.kmax - kmin) + bI;
  for (int i = threadIdx.x; i < g.M; i += kFinThreads) {
    uint32_t kk = keys[2 * i];
    S.C[i] = ((uint64_t)(kk - kmin) << bI) | (uint64_t)(g.M - 1 - i);
  }
  __syncthreads();
  const uint64_t T = radix_threshold<kFinThreads>(S.C, g.M, (uint32_t)g.k, 0, nb, S.hist,
                                                  S.scratch, S.out);
  for (int i = threadIdx.x; i < g.M; i += kFinThreads) {
    uint64_t x = S.C[i];
    if (x >= T) S.sel[atomicAdd(&S.nsel, 1u)] = g.lead + (g.M - 1 - (uint32_t)(x & ((1ull << bI) - 1)));
  }
  __syncthreads();
  const int nsel = (int)S.nsel;
  int n2 = 1;
  while (n2 < nsel) n2 <<= 1;
  for (int i = nsel + threadIdx.x; i < n2; i += kFinThreads) S.sel[i] = 0xFFFFFFFFu;
  __syncthreads();
  bitonic_sort_u32<kFinThreads>(S.sel, n2);
  write_units<kFinThreads>(g, S.sel, nsel, idx_row, count + row);
}

// --------------------------------------------------------------------------------------
// Long rows.
// --------------------------------------------------------------------------------------
template <bool F32>
__global__ void __launch_bounds__(256)
topk_minmax_kernel(const void* __restrict__ scores, Geo g, Ws ws) {
  const int64_t row = blockIdx.y;
  RowState& st = ws.st[row];
  const int64_t i0 = (int64_t)blockIdx.x * kChunk;
  const int64_t i1 = imin64(i0 + kChunk, g.M);
  bool nan = false;
  uint32_t mn = 0xFFFFFFFFu, mx = 0;
  for (int64_t i = i0 + threadIdx.x; i < i1; i += 256) {
    uint32_t kk = load_key<F32>(scores, row * g.n_units + g.lead + i, nan);
    mn = min(mn, kk);
    mx = max(mx, kk);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  }
  if (__any_sync(0xFFFFFFFFu, nan) && (threadIdx.x & 31) == 0) atomicOr(&st.nan, 1u);
  if ((threadIdx.x & 31) == 0) {
    atomicMax(&st.inv_min, ~mn);
    atomicMax(&st.max_key, mx);
  }
}

struct Comp {  // composite-key geometry of a row
  uint32_t kmin;
  int bI, nb, w0, shift0;
};

__device__ __forceinline__ Comp row_comp(const RowState& st, const Geo& g) {
  Comp c;
  c.kmin = ~st.inv_min;
  c.bI = bits_of((uint32_t)(g.M - 1));
  c.nb = bits_of(st.max_key - c.kmin) + c.bI;
  c.w0 = min(kDigit, c.nb);
  c.shift0 = c.nb - c.w0;
  return c;
}

__device__ __forceinline__ uint64_t composite(uint32_t key, int64_t i, const Comp& c, int M) {
  return ((uint64_t)(key - c.kmin) << c.bI) | (uint64_t)(M - 1 - i);
}

template <bool F32>
__global__ void __launch_bounds__(256)
topk_hist_kernel(const void* __restrict__ scores, Geo g, Ws ws, unsigned nchunks) {
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t scratch[32];
  __shared__ uint32_t out[4];
  __shared__ bool last;
  const int64_t row = blockIdx.y;
  RowState& st = ws.st[row];
  if (st.nan || g.M <= g.k) return;
  const Comp c = row_comp(st, g);
  for (int b = threadIdx.x; b < kBins; b += 256) hist[b] = 0;
  __syncthreads();
  const int64_t i0 = (int64_t)blockIdx.x * kChunk;
  const int64_t i1 = imin64(i0 + kChunk, g.M);
  bool nan = false;
  for (int64_t i = i0 + threadIdx.x; i < i1; i += 256) {
    uint32_t kk = load_key<F32>(scores, row * g.n_units + g.lead + i, nan);
    atomicAdd(&hist[(uint32_t)(composite(kk, i, c, g.M) >> c.shift0)], 1u);
  }
  __syncthreads();
  for (int b = threadIdx.x; b < kBins; b += 256)
    if (hist[b]) atomicAdd(&st.hist[b], hist[b]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = (atomicAdd(&st.ticket, 1u) == nchunks - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int b = threadIdx.x; b < kBins; b += 256) hist[b] = __ldcg(&st.hist[b]);
  __syncthreads();
  pick_digit<256>(hist, (uint32_t)g.k, scratch, out);
  if (threadIdx.x == 0) {
    st.digit = out[0];
    st.need = (uint32_t)g.k - out[1];
    st.bucket = hist[out[0]];
  }
}

template <bool F32>
__global__ void __launch_bounds__(256)
topk_filter_kernel(const void* __restrict__ scores, Geo g, Ws ws) {
  const int64_t row = blockIdx.y;
  const RowState& st = ws.st[row];
  if (st.nan || g.M <= g.k) return;
  const Comp c = row_comp(st, g);
  const uint32_t d = st.digit;
  const bool keep_cand = st.bucket <= (uint32_t)kCap;
  uint32_t* above = ws.above + row * kMaxTopK;
  uint64_t* cand = ws.cand + row * kCap;
  RowState& stw = ws.st[row];
  const int lane = threadIdx.x & 31;
  const int64_t i0 = (int64_t)blockIdx.x * kChunk;
  const int64_t i1 = imin64(i0 + kChunk, g.M);
  bool nan = false;
  for (int64_t ib = i0; ib < i1; ib += 256) {
    const int64_t i = ib + threadIdx.x;
    uint64_t x = 0;
    uint32_t dig = 0;
    bool valid = i < i1;
    if (valid) {
      x = composite(load_key<F32>(scores, row * g.n_units + g.lead + i, nan), i, c, g.M);
      dig = (uint32_t)(x >> c.shift0);
    }
    const bool up = valid && dig > d;
    const bool eq = valid && keep_cand && dig == d;
    // warp-aggregated appends
    uint32_t mu = __ballot_sync(0xFFFFFFFFu, up);
    if (mu) {
      uint32_t basep = 0;
      if (lane == 0) basep = atomicAdd(&stw.nabove, __popc(mu));
      basep = __shfl_sync(0xFFFFFFFFu, basep, 0);
      if (up) above[basep + __popc(mu & ((1u << lane) - 1))] = (uint32_t)(g.lead + i);
    }
    uint32_t me = __ballot_sync(0xFFFFFFFFu, eq);
    if (me) {
      uint32_t basep = 0;
      if (lane == 0) basep = atomicAdd(&stw.ncand, __popc(me));
      basep = __shfl_sync(0xFFFFFFFFu, basep, 0);
      if (eq) cand[basep + __popc(me & ((1u << lane) - 1))] = x;
    }
  }
}

template <bool F32>
__global__ void __launch_bounds__(kFinThreads)
topk_finish_kernel(const void* __restrict__ scores, Geo g, Ws ws, int32_t* __restrict__ idx,
                   int64_t idx_stride, int32_t* __restrict__ count) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  FinSmem& S = *reinterpret_cast<FinSmem*>(smem_raw);
  const int64_t row = blockIdx.x;
  const RowState& st = ws.st[row];
  int32_t* idx_row = idx + row * idx_stride;
  if (st.nan) {
    if (threadIdx.x == 0) count[row] = -1;
    return;
  }
  if (threadIdx.x == 0) S.nsel = 0;
  if (g.M <= g.k) {
    for (int i = threadIdx.x; i < g.M; i += kFinThreads) S.sel[i] = g.lead + i;
    __syncthreads();
    write_units<kFinThreads>(g, S.sel, g.M, idx_row, count + row);
    return;
  }
  const Comp c = row_comp(st, g);
  const uint32_t d = st.digit, need = st.need, bucket = st.bucket, nabove = st.nabove;
  const uint32_t* above = ws.above + row * kMaxTopK;
  for (uint32_t i = threadIdx.x; i < nabove; i += kFinThreads) S.sel[i] = above[i];
  if (threadIdx.x == 0) S.nsel = nabove;
  __syncthreads();
  if (bucket <= (uint32_t)kCap) {
    const uint64_t* cand = ws.cand + row * kCap;
    for (uint32_t i = threadIdx.x; i < bucket; i += kFinThreads) S.C[i] = cand[i];
    __syncthreads();
    const uint64_t T = radix_threshold<kFinThreads>(S.C, (int)bucket, need, d, c.shift0,
                                                    S.hist, S.scratch, S.out);
    for (uint32_t i = threadIdx.x; i < bucket; i += kFinThreads) {
      uint64_t x = S.C[i];
      if (x >= T)
        S.sel[atomicAdd(&S.nsel, 1u)] =
            g.lead + (g.M - 1 - (uint32_t)(x & ((1ull << c.bI) - 1)));
    }
  } else {
    // Slow path: resolve the remaining digits with passes over the row.
    uint64_t prefix = d;
    int pos = c.shift0;
    uint32_t r = need;
    bool nan = false;
    while (pos > 0) {
      const int w = min(kDigit, pos);
      const int npos = pos - w;
      for (int b = threadIdx.x; b < kBins; b += kFinThreads) S.hist[b] = 0;
      __syncthreads();
      for (int64_t i = threadIdx.x; i < g.M; i += kFinThreads) {
        uint64_t x = composite(load_key<F32>(scores, row * g.n_units + g.lead + i, nan), i, c, g.M);
        if ((x >> pos) == prefix) atomicAdd(&S.hist[(uint32_t)(x >> npos) & ((1u << w) - 1)], 1u);
      }
      __syncthreads();
      pick_digit<kFinThreads>(S.hist, r, S.scratch, S.out);
      const uint32_t dd = S.out[0], ab = S.out[1], inb = S.hist[dd];
      __syncthreads();
      r -= ab;
      prefix = (prefix << w) | dd;
      pos = npos;
      if (inb == r) break;
    }
    const uint64_t T = prefix << pos;
    const uint64_t lo_d = (uint64_t)d << c.shift0, hi_d = ((uint64_t)d + 1) << c.shift0;
    for (int64_t i = threadIdx.x; i < g.M; i += kFinThreads) {
      uint64_t x = composite(load_key<F32>(scores, row * g.n_units + g.lead + i, nan), i, c, g.M);
      if (x >= lo_d && x < hi_d && x >= T) S.sel[atomicAdd(&S.nsel, 1u)] = (uint32_t)(g.lead + i);
    }
  }
  __syncthreads();
  const int nsel = (int)S.nsel;
  int n2 = 1;
  while (n2 < nsel) n2 <<= 1;
  for (int i = nsel + threadIdx.x; i < n2; i += kFinThreads) S.sel[i] = 0xFFFFFFFFu;
  __syncthreads();
  bitonic_sort_u32<kFinThreads>(S.sel, n2);
  write_units<kFinThreads>(g, S.sel, nsel, idx_row, count + row);
}

template <bool F32>
static int topk_t(const void* scores, int64_t rows, const Geo& g, int32_t* idx,
                  int64_t idx_stride, int32_t* count, void* wsp, size_t ws_bytes,
                  cudaStream_t st) {
  const size_t smem = sizeof(FinSmem);
  if (g.n_units <= kSmallRow) {
    auto kern = topk_small_kernel<F32>;
    if (int rc_ = set_smem_limit((const void*)kern, smem, "topk: smem attribute")) return rc_;
    kern<<<(unsigned)rows, kFinThreads, smem, st>>>(scores, g, idx, idx_stride, count);
    return check_launch("topk_small");
  }
  Ws ws = carve(wsp, rows);
  if (cudaMemsetAsync(ws.st, 0, sizeof(RowState) * rows, st) != cudaSuccess)
    return check_launch("topk: workspace clear");
  const unsigned nchunks = (unsigned)((g.M + kChunk - 1) / kChunk);
  dim3 grid(max(nchunks, 1u), (unsigned)rows);
  topk_minmax_kernel<F32><<<grid, 256, 0, st>>>(scores, g, ws);
  topk_hist_kernel<F32><<<grid, 256, 0, st>>>(scores, g, ws, max(nchunks, 1u));
  topk_filter_kernel<F32><<<grid, 256, 0, st>>>(scores, g, ws);
  auto fin = topk_finish_kernel<F32>;
  if (int rc_ = set_smem_limit((const void*)fin, smem, "topk: smem attribute")) return rc_;
  fin<<<(unsigned)rows, kFinThreads, smem, st>>>(scores, g, ws, idx, idx_stride, count);
  return check_launch("topk");
}

int launch_topk(int score_type, const void* scores, int64_t rows, int64_t n_units,
                int64_t n_tokens, const sd_select& sel, int32_t* idx, int64_t idx_stride,
                int32_t* count, void* ws, size_t ws_bytes, cudaStream_t st) {
  Geo g = make_geo(n_units, n_tokens, sel);
  if (score_type == SD_SCORE_F32)
    return topk_t<true>(scores, rows, g, idx, idx_stride, count, ws, ws_bytes, st);
  return topk_t<false>(scores, rows, g, idx, idx_stride, count, ws, ws_bytes, st);
}

}  // namespace sd
