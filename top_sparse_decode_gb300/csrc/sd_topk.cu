// TOPK: exact top-k per row with forced windows.
//   HashAttention: Semantic Sparsity for Faster Inference, 2.1 (TOPK stage) and
//   3.1 (first and last tokens always kept, budget counted apart);
//   OasisKV: ..., method details (top-K blocks plus the active local block).
//
// Order: score descending, unit ascending.  Within a set of candidates, unit u
// gets a unique 64-bit composite key
//     C(u) = (key(u) - kmin) << bI  |  (M - 1 - (u - lead))
// (key = order-preserving 32-bit image of the score, kmin the candidates' minimum,
// M = tail - lead candidates, bI = bits of M - 1), so "top-k by C" is exactly the
// required order with no ties left, and a radix select over C needs no tie pass.
// Rows of up to kSmallRow units are selected by one CTA in shared memory, or in
// registers when at most kRegRow of their units compete.
// Longer rows take three kernels:
//   1. sample: one CTA per row reads an evenly spaced sample of up to 16K keys
//      and takes T_est = its r-th largest key, r = mu + 5 sqrt(mu) + 2 with
//      mu = k * sample / M the expected number of top-k members in the sample;
//   2. filter: one pass over the row appends (key, unit) of every key >= T_est
//      to the row's candidate list (warp-aggregated atomics);
//   3. finish: one CTA per row selects the top k of the candidates by C in
//      shared memory, sorts them ascending and writes the forced and selected
//      units expanded to tokens.
// The result is exact whatever the sample: if at least k keys are >= T_est, every
// member of the top k (and every key tied with the k-th) is a candidate.  When
// the estimate misses (fewer than k, or more than kCap candidates) the finishing
// CTA selects over the whole row itself: slower, same result.
#include <cooperative_groups.h>

#include <cmath>

#include "sd_attend.cuh"
#include "sd_planes.cuh"

namespace sd {

constexpr int kCap = 8192;          // candidates a finishing CTA holds in shared memory
constexpr int kFinThreads = 256;
constexpr int kChunk = 8192;        // units per CTA in the multi-CTA steps
constexpr int kDigit = 11;
constexpr int kBins = 1 << kDigit;

struct RowState {   // written by the sample CTA before the filter reads it
  uint32_t nan;      // a NaN was seen (sample or filter)
  uint32_t thresh;   // estimate (T_key, i_max): unit u = lead + i is a candidate iff
  uint32_t imax;     //   key > T_key, or key == T_key and i <= i_max
  uint32_t ncand;    // candidates appended by the filter (may exceed kCap)
  uint32_t pad[12];
};

struct Ws {
  RowState* st;      // [rows]
  uint64_t* cand;    // [rows][kCap]: (key << 32) | unit
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static Ws carve(void* base, int64_t rows) {
  uint8_t* p = (uint8_t*)base;
  Ws w;
  w.st = (RowState*)p;
  p += align256(sizeof(RowState) * rows);
  w.cand = (uint64_t*)p;
  return w;
}

size_t topk_workspace_bytes(int64_t rows, int64_t n_units, const sd_select&) {
  if (n_units <= kSmallRow) return 0;
  return align256(sizeof(RowState) * rows) + align256(sizeof(uint64_t) * kCap * rows);
}

struct Geo {  // per-row candidate geometry
  int64_t n_units, n_tokens;
  int lead, tail, M, k, block;
  int r_sample;   // sample rank of the estimate (sample kernel), computed on the host
  int r_cluster;  // the same for the cluster kernel's sample
};

// Rank in a sample of S (out of M candidates) whose key is a safe estimate of the
// k-th largest: mu = k S / M members of the top k are expected in the sample, and
// r = mu + 5 sqrt(mu) + 2 exceeds their count except with negligible probability.
// Host-side: this GPU's double-precision rate is far too low for per-thread use.
static int sample_rank(int64_t k, int64_t S, int64_t M) {
  const double mu = (double)k * (double)S / (double)M;
  const double r = std::ceil(mu + 5.0 * std::sqrt(mu) + 2.0);
  return (int)(r < (double)S ? r : (double)S);
}

__host__ __device__ inline Geo make_geo(int64_t n_units, int64_t n_tokens, const sd_select& s) {
  Geo g;
  g.n_units = n_units;
  g.n_tokens = n_tokens;
  g.lead = (int)imin64(s.sink, n_units);
  g.tail = (int)imax64(n_units - s.local, g.lead);
  g.M = g.tail - g.lead;
  g.k = s.k;
  g.block = s.block;
  g.r_sample = g.r_cluster = 0;
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

// hist[bin] += 1 for every lane with `in` (all 32 lanes call it).  Plain shared
// atomics: measured faster here than aggregating equal bins with match.any, whose
// cost grows with the number of distinct bins in the warp.
__device__ __forceinline__ void hist_add(uint32_t* hist, bool in, uint32_t bin) {
  if (in) atomicAdd(&hist[bin], 1u);
}

// Sorts the nsel distinct units sel[0..nsel) (all < 2^ubits) ascending: a counting
// sort on the top 10 bits (1024 buckets), then each bucket -- usually 0 to 2
// units -- sorted by one thread.  tmp holds >= 2048 words, out >= nsel words.
template <int NT>
__device__ void sort_units(uint32_t* sel, int nsel, int ubits, uint32_t* tmp, uint32_t* out) {
  constexpr int kB = 1024;
  const int shift = ubits > 10 ? ubits - 10 : 0;
  uint32_t* cnt = tmp;         // [kB] counts, then running cursors
  uint32_t* start = tmp + kB;  // [kB] bucket starts
  __shared__ uint32_t wsum[NT / 32];
  for (int b = threadIdx.x; b < kB; b += NT) cnt[b] = 0;
  __syncthreads();
  for (int e = threadIdx.x; e < nsel; e += NT) atomicAdd(&cnt[sel[e] >> shift], 1u);
  __syncthreads();
  // exclusive scan of cnt into start: each thread owns kB / NT consecutive buckets
  constexpr int PER = kB / NT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t loc[PER], tot = 0, most = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    loc[i] = cnt[threadIdx.x * PER + i];
    tot += loc[i];
    most = max(most, loc[i]);
  }
  if (__syncthreads_or(most > 32)) {  // clustered units: bitonic sort instead
    int n2 = 1;
    while (n2 < nsel) n2 <<= 1;
    for (int i = nsel + threadIdx.x; i < n2; i += NT) sel[i] = 0xFFFFFFFFu;
    __syncthreads();
    bitonic_sort_u32<NT>(sel, n2);
    return;
  }
  uint32_t incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  uint32_t run = incl - tot;
  for (int w = 0; w < warp; ++w) run += wsum[w];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    start[threadIdx.x * PER + i] = run;
    cnt[threadIdx.x * PER + i] = run;
    run += loc[i];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < nsel; e += NT) {
    const uint32_t u = sel[e];
    out[atomicAdd(&cnt[u >> shift], 1u)] = u;
  }
  __syncthreads();
  for (int b = threadIdx.x; b < kB; b += NT) {  // cnt[b] is now the bucket's end
    const int s0 = (int)start[b], s1 = (int)cnt[b];
    for (int i = s0 + 1; i < s1; ++i) {  // insertion sort of a short bucket
      const uint32_t x = out[i];
      int j = i - 1;
      while (j >= s0 && out[j] > x) { out[j + 1] = out[j]; --j; }
      out[j + 1] = x;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < nsel; e += NT) sel[e] = out[e];
  __syncthreads();
}

// Finds T such that exactly `need` of the c unique values C[0..c) are >= T,
// given that all of them equal `prefix` in the bits above `pos`.
template <int NT, typename KT>
__device__ uint64_t radix_threshold(const KT* C, int c, uint32_t need, uint64_t prefix,
                                    int pos, uint32_t* hist, uint32_t* scratch, uint32_t* out,
                                    int max_passes = 64) {
  uint32_t r = need;
  for (int pass = 0; pos > 0 && pass < max_passes; ++pass) {
    const int w = min(kDigit, pos);
    const int npos = pos - w;
    for (int b = threadIdx.x; b < kBins; b += NT) hist[b] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < c; i0 += NT) {  // warp-uniform trip count for the match below
      const int i = i0 + threadIdx.x;
      bool in = false;
      uint32_t bin = 0;
      if (i < c) {
        const uint64_t x = (uint64_t)C[i];
        in = (x >> pos) == prefix;
        bin = (uint32_t)(x >> npos) & ((1u << w) - 1);
      }
      hist_add(hist, in, bin);
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
// tail units) expanded to tokens, and the count: thread t of nt threads.
__device__ void write_units_by(const Geo& g, const uint32_t* sel, int nsel, int32_t* idx_row,
                               int32_t* count_row, int t, int nt) {
  const int ntail = (int)(g.n_units - g.tail);
  const int nunits = g.lead + nsel + ntail;
  const int blk = g.block;
  const int total = nunits * blk;  // <= idx_stride < 2^31
  const int ntok = (int)g.n_tokens;
  const int sh = (blk & (blk - 1)) == 0 ? __ffs(blk) - 1 : -1;  // power-of-two blocks shift
#pragma unroll 4
  for (int p = t; p < total; p += nt) {
    const int ui = sh >= 0 ? p >> sh : p / blk;
    const int off = p - ui * blk;
    const int u = ui < g.lead ? ui : (ui < g.lead + nsel ? (int)sel[ui - g.lead]
                                                        : g.tail + (ui - g.lead - nsel));
    const int tok = u * blk + off;
    if (tok < ntok) idx_row[p] = tok;
  }
  if (t == 0) {
    const bool last_in = ntail > 0 || (nsel > 0 && (int64_t)sel[nsel - 1] == g.n_units - 1) ||
                         (nsel == 0 && ntail == 0 && g.lead == g.n_units);
    int64_t cnt = total;
    if (last_in) cnt -= (g.n_units * g.block - g.n_tokens);
    *count_row = (int32_t)cnt;
  }
}

template <int NT>
__device__ void write_units(const Geo& g, const uint32_t* sel, int nsel, int32_t* idx_row,
                            int32_t* count_row) {
  write_units_by(g, sel, nsel, idx_row, count_row, threadIdx.x, NT);
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
  sort_units<kFinThreads>(S.sel, nsel, bits_of((uint32_t)(g.n_units - 1)), S.hist,
                          reinterpret_cast<uint32_t*>(S.C));
  write_units<kFinThreads>(g, S.sel, nsel, idx_row, count + row);
}

// --------------------------------------------------------------------------------------
// Rows of at most kRegRow candidates: one CTA of 4 warps per row, keys in registers.
// --------------------------------------------------------------------------------------
// Warp w holds candidates [w * 32 JW, (w + 1) * 32 JW); candidate i = w * 32 JW +
// j * 32 + lane sits in key[j] of that lane (coalesced loads).  The k-th largest
// key T is found bit by bit from the most significant bit in which the row's keys
// differ: T | bit is kept while at least k keys are >= it.  Each lane counts with
// borrow arithmetic (no compares, no predicates), each warp sums its lanes, and the
// four warp sums meet in a double-buffered shared slot behind one barrier per bit.
// Every key > T is taken, and of the keys == T the lowest-indexed k - #(key > T):
// the composite order of the other kernels, with no 64-bit keys.  One exchange of
// per-warp counts then gives each warp the place of its first taken unit and its
// first tie's rank; walking j upward, ballots place each taken unit, so the units
// come out ascending with no sort, and the lane that takes a unit writes its tokens.
// A single warp per row is latency-bound here (about one instruction per three
// cycles with no other warp to switch to), hence four.
constexpr int kRegRow = 2048;
constexpr int kRegWarps = 4;

// 1 if a < b (unsigned), from the borrow of a - b: no compare, no predicate
__device__ __forceinline__ uint32_t borrow_of(uint32_t a, uint32_t b) {
  return ((~a & b) | (~(a ^ b) & (a - b))) >> 31;
}

// Tokens of unit u at output position pos (units are blk tokens; the last may be
// cut at ntok): 16-byte stores when the row allows them.
__device__ __forceinline__ void put_unit(int32_t* idx_row, int pos, int u, int blk, int ntok,
                                         bool vec) {
  const int t0 = u * blk;
  int32_t* dst = idx_row + (int64_t)pos * blk;
  if (vec && t0 + blk <= ntok) {
    for (int o = 0; o < blk; o += 4)
      *reinterpret_cast<int4*>(dst + o) = make_int4(t0 + o, t0 + o + 1, t0 + o + 2, t0 + o + 3);
  } else {
    for (int o = 0; o < blk && t0 + o < ntok; ++o) dst[o] = t0 + o;
  }
}

template <bool F32, int JW>
__global__ void __launch_bounds__(kRegWarps * 32)
topk_reg_kernel(const void* __restrict__ scores, Geo g, int32_t* __restrict__ idx,
                int64_t idx_stride, int32_t* __restrict__ count) {
  __shared__ uint32_t xch[2][kRegWarps];            // per-bit warp sums, double-buffered
  __shared__ uint32_t mm[2][kRegWarps];             // warp minima and maxima
  __shared__ uint32_t gt_tie[2][kRegWarps];         // warp counts of key > T and key == T
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t row = blockIdx.x;
  const int M = g.M;
  const int u0 = w * 32 * JW;  // this warp's first candidate
  const int64_t base = row * g.n_units + g.lead;
  uint32_t key[JW];
  bool nan = false;
  uint32_t mn = 0xFFFFFFFFu, mx = 0;
  if (M > 0) {
    // addresses clamped into the row, so no load waits on a branch: all in flight
#pragma unroll
    for (int j = 0; j < JW; ++j) {
      const int i = u0 + j * 32 + lane;
      const bool valid = i < M;
      bool nj = false;
      const uint32_t kk = load_key<F32>(scores, base + min(i, M - 1), nj);
      nan = nan || (nj && valid);
      key[j] = valid ? kk : 0u;
      mn = valid ? min(mn, kk) : mn;
      mx = valid ? max(mx, kk) : mx;
    }
  }
  if (__syncthreads_or(nan)) {
    if (threadIdx.x == 0) count[row] = -1;
    return;
  }
  const bool all = M <= g.k;  // every candidate is taken
  int ties = 0, nsel = 0;     // ties and taken units before this warp's first candidate
  uint32_t T = 0;
  int need = 0;               // keys == T taken, lowest index first
  if (!all) {                 // M >= 1 here
    mn = __reduce_min_sync(0xFFFFFFFFu, mn);
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if (lane == 0) { mm[0][w] = mn; mm[1][w] = mx; }
    __syncthreads();
#pragma unroll
    for (int v = 0; v < kRegWarps; ++v) { mn = min(mn, mm[0][v]); mx = max(mx, mm[1][v]); }
    if (mn == mx) {
      T = mn;
    } else {
      // every key shares the bits of mn above hb, so the k-th largest does too;
      // T | bit >= 1 counts the zero padding of i >= M as below it
      const int hb = 31 - __clz(mn ^ mx);
      T = hb == 31 ? 0u : mn & ~((2u << hb) - 1u);
      const int max_below = kRegWarps * 32 * JW - g.k;  // keep T | bit while #(key < it) <= this
      for (int b = hb; b >= 0; --b) {
        const uint32_t c = T | (1u << b);
        uint32_t n_lt[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < JW; ++j) n_lt[j & 1] += borrow_of(key[j], c);
        const uint32_t n = __reduce_add_sync(0xFFFFFFFFu, n_lt[0] + n_lt[1]);
        if (lane == 0) xch[b & 1][w] = n;
        __syncthreads();  // a slot is rewritten two bits later, after another barrier
        uint32_t tot = 0;
#pragma unroll
        for (int v = 0; v < kRegWarps; ++v) tot += xch[b & 1][v];
        if ((int)tot <= max_below) T = c;
      }
    }
    uint32_t n_gt = 0, n_tie = 0;
#pragma unroll
    for (int j = 0; j < JW; ++j) {
      n_gt += key[j] > T ? 1u : 0u;
      n_tie += (key[j] == T && u0 + j * 32 + lane < M) ? 1u : 0u;
    }
    n_gt = __reduce_add_sync(0xFFFFFFFFu, n_gt);
    n_tie = __reduce_add_sync(0xFFFFFFFFu, n_tie);
    if (lane == 0) { gt_tie[0][w] = n_gt; gt_tie[1][w] = n_tie; }
    __syncthreads();
    int gt_all = 0;
#pragma unroll
    for (int v = 0; v < kRegWarps; ++v) gt_all += (int)gt_tie[0][v];
    need = g.k - gt_all;
    for (int v = 0; v < w; ++v) {
      const int tv = (int)gt_tie[1][v];
      nsel += (int)gt_tie[0][v] + max(0, min(tv, need - ties));
      ties += tv;
    }
  } else {
    nsel = min(M, u0);
  }
  const int nsel_all = min(M, g.k);
  int32_t* idx_row = idx + row * idx_stride;
  const int blk = g.block, ntok = (int)g.n_tokens;
  const bool vec = (blk & 3) == 0 && (reinterpret_cast<uintptr_t>(idx_row) & 15) == 0;
  const uint32_t lt = (1u << lane) - 1u;
  const bool last_cand = g.tail == g.n_units && M > 0;  // the row's last unit competes
  bool last_taken = false;
#pragma unroll
  for (int j = 0; j < JW; ++j) {
    const int i = u0 + j * 32 + lane;
    const bool valid = i < M;
    bool take;
    if (all) {
      take = valid;
    } else {
      const bool tie = valid && key[j] == T;
      const uint32_t bt = __ballot_sync(0xFFFFFFFFu, tie);
      take = valid && (key[j] > T || (tie && ties + __popc(bt & lt) < need));
      ties += __popc(bt);
    }
    const uint32_t bs = __ballot_sync(0xFFFFFFFFu, take);
    if (take) put_unit(idx_row, g.lead + nsel + __popc(bs & lt), g.lead + i, blk, ntok, vec);
    if (take && i == M - 1) last_taken = true;
    nsel += __popc(bs);
  }
  // the forced windows: units [0, lead) first, then [tail, n_units) after the taken
  const int lead_tok = g.lead * blk;
  for (int p = threadIdx.x; p < lead_tok && p < ntok; p += kRegWarps * 32) idx_row[p] = p;
  const int ntail = (int)(g.n_units - g.tail);
  const int tail0 = (g.lead + nsel_all) * blk, tail_tok = ntail * blk;
  for (int q = threadIdx.x; q < tail_tok && g.tail * blk + q < ntok; q += kRegWarps * 32)
    idx_row[tail0 + q] = g.tail * blk + q;
  // the count: less the cut of the last unit when that unit is in the output
  const int64_t cut = g.n_units * g.block - g.n_tokens;
  const int64_t total = (int64_t)(g.lead + nsel_all + ntail) * blk;
  if (last_cand) {
    const int owner = (M - 1) / (32 * JW) * 32 + (M - 1) % 32;  // thread holding candidate M - 1
    if ((int)threadIdx.x == owner) count[row] = (int32_t)(last_taken ? total - cut : total);
  } else if (threadIdx.x == 0) {
    const bool last_in = ntail > 0 || (M == 0 && g.lead == g.n_units);
    count[row] = (int32_t)(last_in ? total - cut : total);
  }
}

template <bool F32, int JW>
static int launch_topk_reg(const void* scores, int64_t rows, const Geo& g, int32_t* idx,
                           int64_t idx_stride, int32_t* count, cudaStream_t st) {
  topk_reg_kernel<F32, JW><<<(unsigned)rows, kRegWarps * 32, 0, st>>>(scores, g, idx, idx_stride,
                                                                      count);
  note_launches(1);
  return check_launch("topk_reg");
}

template <bool F32>
static int topk_reg(const void* scores, int64_t rows, const Geo& g, int32_t* idx,
                    int64_t idx_stride, int32_t* count, cudaStream_t st) {
  if (g.M <= 128) return launch_topk_reg<F32, 1>(scores, rows, g, idx, idx_stride, count, st);
  if (g.M <= 256) return launch_topk_reg<F32, 2>(scores, rows, g, idx, idx_stride, count, st);
  if (g.M <= 512) return launch_topk_reg<F32, 4>(scores, rows, g, idx, idx_stride, count, st);
  if (g.M <= 1024) return launch_topk_reg<F32, 8>(scores, rows, g, idx, idx_stride, count, st);
  return launch_topk_reg<F32, 16>(scores, rows, g, idx, idx_stride, count, st);
}

// --------------------------------------------------------------------------------------
// Long rows: sample -> filter -> finish.
// --------------------------------------------------------------------------------------
// The sample CTA estimates a threshold T_est with at least k keys >= T_est from an
// evenly spaced sample; the filter appends every key >= T_est (with its unit) to
// the row's candidate list; the finishing CTA selects exactly among them.  When
// the estimate misses (fewer than k or more than kCap candidates) the finishing
// CTA selects over the whole row itself.  Only speed depends on the sample.
constexpr int kSample = 8192;  // largest sample (composite keys held in shared memory)

__host__ __device__ inline int sample_size(const Geo& g) {
  int64_t s = g.k * 4 > 4096 ? (int64_t)g.k * 4 : 4096;
  if (s > kSample) s = kSample;
  return (int)imin64(g.M, s);
}

// The estimate is taken on composite keys (unique, ties broken by index), so the
// candidate count stays near r * M / sample even when a huge group of units ties
// on one score (integer Hamming scores do).  Two 11-bit radix passes suffice: the
// lower bound of the bucket that holds the r-th largest sample is a valid estimate
// (at least r sampled keys are >= it).
template <bool F32>
__global__ void __launch_bounds__(kFinThreads)
topk_sample_kernel(const void* __restrict__ scores, Geo g, Ws ws) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint64_t* C = reinterpret_cast<uint64_t*>(smem_raw);  // [kSample]
  uint32_t* hist = reinterpret_cast<uint32_t*>(C + kSample);  // [kBins]
  __shared__ uint32_t scratch[32], out[4], kmin_s, kmax_s;
  __shared__ int nan_s;
  const int64_t row = blockIdx.x;
  RowState& st = ws.st[row];
  if (threadIdx.x == 0) { nan_s = 0; kmin_s = 0xFFFFFFFFu; kmax_s = 0; }
  __syncthreads();
  const int S = sample_size(g);
  // sample i sits at unit lead + floor(i * step), step = M / S in 32.32 fixed point
  const uint64_t step = ((uint64_t)g.M << 32) / (uint64_t)S;
  const float* fs = reinterpret_cast<const float*>(scores) + row * g.n_units + g.lead;
  const int32_t* is = reinterpret_cast<const int32_t*>(scores) + row * g.n_units + g.lead;
  bool nan = false;
  uint32_t mn = 0xFFFFFFFFu, mx = 0;
  constexpr int kBatch = 8;  // independent loads in flight per thread
  for (int i0 = 0; i0 < S; i0 += kFinThreads * kBatch) {
    uint32_t v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * kFinThreads + threadIdx.x;
      if (i < S) {
        const uint32_t iu = (uint32_t)(((uint64_t)i * step) >> 32);
        if (F32) {
          const float f = __ldg(fs + iu);
          if ((__float_as_uint(f) & 0x7FFFFFFFu) > 0x7F800000u) nan = true;
          v[u] = key_of_f32(f);
        } else {
          v[u] = key_of_i32(__ldg(is + iu));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * kFinThreads + threadIdx.x;
      if (i < S) {
        C[i] = v[u];
        mn = min(mn, v[u]);
        mx = max(mx, v[u]);
      }
    }
  }
  if (nan) nan_s = 1;
  atomicMin(&kmin_s, mn);
  atomicMax(&kmax_s, mx);
  __syncthreads();
  const int r = g.r_sample;
  uint32_t T_key = 0, imax = (uint32_t)g.M;  // default: every unit is a candidate
  if (!nan_s && g.M > g.k && r < S) {
    const uint32_t kmin = kmin_s;
    const int bI = bits_of((uint32_t)(g.M - 1));
    const int nb = bits_of(kmax_s - kmin) + bI;
    for (int i = threadIdx.x; i < S; i += kFinThreads) {
      const uint32_t iu = (uint32_t)(((uint64_t)i * step) >> 32);  // sampled unit - lead
      C[i] = ((uint64_t)((uint32_t)C[i] - kmin) << bI) | (uint64_t)((uint32_t)(g.M - 1) - iu);
    }
    __syncthreads();
    const uint64_t T = radix_threshold<kFinThreads>(C, S, (uint32_t)r, 0, nb, hist, scratch, out, 2);
    T_key = kmin + (uint32_t)(T >> bI);
    imax = (uint32_t)(g.M - 1) - (uint32_t)(T & ((1ull << bI) - 1));
  }
  if (threadIdx.x == 0) {
    st.nan = nan_s;
    st.thresh = T_key;
    st.imax = imax;
    st.ncand = 0;
  }
}

// One pass over the row: every unit with (key, index) at or above the estimate
// is appended with its key; 8 groups of 4 units per thread are loaded up front.
constexpr int kFilterGroups = kChunk / (256 * 4);

template <bool F32>
__global__ void __launch_bounds__(256)
topk_filter_kernel(const void* __restrict__ scores, Geo g, Ws ws, bool vec) {
  const int64_t row = blockIdx.y;
  RowState& st = ws.st[row];
  if (st.nan || g.M <= g.k) return;
  const uint32_t T = st.thresh;
  const uint32_t imax = st.imax;
  uint64_t* cand = ws.cand + row * kCap;
  const int lane = threadIdx.x & 31;
  const float* frow = reinterpret_cast<const float*>(scores) + row * g.n_units;
  const int32_t* irow = reinterpret_cast<const int32_t*>(scores) + row * g.n_units;
  const int lead = g.lead, tail = g.tail, nu = (int)g.n_units;
  const int a0 = (lead & ~3) + (int)blockIdx.x * kChunk;  // aligned chunk start
  uint32_t kk[kFilterGroups][4];
  bool nan = false;
#pragma unroll
  for (int gi = 0; gi < kFilterGroups; ++gi) {
    const int gs = a0 + (gi * 256 + (int)threadIdx.x) * 4;
    if (vec && gs + 4 <= nu) {
      if (F32) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(frow + gs));
        const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          kk[gi][e] = key_of_f32(f[e]);
          if ((__float_as_uint(f[e]) & 0x7FFFFFFFu) > 0x7F800000u && gs + e >= lead && gs + e < tail)
            nan = true;
        }
      } else {
        const int4 v = __ldg(reinterpret_cast<const int4*>(irow + gs));
        kk[gi][0] = key_of_i32(v.x); kk[gi][1] = key_of_i32(v.y);
        kk[gi][2] = key_of_i32(v.z); kk[gi][3] = key_of_i32(v.w);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kk[gi][e] = 0u;
        if (gs + e >= lead && gs + e < tail) {
          if (F32) {
            const float f = __ldg(frow + gs + e);
            if ((__float_as_uint(f) & 0x7FFFFFFFu) > 0x7F800000u) nan = true;
            kk[gi][e] = key_of_f32(f);
          } else {
            kk[gi][e] = key_of_i32(__ldg(irow + gs + e));
          }
        }
      }
    }
  }
  if (nan) atomicOr(&st.nan, 1u);
#pragma unroll
  for (int gi = 0; gi < kFilterGroups; ++gi) {
    const int gs = a0 + (gi * 256 + (int)threadIdx.x) * 4;
    uint32_t hit = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int u = gs + e;
      const bool inr = u >= lead && u < tail;
      const uint32_t k = kk[gi][e];
      if (inr && (k > T || (k == T && (uint32_t)(u - lead) <= imax))) hit |= 1u << e;
    }
    if (!__any_sync(0xFFFFFFFFu, hit != 0)) continue;
    const uint32_t mine = __popc(hit);
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
    uint32_t basep = 0;
    if (lane == 31) basep = atomicAdd(&st.ncand, tot);
    basep = __shfl_sync(0xFFFFFFFFu, basep, 31) + incl - mine;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (hit & (1u << e)) {
        if (basep < (uint32_t)kCap) cand[basep] = ((uint64_t)kk[gi][e] << 32) | (uint32_t)(gs + e);
        ++basep;
      }
  }
}

// Finishes a row whose c candidates (key << 32 | unit) are in S.C: the exact top k
// among them when c >= k and they all fit (c <= kCap), else an exact selection
// over the whole row in this CTA; then sorts and writes the units.  (Every
// thread of the CTA calls it; S.nsel is zero and M > k.)
template <bool F32, int NT>
__device__ void finish_row(FinSmem& S, const void* __restrict__ scores, const Geo& g,
                           int64_t row, uint32_t c, int32_t* __restrict__ idx_row,
                           int32_t* __restrict__ count_row) {
  const int bI = bits_of((uint32_t)(g.M - 1));
  const uint64_t imask = (1ull << bI) - 1;
  if (threadIdx.x == 0) { S.kmin = 0xFFFFFFFFu; S.kmax = 0; }
  __syncthreads();
  if (c >= (uint32_t)g.k && c <= (uint32_t)kCap) {
    uint32_t mn = 0xFFFFFFFFu, mx = 0;
    for (uint32_t i = threadIdx.x; i < c; i += NT) {
      const uint32_t kk = (uint32_t)(S.C[i] >> 32);
      mn = min(mn, kk);
      mx = max(mx, kk);
    }
    atomicMin(&S.kmin, mn);
    atomicMax(&S.kmax, mx);
    __syncthreads();
    const uint32_t kmin = S.kmin;
    const int nb = bits_of(S.kmax - kmin) + bI;
    for (uint32_t i = threadIdx.x; i < c; i += NT) {
      uint64_t x = S.C[i];
      uint32_t u = (uint32_t)x;
      S.C[i] = ((uint64_t)((uint32_t)(x >> 32) - kmin) << bI) | (uint64_t)(g.M - 1 - (u - g.lead));
    }
    __syncthreads();
    const uint64_t T = radix_threshold<NT>(S.C, (int)c, (uint32_t)g.k, 0, nb, S.hist, S.scratch,
                                           S.out);
    for (uint32_t i = threadIdx.x; i < c; i += NT) {
      uint64_t x = S.C[i];
      if (x >= T) S.sel[atomicAdd(&S.nsel, 1u)] = g.lead + (g.M - 1 - (uint32_t)(x & imask));
    }
  } else {
    // The estimate missed: exact selection over the whole row in this CTA.
    bool nan = false;
    uint32_t mn = 0xFFFFFFFFu, mx = 0;
    for (int64_t i = threadIdx.x; i < g.M; i += NT) {
      uint32_t kk = load_key<F32>(scores, row * g.n_units + g.lead + i, nan);
      mn = min(mn, kk);
      mx = max(mx, kk);
    }
    atomicMin(&S.kmin, mn);
    atomicMax(&S.kmax, mx);
    __syncthreads();
    const uint32_t kmin = S.kmin;
    const int nb = bits_of(S.kmax - kmin) + bI;
    uint64_t prefix = 0;
    int pos = nb;
    uint32_t r = (uint32_t)g.k;
    while (pos > 0) {
      const int w = min(kDigit, pos);
      const int npos = pos - w;
      for (int b = threadIdx.x; b < kBins; b += NT) S.hist[b] = 0;
      __syncthreads();
      for (int64_t i = threadIdx.x; i < g.M; i += NT) {
        uint32_t kk = load_key<F32>(scores, row * g.n_units + g.lead + i, nan);
        uint64_t x = ((uint64_t)(kk - kmin) << bI) | (uint64_t)(g.M - 1 - i);
        if ((x >> pos) == prefix) atomicAdd(&S.hist[(uint32_t)(x >> npos) & ((1u << w) - 1)], 1u);
      }
      __syncthreads();
      pick_digit<NT>(S.hist, r, S.scratch, S.out);
      const uint32_t dd = S.out[0], ab = S.out[1], inb = S.hist[dd];
      __syncthreads();
      r -= ab;
      prefix = (prefix << w) | dd;
      pos = npos;
      if (inb == r) break;
    }
    const uint64_t T = prefix << pos;
    for (int64_t i = threadIdx.x; i < g.M; i += NT) {
      uint32_t kk = load_key<F32>(scores, row * g.n_units + g.lead + i, nan);
      uint64_t x = ((uint64_t)(kk - kmin) << bI) | (uint64_t)(g.M - 1 - i);
      if (x >= T) S.sel[atomicAdd(&S.nsel, 1u)] = (uint32_t)(g.lead + i);
    }
  }
  __syncthreads();
  const int nsel = (int)S.nsel;
  sort_units<NT>(S.sel, nsel, bits_of((uint32_t)(g.n_units - 1)), S.hist,
                 reinterpret_cast<uint32_t*>(S.C));
  write_units<NT>(g, S.sel, nsel, idx_row, count_row);
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
  const uint32_t c = st.ncand;
  if (c >= (uint32_t)g.k && c <= (uint32_t)kCap) {
    const uint64_t* cand = ws.cand + row * kCap;
    for (uint32_t i = threadIdx.x; i < c; i += kFinThreads) S.C[i] = cand[i];
  }
  finish_row<F32, kFinThreads>(S, scores, g, row, c, idx_row, count + row);
}

// The fused scan + top-k's selection: one CTA per row gathers the units the scan
// marked (PsCand hit masks) as its candidates, then finishes the row.
constexpr int kMarkThreads = 1024;

template <bool F32>
__global__ void __launch_bounds__(kMarkThreads)
topk_marked_kernel(const void* __restrict__ scores, Geo g, const uint32_t* __restrict__ hits,
                   const uint32_t* __restrict__ cnan, int64_t n32, int32_t* __restrict__ idx,
                   int64_t idx_stride, int32_t* __restrict__ count) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  FinSmem& S = *reinterpret_cast<FinSmem*>(smem_raw);
  const int64_t row = blockIdx.x;
  int32_t* idx_row = idx + row * idx_stride;
  if (__ldg(cnan + row)) {
    if (threadIdx.x == 0) count[row] = -1;
    return;
  }
  if (threadIdx.x == 0) { S.nsel = 0; S.flag = 0; }
  __syncthreads();
  const float* frow = reinterpret_cast<const float*>(scores) + row * g.n_units;
  const int32_t* irow = reinterpret_cast<const int32_t*>(scores) + row * g.n_units;
  const uint32_t* hrow = hits + row * n32;
  for (int64_t w = threadIdx.x; w < n32; w += kMarkThreads) {
    uint32_t m = __ldg(hrow + w);
    while (m) {
      const uint32_t u = (uint32_t)(w * 32) + (uint32_t)(__ffs(m) - 1);
      m &= m - 1;
      const uint32_t key = F32 ? key_of_f32(__ldg(frow + u)) : key_of_i32(__ldg(irow + u));
      const uint32_t p = atomicAdd(&S.flag, 1u);
      if (p < (uint32_t)kCap) S.C[p] = ((uint64_t)key << 32) | u;
    }
  }
  __syncthreads();
  finish_row<F32, kMarkThreads>(S, scores, g, row, S.flag, idx_row, count + row);
}

// --------------------------------------------------------------------------------------
// Long rows, one launch: a thread-block cluster of CS CTAs per row.
// --------------------------------------------------------------------------------------
// The same three steps as above, but the CTAs of a row share distributed shared
// memory and cluster barriers instead of global memory and kernel boundaries:
//   1. each CTA samples its share of the evenly spaced positions; the composite
//      keys are gathered in CTA 0, which picks the estimate (T_key, i_max);
//   2. each CTA filters its slice of the row into a local candidate list; the
//      lists are gathered in CTA 0, which selects exactly (radix over composite
//      keys) and broadcasts the exact threshold;
//   3. each CTA keeps its own candidates above the threshold, sorts them (they lie
//      in its slice, so the slices' lists concatenate in ascending order) and
//      writes them at the offset given by the ranks before it.
// If the estimate admits fewer than k or too many candidates, step 2 is replaced
// by an exact radix select over the whole row, distributed over the cluster (each
// CTA histograms its slice, the histograms are summed in CTA 0).
namespace cg = cooperative_groups;
constexpr int kLocCap = 2048;  // local candidates per CTA of a cluster
constexpr int kClThreads = 1024;
constexpr int kClBuf = kCap;   // CTA 0's gather buffer (samples, then candidates)

struct ClSmem {
  uint64_t buf[kClBuf];    // CTA 0: gathered samples, then gathered candidates / row histogram
  uint64_t cand[kLocCap];  // local candidates (key << 32 | unit); samples in step 1
  uint32_t sel[kMaxTopK];  // local selected units
  uint32_t hist[kBins];
  uint32_t scratch[32], out[4];
  uint32_t kmin, kmax, nan, nbuf, ovf, ncand, nsel, mode;
  uint32_t T_key, imax;
  uint32_t cnt[16];
  uint32_t pwh[(kClThreads / 32) * 256];  // per-warp radix histograms
};

// 4096 samples (2k for large k) keep the candidates near 3K at k = 512 and within
// the gather buffer up to k = 4096, while the estimate's serial radix stays short
__host__ __device__ inline int cluster_sample_size(const Geo& g) {
  const int64_t s = g.k * 2 > 4096 ? (int64_t)g.k * 2 : 4096;
  return (int)imin64(g.M, imin64(s, kClBuf));
}


template <bool F32>
__device__ __forceinline__ uint32_t key_at(const float* frow, const int32_t* irow, int64_t u,
                                           bool& nan) {
  if (F32) {
    const float f = __ldg(frow + u);
    if ((__float_as_uint(f) & 0x7FFFFFFFu) > 0x7F800000u) nan = true;
    return key_of_f32(f);
  }
  return key_of_i32(__ldg(irow + u));
}

// Radix select over 8-bit digits with per-warp private histograms (pwh: one
// 256-bin table per warp), so crowded score ranges do not serialise on shared
// atomics.  Finds T with at least `need` of C[0..c) >= T, all C < 2^nb; exact
// (exactly `need` values >= T, C unique) unless max_passes stops it first, in
// which case T is the lower bound of the bucket holding the need-th value.
template <int NT, typename KT>
__device__ uint64_t radix_select_pw(const KT* C, int c, uint32_t need, int nb,
                                    int max_passes, uint32_t* pwh, uint32_t* out) {
  constexpr int NW = NT / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* mine = pwh + warp * 256;
  uint64_t prefix = 0;
  int pos = nb;
  uint32_t r = need;
  for (int pass = 0; pos > 0 && pass < max_passes; ++pass) {
    const int w = min(8, pos), npos = pos - w;
    const uint32_t mask = (1u << w) - 1;
#pragma unroll
    for (int b = lane; b < 256; b += 32) mine[b] = 0;
    __syncwarp();
    for (int i = threadIdx.x; i < c; i += NT) {
      const uint64_t x = C[i];
      if (pos >= 64 || (x >> pos) == prefix) atomicAdd(&mine[(uint32_t)(x >> npos) & mask], 1u);
    }
    __syncthreads();
    // bin totals over the warps' tables, one bin per thread, into warp 0's table
    for (int b = threadIdx.x; b < 256; b += NT) {
      uint32_t v = 0;
#pragma unroll 8
      for (int ww = 0; ww < NW; ++ww) v += pwh[ww * 256 + b];
      pwh[b] = v;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 8l..8l+7; suffix scan over lanes
      uint32_t h[8], tot = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        h[i] = pwh[lane * 8 + i];
        tot += h[i];
      }
      uint32_t suf = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xFFFFFFFFu, suf, o);
        if (lane + o < 32) suf += y;
      }
      uint32_t above = suf - tot;  // bins of higher lanes
#pragma unroll
      for (int i = 7; i >= 0; --i) {
        if (above < r && r <= above + h[i]) { out[0] = lane * 8 + i; out[1] = above; out[2] = h[i]; }
        above += h[i];
      }
    }
    __syncthreads();
    const uint32_t d = out[0], ab = out[1], inb = out[2];
    __syncthreads();
    r -= ab;
    prefix = (prefix << w) | d;
    pos = npos;
    if (inb == r) break;
  }
  return prefix << pos;
}

template <bool F32, int CS>
__global__ void __launch_bounds__(kClThreads)
topk_cluster_kernel(const void* __restrict__ scores, Geo g, int32_t* __restrict__ idx,
                    int64_t idx_stride, int32_t* __restrict__ count) {
  constexpr int NT = kClThreads;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ClSmem& S = *reinterpret_cast<ClSmem*>(smem_raw);
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  ClSmem* S0 = cl.map_shared_rank(&S, 0);
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t row = blockIdx.y;
  const float* frow = reinterpret_cast<const float*>(scores) + row * g.n_units;
  const int32_t* irow = reinterpret_cast<const int32_t*>(scores) + row * g.n_units;
  int32_t* idx_row = idx + row * idx_stride;
  const int M = g.M, lead = g.lead, k = g.k, blk = g.block;
  const int ntail = (int)(g.n_units - g.tail);
  const int i_lo = (int)(((int64_t)rank * M) / CS), i_hi = (int)(((int64_t)(rank + 1) * M) / CS);
  const int bI = bits_of((uint32_t)(M - 1));
  const uint32_t imask = (uint32_t)((1ull << bI) - 1);

  if (tid == 0) {
    S.kmin = 0xFFFFFFFFu; S.kmax = 0; S.nan = 0; S.nbuf = 0; S.ovf = 0;
    S.ncand = 0; S.nsel = 0; S.mode = 0;
  }
  cl.sync();

  // ---- step 1: sample ----
  const int Ssz = cluster_sample_size(g);
  const uint64_t step = ((uint64_t)M << 32) / (uint64_t)Ssz;
  const int s_lo = (int)(((int64_t)rank * Ssz) / CS), s_hi = (int)(((int64_t)(rank + 1) * Ssz) / CS);
  {
    bool nan = false;
    uint32_t mn = 0xFFFFFFFFu, mx = 0;
    for (int s0 = s_lo; s0 < s_hi; s0 += NT * 4) {
      uint32_t v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int sidx = s0 + u * NT + tid;
        if (sidx < s_hi) v[u] = key_at<F32>(frow, irow, lead + (int64_t)(((uint64_t)sidx * step) >> 32), nan);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int sidx = s0 + u * NT + tid;
        if (sidx < s_hi) {
          S.cand[sidx - s_lo] = v[u];
          mn = min(mn, v[u]);
          mx = max(mx, v[u]);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
      mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    }
    if (lane == 0) {
      atomicMin(&S0->kmin, mn);
      atomicMax(&S0->kmax, mx);
    }
    if (__any_sync(0xFFFFFFFFu, nan) && lane == 0) atomicOr(&S0->nan, 1u);
  }
  cl.sync();
  if (S0->nan) {  // uniform over the cluster
    if (rank == 0 && tid == 0) count[row] = -1;
    cl.sync();
    return;
  }
  {
    const uint32_t kmin = S0->kmin;
    for (int sidx = s_lo + tid; sidx < s_hi; sidx += NT) {
      const uint32_t iu = (uint32_t)(((uint64_t)sidx * step) >> 32);
      S0->buf[sidx] = ((uint64_t)((uint32_t)S.cand[sidx - s_lo] - kmin) << bI) |
                      (uint64_t)((uint32_t)(M - 1) - iu);
    }
  }
  cl.sync();
  if (rank == 0) {
    const int r = g.r_cluster;
    uint32_t T_key = 0, imax = (uint32_t)M;
    if (r < Ssz) {
      const int nb = bits_of(S.kmax - S.kmin) + bI;
      const uint64_t T = radix_select_pw<NT>(S.buf, Ssz, (uint32_t)r, nb, 3, S.pwh, S.out);
      T_key = S.kmin + (uint32_t)(T >> bI);
      imax = (uint32_t)(M - 1) - (uint32_t)(T & imask);
    }
    if (tid == 0) { S.T_key = T_key; S.imax = imax; }
  }
  cl.sync();

  // ---- step 2: filter this CTA's slice ----
  {
    const uint32_t T = S0->T_key, imax = S0->imax;
    // the threshold in the score domain (the key map preserves order, -0 == +0)
    const float Tf = __uint_as_float((T & 0x80000000u) ? (T & 0x7FFFFFFFu) : ~T);
    const int32_t Ti = (int32_t)(T ^ 0x80000000u);
    const bool take_all = T == 0;  // key 0 is below every score's key
    bool nan = false;
    const int u_lo = lead + i_lo, u_hi = lead + i_hi;
    const int a_lo = u_lo & ~3;
    const int nu = (int)g.n_units;
    const bool vec = ((uintptr_t)frow % 16 == 0) && (nu % 4 == 0);
    constexpr int kG = 4;  // groups of 4 units per thread per batch
    // Batches are software-pipelined: batch i+1's loads are issued before batch i
    // is tested, so every thread keeps 8 to 16 loads in flight.
    const uint32_t* src = F32 ? reinterpret_cast<const uint32_t*>(frow) : reinterpret_cast<const uint32_t*>(irow);
    auto load_batch = [&](int b0, uint4 (&raw)[kG]) {
#pragma unroll
      for (int gi = 0; gi < kG; ++gi) {
        const int gs = b0 + (gi * NT + tid) * 4;
        if (vec && gs >= u_lo && gs + 4 <= u_hi) {
          raw[gi] = __ldg(reinterpret_cast<const uint4*>(src + gs));
        } else {
          raw[gi].x = (gs + 0 >= u_lo && gs + 0 < u_hi) ? __ldg(src + gs + 0) : 0u;
          raw[gi].y = (gs + 1 >= u_lo && gs + 1 < u_hi) ? __ldg(src + gs + 1) : 0u;
          raw[gi].z = (gs + 2 >= u_lo && gs + 2 < u_hi) ? __ldg(src + gs + 2) : 0u;
          raw[gi].w = (gs + 3 >= u_lo && gs + 3 < u_hi) ? __ldg(src + gs + 3) : 0u;
        }
      }
    };
    constexpr int kBatch = NT * 4 * kG;
    uint4 cur[kG], nxt[kG];
    if (a_lo < u_hi) load_batch(a_lo, cur);
    for (int b0 = a_lo; b0 < u_hi; b0 += kBatch) {  // uniform trip count
      if (b0 + kBatch < u_hi) load_batch(b0 + kBatch, nxt);
#pragma unroll
      for (int gi = 0; gi < kG; ++gi) {
        const int gs = b0 + (gi * NT + tid) * 4;
        const uint32_t rv[4] = {cur[gi].x, cur[gi].y, cur[gi].z, cur[gi].w};
        // group pre-test: almost every group lies below the threshold; only a
        // group whose maximum reaches it (or holds a NaN) is examined unit by unit
        bool maybe;
        if (F32) {
          const float m = fmax_nan(fmax_nan(__uint_as_float(rv[0]), __uint_as_float(rv[1])),
                                   fmax_nan(__uint_as_float(rv[2]), __uint_as_float(rv[3])));
          maybe = !(m < Tf);  // true for m >= Tf and for NaN
        } else {
          const int32_t m = max(max((int32_t)rv[0], (int32_t)rv[1]), max((int32_t)rv[2], (int32_t)rv[3]));
          maybe = m >= Ti;
        }
        if (!__any_sync(0xFFFFFFFFu, maybe || take_all)) continue;
        const bool inner = gs >= u_lo && gs + 4 <= u_hi;
        uint32_t hit = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          bool above, equal;
          if (F32) {
            const float f = __uint_as_float(rv[e]);
            nan |= f != f;  // masked units read 0
            above = f > Tf;
            equal = f == Tf;
          } else {
            const int32_t x = (int32_t)rv[e];
            above = x > Ti;
            equal = x == Ti;
          }
          const int u = gs + e;
          const bool in = inner || (u >= u_lo && u < u_hi);
          if (in && (take_all || above || (equal && (uint32_t)(u - lead) <= imax))) hit |= 1u << e;
        }
        if (!__any_sync(0xFFFFFFFFu, hit != 0)) continue;
        const uint32_t mine = __popc(hit);
        uint32_t incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
        uint32_t basep = 0;
        if (lane == 31) basep = atomicAdd(&S.ncand, tot);
        basep = __shfl_sync(0xFFFFFFFFu, basep, 31) + incl - mine;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (hit & (1u << e)) {
            const uint32_t key = F32 ? key_of_f32(__uint_as_float(rv[e])) : key_of_i32((int32_t)rv[e]);
            if (basep < (uint32_t)kLocCap) S.cand[basep] = ((uint64_t)key << 32) | (uint32_t)(gs + e);
            ++basep;
          }
      }
#pragma unroll
      for (int gi = 0; gi < kG; ++gi) cur[gi] = nxt[gi];
    }
    if (__any_sync(0xFFFFFFFFu, nan) && lane == 0) atomicOr(&S.nan, 1u);
  }
  __syncthreads();
  const uint32_t nloc = S.ncand;
  const uint32_t nkeep = min(nloc, (uint32_t)kLocCap);
  if (tid == 0) {
    if (S.nan) atomicOr(&S0->nan, 1u);
    if (nloc > (uint32_t)kLocCap) atomicOr(&S0->ovf, 1u);
    S.out[3] = atomicAdd(&S0->nbuf, nkeep);
  }
  __syncthreads();
  {
    const uint32_t base = S.out[3];
    for (uint32_t j = tid; j < nkeep; j += NT)
      if (base + j < (uint32_t)kClBuf) S0->buf[base + j] = S.cand[j];
  }
  cl.sync();
  if (rank == 0) {  // decide: 0 exact among candidates, 1 whole-row fallback, 2 NaN
    uint32_t mode = 0;
    const uint32_t total = S.nbuf;
    if (S.nan) mode = 2;
    else if (S.ovf || total > (uint32_t)kClBuf || total < (uint32_t)k) mode = 1;
    if (mode == 0) {
      if (tid == 0) { S.kmin = 0xFFFFFFFFu; S.kmax = 0; }
      __syncthreads();
      uint32_t mn = 0xFFFFFFFFu, mx = 0;
      for (uint32_t j = tid; j < total; j += NT) {
        const uint32_t kk = (uint32_t)(S.buf[j] >> 32);
        mn = min(mn, kk);
        mx = max(mx, kk);
      }
      atomicMin(&S.kmin, mn);
      atomicMax(&S.kmax, mx);
      __syncthreads();
      const uint32_t kmin = S.kmin;
      const int nb = bits_of(S.kmax - kmin) + bI;
      for (uint32_t j = tid; j < total; j += NT) {
        const uint64_t x = S.buf[j];
        S.buf[j] = ((uint64_t)((uint32_t)(x >> 32) - kmin) << bI) |
                   (uint64_t)((uint32_t)(M - 1) - ((uint32_t)x - (uint32_t)lead));
      }
      __syncthreads();
      const uint64_t T = radix_threshold<NT>(S.buf, (int)total, (uint32_t)k, 0, nb, S.hist,
                                             S.scratch, S.out);
      if (tid == 0) {
        S.T_key = kmin + (uint32_t)(T >> bI);
        S.imax = (uint32_t)(M - 1) - (uint32_t)(T & imask);
      }
    } else if (mode == 1) {
      uint32_t* gh = reinterpret_cast<uint32_t*>(S.buf);
      for (int b = tid; b < kBins; b += NT) gh[b] = 0;
      if (tid == 0) { S.kmin = 0xFFFFFFFFu; S.kmax = 0; }
    }
    if (tid == 0) S.mode = mode;
  }
  cl.sync();
  const uint32_t mode = S0->mode;
  if (mode == 2) {
    if (rank == 0 && tid == 0) count[row] = -1;
    cl.sync();
    return;
  }
  uint32_t T_key, imax;
  if (mode == 0) {
    T_key = S0->T_key;
    imax = S0->imax;
  } else {
    // exact radix select over the whole row, distributed over the cluster
    const int u_lo = lead + i_lo, u_hi = lead + i_hi;
    bool nan = false;
    {
      uint32_t mn = 0xFFFFFFFFu, mx = 0;
      for (int u = u_lo + tid; u < u_hi; u += NT) {
        const uint32_t kk = key_at<F32>(frow, irow, u, nan);
        mn = min(mn, kk);
        mx = max(mx, kk);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
        mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      }
      if (lane == 0) { atomicMin(&S0->kmin, mn); atomicMax(&S0->kmax, mx); }
    }
    cl.sync();
    const uint32_t kmin = S0->kmin;
    const int nb = bits_of(S0->kmax - kmin) + bI;
    uint32_t* gh0 = reinterpret_cast<uint32_t*>(S0->buf);
    uint64_t prefix = 0;
    int pos = nb;
    uint32_t r = (uint32_t)k;
    while (pos > 0) {
      const int w = min(kDigit, pos);
      const int npos = pos - w;
      for (int b = tid; b < kBins; b += NT) S.hist[b] = 0;
      __syncthreads();
      for (int u0 = u_lo; u0 < u_hi; u0 += NT) {  // uniform trip count
        const int u = u0 + tid;
        bool in = false;
        uint32_t bin = 0;
        if (u < u_hi) {
          const uint64_t x = ((uint64_t)(key_at<F32>(frow, irow, u, nan) - kmin) << bI) |
                             (uint64_t)((uint32_t)(M - 1) - (uint32_t)(u - lead));
          in = (x >> pos) == prefix;
          bin = (uint32_t)(x >> npos) & ((1u << w) - 1);
        }
        hist_add(S.hist, in, bin);
      }
      __syncthreads();
      for (int b = tid; b < kBins; b += NT)
        if (S.hist[b]) atomicAdd(&gh0[b], S.hist[b]);
      cl.sync();
      if (rank == 0) {
        pick_digit<NT>(gh0, r, S.scratch, S.out);
        if (tid == 0) S.out[2] = gh0[S.out[0]];
        __syncthreads();
        for (int b = tid; b < kBins; b += NT) gh0[b] = 0;
      }
      cl.sync();
      const uint32_t d = S0->out[0], above = S0->out[1], inb = S0->out[2];
      r -= above;
      prefix = (prefix << w) | d;
      pos = npos;
      if (inb == r) break;
    }
    const uint64_t T = prefix << pos;
    T_key = kmin + (uint32_t)(T >> bI);
    imax = (uint32_t)(M - 1) - (uint32_t)(T & imask);
  }

  // ---- step 3: keep, sort and write this CTA's share ----
  if (mode == 0) {
    for (uint32_t j = tid; j < nkeep; j += NT) {
      const uint64_t x = S.cand[j];
      const uint32_t kk = (uint32_t)(x >> 32), u = (uint32_t)x;
      if (kk > T_key || (kk == T_key && u - (uint32_t)lead <= imax))
        S.sel[atomicAdd(&S.nsel, 1u)] = u;
    }
  } else {
    bool nan = false;
    for (int u = lead + i_lo + tid; u < lead + i_hi; u += NT) {
      const uint32_t kk = key_at<F32>(frow, irow, u, nan);
      if (kk > T_key || (kk == T_key && (uint32_t)(u - lead) <= imax))
        S.sel[atomicAdd(&S.nsel, 1u)] = (uint32_t)u;
    }
  }
  __syncthreads();
  const int nsel = (int)S.nsel;
  if (tid == 0) S0->cnt[rank] = (uint32_t)nsel;
  sort_units<NT>(S.sel, nsel, bits_of((uint32_t)(g.n_units - 1)), S.hist,
                 reinterpret_cast<uint32_t*>(S.cand));
  cl.sync();
  int off = 0, ktot = 0;
  for (int q = 0; q < CS; ++q) {
    const int c = (int)S0->cnt[q];
    if (q < rank) off += c;
    ktot += c;
  }
  // units at output positions: lead units, then ranks' selections, then tail units
  for (int p = tid; p < nsel * blk; p += NT) {
    const int j = blk == 1 ? p : p / blk, o = p - j * blk;
    const int tok = (int)S.sel[j] * blk + o;
    if (tok < (int)g.n_tokens) idx_row[(int64_t)(lead + off + j) * blk + o] = tok;
  }
  if (rank == 0)
    for (int p = tid; p < lead * blk; p += NT) idx_row[p] = p;  // lead units are full blocks
  if (rank == CS - 1) {
    for (int p = tid; p < ntail * blk; p += NT) {
      const int tok = g.tail * blk + p;
      if (tok < (int)g.n_tokens) idx_row[(int64_t)(lead + ktot) * blk + p] = tok;
    }
    if (tid == 0) {
      const bool last_in = ntail > 0 || (nsel > 0 && (int64_t)S.sel[nsel - 1] == g.n_units - 1);
      int64_t cnt = (int64_t)(lead + ktot + ntail) * blk;
      if (last_in) cnt -= (g.n_units * g.block - g.n_tokens);
      count[row] = (int32_t)cnt;
    }
  }
  cl.sync();  // CTA 0's shared memory stays alive until every rank has read it
}

// How many clusters of CS CTAs can be resident at once on this device (0 if the
// configuration cannot run), cached per device.  GB300 places at most a few
// 16-CTA clusters at a time, so the launcher picks the largest CS whose clusters
// all fit in one wave.
template <bool F32, int CS>
static int cluster_capacity() {
  if (fallback_forced()) return 0;
  static std::atomic<int> cap[kMaxDev];
  return per_device_cached(cap, [] {
    auto kern = topk_cluster_kernel<F32, CS>;
    int n = 0;
    bool yes = set_smem_limit((const void*)kern, sizeof(ClSmem), "topk cluster") == SD_OK;
    if (yes && CS > 8)
      yes = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess;
    if (yes) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(CS, 1, 1);
      cfg.blockDim = dim3(kClThreads, 1, 1);
      cfg.dynamicSmemBytes = sizeof(ClSmem);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = CS;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    return n;
  });
}

template <bool F32, int CS>
static int launch_cluster(const void* scores, int64_t rows, const Geo& g, int32_t* idx,
                          int64_t idx_stride, int32_t* count, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS, (unsigned)rows, 1);
  cfg.blockDim = dim3(kClThreads, 1, 1);
  cfg.dynamicSmemBytes = sizeof(ClSmem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, topk_cluster_kernel<F32, CS>, scores, g, idx, idx_stride, count) !=
      cudaSuccess)
    return check_launch("topk_cluster");
  note_launches(1);
  return check_launch("topk_cluster");
}

// The largest cluster size whose row-clusters are all resident in one wave (0:
// no cluster configuration applies).
template <bool F32>
static int pick_cluster(int64_t rows, const Geo& g) {
  if (!(g.M > g.k && g.M >= 4 * 16 && rows <= 65535)) return 0;
  if (rows <= cluster_capacity<F32, 16>()) return 16;
  if (rows <= cluster_capacity<F32, 8>()) return 8;
  if (rows <= cluster_capacity<F32, 4>()) return 4;
  if (cluster_capacity<F32, 2>() > 0) return 2;
  return 0;
}

template <bool F32>
static int launch_cluster_cs(int cs, const void* scores, int64_t rows, const Geo& g, int32_t* idx,
                             int64_t idx_stride, int32_t* count, cudaStream_t st) {
  switch (cs) {
    case 16: return launch_cluster<F32, 16>(scores, rows, g, idx, idx_stride, count, st);
    case 8: return launch_cluster<F32, 8>(scores, rows, g, idx, idx_stride, count, st);
    case 4: return launch_cluster<F32, 4>(scores, rows, g, idx, idx_stride, count, st);
    default: return launch_cluster<F32, 2>(scores, rows, g, idx, idx_stride, count, st);
  }
}

template <bool F32>
static int topk_t(const void* scores, int64_t rows, const Geo& g, int32_t* idx,
                  int64_t idx_stride, int32_t* count, void* wsp, cudaStream_t st) {
  const size_t smem = sizeof(FinSmem);
  if (g.n_units <= kSmallRow && g.M <= kRegRow)
    return topk_reg<F32>(scores, rows, g, idx, idx_stride, count, st);
  if (g.n_units <= kSmallRow) {
    auto kern = topk_small_kernel<F32>;
    if (int rc_ = set_smem_limit((const void*)kern, smem, "topk: smem attribute")) return rc_;
    kern<<<(unsigned)rows, kFinThreads, smem, st>>>(scores, g, idx, idx_stride, count);
    note_launches(1);
    return check_launch("topk_small");
  }
  if (const int cs = pick_cluster<F32>(rows, g))
    return launch_cluster_cs<F32>(cs, scores, rows, g, idx, idx_stride, count, st);
  Ws ws = carve(wsp, rows);
  const size_t smem_s = (size_t)kSample * 8 + kBins * 4;
  auto samp = topk_sample_kernel<F32>;
  if (int rc_ = set_smem_limit((const void*)samp, smem_s, "topk: smem attribute")) return rc_;
  samp<<<(unsigned)rows, kFinThreads, smem_s, st>>>(scores, g, ws);
  const unsigned nchunks = (unsigned)((g.tail - (g.lead & ~3) + kChunk - 1) / kChunk);
  const bool vec = ((uintptr_t)scores % 16 == 0) && (g.n_units % 4 == 0);
  topk_filter_kernel<F32><<<dim3(nchunks, (unsigned)rows), 256, 0, st>>>(scores, g, ws, vec);
  auto fin = topk_finish_kernel<F32>;
  if (int rc_ = set_smem_limit((const void*)fin, smem, "topk: smem attribute")) return rc_;
  fin<<<(unsigned)rows, kFinThreads, smem, st>>>(scores, g, ws, idx, idx_stride, count);
  note_launches(3);
  return check_launch("topk");
}

int launch_topk(int score_type, const void* scores, int64_t rows, int64_t n_units,
                int64_t n_tokens, const sd_select& sel, int32_t* idx, int64_t idx_stride,
                int32_t* count, void* ws, size_t, cudaStream_t st) {
  Geo g = make_geo(n_units, n_tokens, sel);
  if (g.M > 0) {
    g.r_sample = sample_rank(g.k, sample_size(g), g.M);
    g.r_cluster = sample_rank(g.k, cluster_sample_size(g), g.M);
  }
  if (score_type == SD_SCORE_F32)
    return topk_t<true>(scores, rows, g, idx, idx_stride, count, ws, st);
  return topk_t<false>(scores, rows, g, idx, idx_stride, count, ws, st);
}

// --------------------------------------------------------------------------------------
// fp32 rows with known 32-unit maxima (sd_topk_wmax): one CTA per row.
// --------------------------------------------------------------------------------------
// A word is 32 consecutive units; its competing maximum is the largest score of its
// units inside [lead, tail).  If at least k competing units have key >= T, the
// k-th largest key is >= T, so every member of the top k has key >= T and lies in a
// word whose competing maximum is >= T.  Per row:
//   1. the keys of the words' competing maxima go to shared memory (coalesced loads;
//      the at most two words cut by lead or tail are recomputed from their scores;
//      a NaN anywhere marks the row);
//   2. T_est = a lower bound of the r-th largest key of an evenly spaced sample of
//      words (r as for the sampled top-k, mu = k S / W; two radix digits), and the
//      words whose key is >= T_est are listed in ascending order (each thread owns
//      a contiguous run of words; one block-wide scan gives the offsets);
//   3. those words' scores are read (one warp per word, one coalesced 128-byte
//      line) and every competing unit with key >= T_est becomes a candidate,
//      named by its position in the word list (list entry * 32 + unit in word),
//      which orders candidates as their units;
//   4. with at least k candidates, a radix select over (key, position descending)
//      marks the top k in a bit mask per listed word; one block-wide scan over the
//      masks' populations places them, so the units come out ascending unsorted.
// When the estimate leaves fewer than k candidates, or a list overflows, an exact
// path replaces 3-4: the k largest words by (key descending, word ascending) hold
// the top k (a unit outside them is beaten by each of their maxima: a larger key,
// or an equal key at a lower unit), and a radix select over those words' units,
// reading their scores at every pass, picks the top k; a counting sort orders them.
constexpr int kWmThreads = 1024;
constexpr int kWmWords = 36864;   // words per row (n <= ~1.18M): at most 36 per thread
constexpr int kWmMaxK = 1024;     // largest k of this path
constexpr int kWmSample = 2048;   // sampled words
constexpr int kWmCandWords = 4096;
constexpr int kWmCand = 4096;     // candidate units

struct WmSmem {
  // word keys at wpos(i); on the estimate path the selection masks (one per listed
  // word) reuse its start once the keys are no longer read
  uint32_t wk[kWmWords];  // padded runs end below kWmWords: PER + padw <= 36 per thread
  uint32_t cw[kWmCandWords];        // listed words (exact path: the k selected words)
  uint64_t ct[kWmCand];             // candidates (key << 32 | position); the sample in
                                    // step 2; the exact path's sort scratch
  uint32_t sel[kWmMaxK];
  uint32_t hist[kBins];
  uint32_t scratch[32], out[4], wsum[32];
  uint32_t nan, nct, nsel, nlist, kmin, kmax;
};

// Exclusive prefix of v over the block's threads (in thread order) and the total.
// Uses wsum[32]; contains two __syncthreads.
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* wsum, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  uint32_t w = lane < NT / 32 ? wsum[lane] : 0u, wincl = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, wincl, o);
    if (lane >= o) wincl += y;
  }
  total = __shfl_sync(0xFFFFFFFFu, wincl, 31);
  const uint32_t before = __shfl_sync(0xFFFFFFFFu, wincl - w, warp);
  __syncthreads();
  return before + incl - v;
}

// Radix select of the `need` largest of c unique 64-bit values produced by
// get(i, x) (false: i holds no value), all < 2^nb: returns T with exactly `need`
// values >= T.  11-bit digits; get is called once per value and pass.
template <int NT, class Get>
__device__ uint64_t radix_select_fn(int c, Get get, uint32_t need, int nb, uint32_t* hist,
                                    uint32_t* scratch, uint32_t* out) {
  uint64_t prefix = 0;
  int pos = nb;
  uint32_t r = need;
  while (pos > 0) {
    const int w = min(kDigit, pos), npos = pos - w;
    for (int b = threadIdx.x; b < kBins; b += NT) hist[b] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < c; i += NT) {
      uint64_t x;
      if (get(i, x) && (pos >= 64 || (x >> pos) == prefix))
        atomicAdd(&hist[(uint32_t)(x >> npos) & ((1u << w) - 1)], 1u);
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

__global__ void __launch_bounds__(kWmThreads)
topk_wmax_kernel(const float* __restrict__ scores, const float* __restrict__ wmax, Geo g,
                 int32_t* __restrict__ idx, int64_t idx_stride, int32_t* __restrict__ count) {
  constexpr int NT = kWmThreads;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  WmSmem& S = *reinterpret_cast<WmSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int64_t n = g.n_units, nw = (n + 31) >> 5;  // word maxima per row (a last word may be partial)
  const float* srow = scores + row * n;
  int32_t* idx_row = idx + row * idx_stride;
  const int lead = g.lead, tail = g.tail, M = g.M, k = g.k;
  const int w0 = lead >> 5, W = ((tail - 1) >> 5) - w0 + 1;  // words meeting [lead, tail)
  // step 2 gives each thread a run of PER words, read as 16-byte vectors; runs are
  // padded to an odd number of vectors so that a quarter warp's reads hit distinct banks
  const int PER = 4 * ((W + 4 * NT - 1) / (4 * NT));  // <= 36
  const int padw = ((PER >> 2) & 1) ? 0 : 4;          // PER + padw <= 36
  const uint32_t magic = (uint32_t)((0x100000000ull + PER - 1) / PER);  // i / PER, i < 2^16
  auto wpos = [&](int i) { return i + (int)__umulhi((uint32_t)i, magic) * padw; };
  const bool cut0 = (lead & 31) != 0, cut1 = (tail & 31) != 0;
  if (tid == 0) { S.nan = 0; S.nct = 0; S.nsel = 0; S.kmin = 0xFFFFFFFFu; S.kmax = 0; }

  // ---- 1. word keys ----
  {
    // the cut words' scores (warps 0 and 1), in flight with the maxima
    const bool cw0 = warp == 0 && cut0;
    const bool cw1 = warp == 1 && cut1 && !(cut0 && W == 1);  // W == 1: warp 0 covers both
    float xc = -INFINITY;
    if (cw0 || cw1) {
      const int u = (w0 + (cw0 ? 0 : W - 1)) * 32 + lane;
      if (u >= lead && u < tail) xc = __ldg(srow + u);
    }
    const float* base = wmax + row * nw + w0;
    constexpr int kL = kWmWords / NT;  // coalesced 4-byte loads per thread, all in flight
    float v[kL];
#pragma unroll
    for (int j = 0; j < kL; ++j) {
      const int i = j * NT + tid;
      v[j] = i < W ? __ldg(base + i) : 0.f;
    }
    bool nan = false;
#pragma unroll
    for (int j = 0; j < kL; ++j) {
      const int i = j * NT + tid;
      if (i < W) {
        if (!((i == 0 && cut0) || (i == W - 1 && cut1))) nan |= v[j] != v[j];
        S.wk[wpos(i)] = key_of_f32(v[j]);
      }
    }
    __syncthreads();
    if (cw0 || cw1) {
      nan |= xc != xc;
      float m = xc;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmax_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      if (lane == 0) S.wk[wpos(cw0 ? 0 : W - 1)] = key_of_f32(m);
    }
    if (__any_sync(0xFFFFFFFFu, nan) && lane == 0) atomicOr(&S.nan, 1u);
    __syncthreads();
  }
  if (S.nan) {
    if (tid == 0) count[row] = -1;
    return;
  }

  // ---- 2. estimate and listed words ----
  bool exact = true;
  {
    const int Ssz = min(W, kWmSample);
    uint32_t* samp = reinterpret_cast<uint32_t*>(S.ct);
    for (int s = tid; s < Ssz; s += NT) samp[s] = S.wk[wpos((int)(((int64_t)s * W) / Ssz))];
    __syncthreads();
    // two 11-bit digits: T is the low end of the 22-bit bin holding the r-th largest
    const uint32_t T = (uint32_t)radix_threshold<NT, uint32_t>(
        samp, Ssz, (uint32_t)min(g.r_sample, Ssz), 0, 32, S.hist, S.scratch, S.out, 2);
    const int i0 = tid * PER;
    const uint32_t* run = &S.wk[tid * (PER + padw)];
    uint64_t hitm = 0;
    for (int m = 0; 4 * m < PER; ++m) {
      const uint4 x = *reinterpret_cast<const uint4*>(run + 4 * m);
      const int i = i0 + 4 * m;
      const uint32_t b = (uint32_t)(x.x >= T && i < W) | ((uint32_t)(x.y >= T && i + 1 < W) << 1) |
                         ((uint32_t)(x.z >= T && i + 2 < W) << 2) |
                         ((uint32_t)(x.w >= T && i + 3 < W) << 3);
      hitm |= (uint64_t)b << (4 * m);
    }
    uint32_t ncw;
    uint32_t p = block_excl_scan<NT>((uint32_t)__popcll(hitm), S.wsum, ncw);
    if (ncw <= (uint32_t)kWmCandWords)
      for (uint64_t h = hitm; h; h &= h - 1) S.cw[p++] = (uint32_t)(i0 + __ffsll((long long)h) - 1);
    __syncthreads();

    if (ncw <= (uint32_t)kWmCandWords) {
      // ---- 3. candidates: one warp per listed word, eight words in flight ----
      uint32_t mn = 0xFFFFFFFFu, mx = 0;
      for (int c0 = warp * 8; c0 < (int)ncw; c0 += 8 * (NT / 32)) {  // warp-uniform
        float x[8];
        int ub[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = c0 + u;
          ub[u] = c < (int)ncw ? (w0 + (int)S.cw[c]) * 32 : -64;
          x[u] = c < (int)ncw && ub[u] + lane < n ? __ldg(srow + ub[u] + lane) : -INFINITY;
        }
        uint32_t msk[8], tot = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int un = ub[u] + lane;
          msk[u] = __ballot_sync(0xFFFFFFFFu, un >= lead && un < tail && key_of_f32(x[u]) >= T);
          tot += __popc(msk[u]);
        }
        uint32_t basep = 0;
        if (lane == 0 && tot) basep = atomicAdd(&S.nct, tot);
        basep = __shfl_sync(0xFFFFFFFFu, basep, 0);
        const uint32_t below = (1u << lane) - 1u;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if ((msk[u] >> lane) & 1u) {
            const uint32_t slot = basep + __popc(msk[u] & below);
            const uint32_t key = key_of_f32(x[u]);
            if (slot < (uint32_t)kWmCand)
              S.ct[slot] = ((uint64_t)key << 32) | (uint32_t)((c0 + u) * 32 + lane);
            mn = min(mn, key);
            mx = max(mx, key);
          }
          basep += __popc(msk[u]);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
        mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      }
      if (lane == 0 && mn <= mx) { atomicMin(&S.kmin, mn); atomicMax(&S.kmax, mx); }
      __syncthreads();
      const uint32_t nct = S.nct;
      exact = nct < (uint32_t)k || nct > (uint32_t)kWmCand;
      if (!exact) {
        // ---- 4. the top k of the candidates, marked per listed word ----
        const uint32_t kmin = S.kmin;
        const uint32_t plast = ncw * 32 - 1;  // positions are < ncw * 32
        const int bC = bits_of(plast);
        const int nb = bits_of(S.kmax - kmin) + bC;
        uint32_t* selm = S.wk;  // the word keys are no longer read
        for (int c = tid; c < (int)ncw; c += NT) selm[c] = 0;
        for (uint32_t j = tid; j < nct; j += NT) {
          const uint64_t e = S.ct[j];
          S.ct[j] = ((uint64_t)((uint32_t)(e >> 32) - kmin) << bC) | (uint64_t)(plast - (uint32_t)e);
        }
        __syncthreads();
        const uint64_t Tc = nct == (uint32_t)k
                                ? 0
                                : radix_threshold<NT, uint64_t>(S.ct, (int)nct, (uint32_t)k, 0,
                                                                nb, S.hist, S.scratch, S.out);
        const uint64_t pmask = (1ull << bC) - 1;
        for (uint32_t j = tid; j < nct; j += NT) {
          const uint64_t e = S.ct[j];
          if (e >= Tc) {
            const uint32_t pp = plast - (uint32_t)(e & pmask);
            atomicOr(&selm[pp >> 5], 1u << (pp & 31));
          }
        }
        __syncthreads();
        // ---- 5. ascending placement: each thread a run of q listed words ----
        const int q = ((int)ncw + NT - 1) / NT;  // <= 4
        uint32_t cnt = 0;
        for (int e = 0; e < q; ++e) {
          const int c = tid * q + e;
          if (c < (int)ncw) cnt += __popc(selm[c]);
        }
        uint32_t total;
        uint32_t off = block_excl_scan<NT>(cnt, S.wsum, total);
        int32_t* sel_out = idx_row + lead;
        for (int e = 0; e < q; ++e) {
          const int c = tid * q + e;
          if (c < (int)ncw) {
            const int ubase = (w0 + (int)S.cw[c]) * 32;
            for (uint32_t b = selm[c]; b; b &= b - 1) sel_out[off++] = ubase + __ffs((int)b) - 1;
          }
        }
        for (int p2 = tid; p2 < lead; p2 += NT) idx_row[p2] = p2;
        const int ntail = (int)(n - tail);
        for (int p2 = tid; p2 < ntail; p2 += NT) idx_row[lead + k + p2] = tail + p2;
        if (tid == 0) count[row] = lead + k + ntail;
      }
    }
    __syncthreads();
  }
  if (!exact) return;

  // ---- the exact path: the k largest words, then their units ----
  const int kw = min(k, W);
  const int bW = bits_of((uint32_t)(W - 1));
  const int bI = bits_of((uint32_t)(M - 1));
  auto wkey = [&](int i) { return ((uint64_t)S.wk[wpos(i)] << bW) | (uint64_t)(W - 1 - i); };
  uint64_t Tw = 0;
  if (W > k)
    Tw = radix_select_fn<NT>(W, [&](int i, uint64_t& x) { x = wkey(i); return true; },
                             (uint32_t)k, 32 + bW, S.hist, S.scratch, S.out);
  if (tid == 0) S.nlist = 0;
  __syncthreads();
  for (int i = tid; i < W; i += NT)
    if (wkey(i) >= Tw) S.cw[atomicAdd(&S.nlist, 1u)] = (uint32_t)i;
  __syncthreads();
  // units of the kw words: entry e = 32 * (word's list position) + unit in word
  auto unit_of = [&](int e) { return (w0 + (int)S.cw[e >> 5]) * 32 + (e & 31); };
  auto get = [&](int e, uint64_t& x) {
    const int u = unit_of(e);
    if (u < lead || u >= tail) return false;
    x = ((uint64_t)key_of_f32(__ldg(srow + u)) << bI) |
        (uint64_t)((uint32_t)(M - 1) - (uint32_t)(u - lead));
    return true;
  };
  const uint64_t Tu = radix_select_fn<NT>(kw * 32, get, (uint32_t)k, 32 + bI, S.hist,
                                          S.scratch, S.out);
  for (int e = tid; e < kw * 32; e += NT) {
    uint64_t x;
    if (get(e, x) && x >= Tu) S.sel[atomicAdd(&S.nsel, 1u)] = (uint32_t)unit_of(e);
  }
  __syncthreads();
  const int nsel = (int)S.nsel;
  uint32_t* tmp = reinterpret_cast<uint32_t*>(S.ct);
  sort_units<NT>(S.sel, nsel, bits_of((uint32_t)(n - 1)), tmp, tmp + 2048);
  write_units<NT>(g, S.sel, nsel, idx_row, count + row);
}

// --------------------------------------------------------------------------------------
// The same selection, one thread-block cluster of CS CTAs per row (sd_topk_wmax on
// few long rows): a row's words are split evenly over the cluster's CTAs.
// --------------------------------------------------------------------------------------
//   1. each CTA loads its words' maxima (coalesced; the cut words recomputed) and
//      the same evenly spaced sample of the row's maxima, and takes T_est from the
//      sample as the single-CTA kernel does (every CTA the same T_est, no exchange);
//   2. each CTA lists its words with key >= T_est, reads their scores (one warp per
//      word, one 128-byte line), and sends every competing unit with key >= T_est
//      to CTA 0 as (key << 21 | 2^21 - 1 - unit): unique, and larger for a larger
//      key or, at equal keys, a lower unit;
//   3. with at least k candidates in all, CTA 0 radix-selects the k largest, counts
//      the selected units each CTA sent and hands every CTA the threshold and its
//      output offset; each CTA marks its selected units in a bit mask per word and
//      writes them ascending from its offset.
// Two cluster barriers in all (after the sends, after the hand-out).  NaN rows are
// reported through CTA 0.  An estimate that leaves fewer than k candidates, or
// candidates beyond the buffers (heavy ties), sends CTA 0 alone down the single-CTA
// kernel's exact path (word keys read from wmax).
constexpr int kWcThreads = 512;
constexpr int kWcWords = kWmWords / 8;  // words per CTA at CS >= 8 (9 per thread)
constexpr int kWcLocal = 3072;          // candidates a CTA holds
constexpr int kWcGather = 4096;         // candidates CTA 0 gathers

struct WcSmem {
  uint32_t wk[kWcWords];    // word keys; then the selection masks per word
  uint32_t lw[kWcWords];    // listed words; the exact path's word list
  uint64_t lc[kWcLocal];    // this CTA's candidates; the sample before them
  uint64_t gb[kWcGather];   // CTA 0: everyone's candidates; the exact path's sort scratch
  uint32_t pwh[(kWcThreads / 32) * 256];  // radix tables (per warp); the exact
                                          // path's histogram [0, 2048), units
                                          // [2048, 3072) and scratch [3072, 3104)
  uint32_t cbase[16], clen[16];  // CTA 0: where each CTA's candidates went
  uint32_t wsum[32], out[4];
  unsigned long long tc;      // CTA 0 -> all: the k-th largest candidate
  uint32_t mode;              // CTA 0 -> all: 0 thresholds, 1 the exact path, 2 NaN row
  uint32_t off;               // CTA 0 -> all: the CTA's first output slot
  uint32_t nan, nlc, ngb, ovf, kmax, nsel, nlist;
};

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// The exact path of the word-maxima selection (CTA 0 alone, rare: fewer than k
// candidates, a candidate buffer overflow): kept out of line so that the common
// path's code stays small.
__device__ __noinline__ void wc_exact(WcSmem& S, const float* __restrict__ srow,
                                      const float* __restrict__ wrow, const Geo& g,
                                      int32_t* __restrict__ idx_row, int32_t* __restrict__ count_row,
                                      int w0, int W, int64_t n) {
  constexpr int NT = kWcThreads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int lead = g.lead, tail = g.tail, k = g.k;
  const bool cut0 = (lead & 31) != 0, cut1 = (tail & 31) != 0;
  // ---- the exact path (CTA 0 alone): the k largest words, then their units ----
  // word keys from wmax, the cut words' competing maxima recomputed
  uint32_t* hist = S.pwh;
  uint32_t* sel = S.pwh + 2048;
  uint32_t* scratch = S.pwh + 3072;
  if (warp < 2) {
    const int i = warp == 0 ? 0 : W - 1;
    const int u = (w0 + i) * 32 + lane;
    float m = u >= lead && u < tail ? __ldg(srow + u) : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmax_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) S.out[2 + warp] = key_of_f32(m);
  }
  if (tid == 0) { S.nlist = 0; S.nsel = 0; }
  __syncthreads();
  const uint32_t kc0 = S.out[2], kc1 = S.out[3];
  const int M = g.M;
  const int kw = min(k, W);
  const int bW = bits_of((uint32_t)(W - 1));
  const int bI = bits_of((uint32_t)(M - 1));
  auto wkey = [&](int i) {
    const uint32_t key = (i == 0 && cut0) ? kc0
                       : (i == W - 1 && cut1) ? kc1 : key_of_f32(__ldg(wrow + i));
    return ((uint64_t)key << bW) | (uint64_t)(W - 1 - i);
  };
  uint64_t Tw = 0;
  if (W > k)
    Tw = radix_select_fn<NT>(W, [&](int i, uint64_t& x) { x = wkey(i); return true; },
                             (uint32_t)k, 32 + bW, hist, scratch, S.out);
  for (int i = tid; i < W; i += NT)
    if (wkey(i) >= Tw) S.lw[atomicAdd(&S.nlist, 1u)] = (uint32_t)i;
  __syncthreads();
  auto unit_of = [&](int e) { return (w0 + (int)S.lw[e >> 5]) * 32 + (e & 31); };
  auto get = [&](int e, uint64_t& x) {
    const int u = unit_of(e);
    if (u < lead || u >= tail) return false;
    x = ((uint64_t)key_of_f32(__ldg(srow + u)) << bI) |
        (uint64_t)((uint32_t)(M - 1) - (uint32_t)(u - lead));
    return true;
  };
  const uint64_t Tu = radix_select_fn<NT>(kw * 32, get, (uint32_t)k, 32 + bI, hist, scratch,
                                          S.out);
  for (int e = tid; e < kw * 32; e += NT) {
    uint64_t x;
    if (get(e, x) && x >= Tu) sel[atomicAdd(&S.nsel, 1u)] = (uint32_t)unit_of(e);
  }
  __syncthreads();
  const int nsel = (int)S.nsel;
  uint32_t* tmp = reinterpret_cast<uint32_t*>(S.gb);
  sort_units<NT>(sel, nsel, bits_of((uint32_t)(n - 1)), tmp, tmp + 2048);
  write_units<NT>(g, sel, nsel, idx_row, count_row);
}

// The selection of one row by its cluster (every thread of every CTA runs it; CTAs
// leave it at different points: mode 0 after writing their share, mode 2 at once,
// mode 1 all but CTA 0 at once and CTA 0 after the exact path).
template <int CS>
__device__ __forceinline__ void wc_select(WcSmem& S, const float* __restrict__ scores,
                                          const float* __restrict__ wmax, const Geo& g,
                                          int32_t* __restrict__ idx, int64_t idx_stride,
                                          int32_t* __restrict__ count) {
  constexpr int NT = kWcThreads;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.y;
  const int64_t n = g.n_units, nw = (n + 31) >> 5;  // word maxima per row (a last word may be partial)
  const float* srow = scores + row * n;
  int32_t* idx_row = idx + row * idx_stride;
  const int lead = g.lead, tail = g.tail, k = g.k;
  const int w0 = lead >> 5, W = ((tail - 1) >> 5) - w0 + 1;  // words meeting [lead, tail)
  const int wlo = (int)(((int64_t)rank * W) / CS), whi = (int)(((int64_t)(rank + 1) * W) / CS);
  const int Wc = whi - wlo;                                  // this CTA's words
  const bool cut0 = (lead & 31) != 0, cut1 = (tail & 31) != 0;
  if (tid == 0) { S.nan = 0; S.nlc = 0; S.ngb = 0; S.ovf = 0; S.kmax = 0; }
  // remote accesses start after every CTA has started and set its counters: the
  // arrival is here, the wait just before the first remote access
  cluster_arrive_release();

  // ---- 1. word keys, the sample, T_est ----
  const float* wrow = wmax + row * nw + w0;
  const int Ssz = min(W, kWmSample);
  uint32_t* samp = reinterpret_cast<uint32_t*>(S.lc);
  {
    // a cut word's competing maximum, from its scores (warps 0 and 1 of its owner)
    const bool own0 = rank == 0 && warp == 0 && cut0;
    const bool own1 = rank == CS - 1 && warp == 1 && cut1 && !(cut0 && W == 1);
    float xc = -INFINITY;
    if (own0 || own1) {
      const int u = (w0 + (own0 ? 0 : W - 1)) * 32 + lane;
      if (u >= lead && u < tail) xc = __ldg(srow + u);
    }
    constexpr int kL = kWcWords / NT;
    constexpr int kS = kWmSample / NT;
    float v[kL], sv[kS];
#pragma unroll
    for (int j = 0; j < kL; ++j) {
      const int i = j * NT + tid;
      v[j] = i < Wc ? __ldg(wrow + wlo + i) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kS; ++j) {
      const int s = j * NT + tid;
      sv[j] = s < Ssz ? __ldg(wrow + (int)(((int64_t)s * W) / Ssz)) : 0.f;
    }
    bool nan = false;
#pragma unroll
    for (int j = 0; j < kL; ++j) {
      const int i = j * NT + tid, wi = wlo + i;
      if (i < Wc) {
        if (!((wi == 0 && cut0) || (wi == W - 1 && cut1))) nan |= v[j] != v[j];
        S.wk[i] = key_of_f32(v[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < kS; ++j) {
      const int s = j * NT + tid;
      if (s < Ssz) samp[s] = key_of_f32(sv[j]);
    }
    __syncthreads();
    if (own0 || own1) {
      nan |= xc != xc;
      float m = xc;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmax_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      if (lane == 0) S.wk[own0 ? 0 : Wc - 1] = key_of_f32(m);
    }
    if (__any_sync(0xFFFFFFFFu, nan) && lane == 0) S.nan = 1;
  }
  __syncthreads();
  // two 8-bit digits: T is the low end of the 16-bit bin holding the r-th largest
  const uint32_t T = (uint32_t)radix_select_pw<NT, uint32_t>(
      samp, Ssz, (uint32_t)min(g.r_sample, Ssz), 32, 2, S.pwh, S.out);

  // ---- 2. listed words and their candidates, sent to CTA 0 ----
  {
    constexpr int kR = (kWcWords + NT - 1) / NT;  // words per thread run (<= 9)
    const int R = (Wc + NT - 1) / NT, i0 = tid * R;
    uint32_t hitm = 0;
#pragma unroll
    for (int j = 0; j < kR; ++j)
      if (j < R && i0 + j < Wc && S.wk[i0 + j] >= T) hitm |= 1u << j;
    uint32_t nl;
    uint32_t p = block_excl_scan<NT>((uint32_t)__popc(hitm), S.wsum, nl);
    for (uint32_t h = hitm; h; h &= h - 1) S.lw[p++] = (uint32_t)(wlo + i0 + __ffs((int)h) - 1);
    __syncthreads();
    uint32_t mx = 0;
    for (int c0 = warp * 8; c0 < (int)nl; c0 += 8 * (NT / 32)) {  // warp-uniform
      float x[8];
      int ub[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u;
        ub[u] = c < (int)nl ? (w0 + (int)S.lw[c]) * 32 : -64;
        x[u] = c < (int)nl && ub[u] + lane < n ? __ldg(srow + ub[u] + lane) : -INFINITY;
      }
      uint32_t msk[8], tot = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int un = ub[u] + lane;
        msk[u] = __ballot_sync(0xFFFFFFFFu, un >= lead && un < tail && key_of_f32(x[u]) >= T);
        tot += __popc(msk[u]);
      }
      uint32_t basep = 0;
      if (lane == 0 && tot) basep = atomicAdd(&S.nlc, tot);
      basep = __shfl_sync(0xFFFFFFFFu, basep, 0);
      const uint32_t below = (1u << lane) - 1u;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if ((msk[u] >> lane) & 1u) {
          const uint32_t slot = basep + __popc(msk[u] & below);
          const uint32_t key = key_of_f32(x[u]);
          if (slot < (uint32_t)kWcLocal)
            S.lc[slot] = ((uint64_t)key << 21) | (uint64_t)(0x1FFFFFu - (uint32_t)(ub[u] + lane));
          mx = max(mx, key);
        }
        basep += __popc(msk[u]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    if (lane == 0 && mx) atomicMax(&S.kmax, mx);
    __syncthreads();
    cluster_wait_acquire();  // every CTA has started
    const uint32_t nlc = S.nlc;
    WcSmem* S0 = cl.map_shared_rank(&S, 0);
    if (tid == 0) {
      uint32_t gbase = 0xFFFFFFFFu;
      if (S.nan) atomicOr(&S0->nan, 1u);
      if (nlc > (uint32_t)kWcLocal) {
        atomicOr(&S0->ovf, 1u);
      } else {
        gbase = nlc ? atomicAdd(&S0->ngb, nlc) : 0u;
        if (gbase + nlc > (uint32_t)kWcGather) gbase = 0xFFFFFFFFu;  // CTA 0 sees ngb > cap
        atomicMax(&S0->kmax, S.kmax);
      }
      S0->cbase[rank] = gbase;
      S0->clen[rank] = nlc;
      S.out[2] = gbase;
    }
    __syncthreads();
    const uint32_t gbase = S.out[2];
    if (gbase != 0xFFFFFFFFu)
      for (uint32_t i = tid; i < nlc; i += NT) S0->gb[gbase + i] = S.lc[i];
  }
  __syncthreads();
  cl.sync();  // B1: CTA 0 holds the candidates (or knows that they overflowed)

  // ---- 3. CTA 0: the k-th largest candidate, counts and offsets, handed out ----
  if (rank == 0) {
    const uint32_t ngb = S.ngb;
    uint32_t mode = S.nan ? 2u : (S.ovf || ngb > (uint32_t)kWcGather || ngb < (uint32_t)k) ? 1u : 0u;
    uint64_t tc = 0;
    if (mode == 0) {
      // keys are >= T: subtract T's place so that the select starts at the bits that differ
      const uint64_t base = (uint64_t)T << 21;
      for (uint32_t i = tid; i < ngb; i += NT) S.gb[i] -= base;
      __syncthreads();
      const int nb = bits_of(S.kmax - T) + 21;
      if (ngb > (uint32_t)k)
        tc = radix_threshold<NT, uint64_t>(S.gb, (int)ngb, (uint32_t)k, 0, nb, S.pwh,
                                           S.pwh + kBins, S.out);  // 11-bit digits
      // selected units per sending CTA (warp r counts CTA r's candidates)
      if (warp < CS) {
        const uint32_t b0 = S.cbase[warp], len = S.clen[warp];
        uint32_t c = 0;
        for (uint32_t i = lane; i < len; i += 32) c += S.gb[b0 + i] >= tc ? 1u : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
        if (lane == 0) S.pwh[warp] = c;  // the select is done with the tables
      }
      __syncthreads();
      tc += base;
    }
    if (tid < CS) {
      uint32_t off = 0;
      for (int r = 0; r < tid; ++r) off += mode == 0 ? S.pwh[r] : 0u;
      WcSmem* Sr = cl.map_shared_rank(&S, tid);
      Sr->tc = tc;
      Sr->mode = mode;
      Sr->off = off;
    }
  }
  __syncthreads();
  cl.sync();  // B2: no shared memory is accessed remotely after this

  if (S.mode == 2) {  // a NaN among the competing scores
    if (rank == 0 && tid == 0) count[row] = -1;
    return;
  }
  if (S.mode == 0) {
    // ---- 4. mark and write ----
    const uint64_t tc = S.tc;
    const uint32_t nlc = S.nlc;
    uint32_t* selm = S.wk;  // one mask per word of this CTA
    for (int i = tid; i < Wc; i += NT) selm[i] = 0;
    __syncthreads();
    for (uint32_t i = tid; i < nlc; i += NT) {
      const uint64_t e = S.lc[i];
      if (e >= tc) {
        const uint32_t u = 0x1FFFFFu - (uint32_t)(e & 0x1FFFFFu);
        atomicOr(&selm[(int)(u >> 5) - w0 - wlo], 1u << (u & 31));
      }
    }
    __syncthreads();
    constexpr int kR = (kWcWords + NT - 1) / NT;
    const int R = (Wc + NT - 1) / NT, i0 = tid * R;
    uint32_t cnt = 0;
#pragma unroll
    for (int j = 0; j < kR; ++j)
      if (j < R && i0 + j < Wc) cnt += __popc(selm[i0 + j]);
    uint32_t mine;
    uint32_t off = S.off + block_excl_scan<NT>(cnt, S.wsum, mine);
    int32_t* sel_out = idx_row + lead;
#pragma unroll
    for (int j = 0; j < kR; ++j) {
      if (j < R && i0 + j < Wc) {
        const int ubase = (w0 + wlo + i0 + j) * 32;
        for (uint32_t b = selm[i0 + j]; b; b &= b - 1) sel_out[off++] = ubase + __ffs((int)b) - 1;
      }
    }
    const int ntail = (int)(n - tail);
    if (rank == 0) {
      for (int p2 = tid; p2 < lead; p2 += NT) idx_row[p2] = p2;
      if (tid == 0) count[row] = lead + k + ntail;
    }
    if (rank == CS - 1)
      for (int p2 = tid; p2 < ntail; p2 += NT) idx_row[lead + k + p2] = tail + p2;
    return;
  }
  if (rank != 0) return;

  wc_exact(S, srow, wrow, g, idx_row, count + row, w0, W, n);
}


template <int CS>
__global__ void __launch_bounds__(kWcThreads, 2)
topk_wmax_cluster_kernel(const float* __restrict__ scores, const float* __restrict__ wmax, Geo g,
                         int32_t* __restrict__ idx, int64_t idx_stride,
                         int32_t* __restrict__ count) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  wc_select<CS>(*reinterpret_cast<WcSmem*>(smem_raw), scores, wmax, g, idx, idx_stride, count);
}

// sd_select_attend: the selection above, then gather-attend over the selected rows
// in the same 16-CTA cluster (at_cluster_row, as attend_cluster_kernel runs it, on
// threads 0..127 of each CTA), with one cluster barrier between them instead of a
// kernel boundary.  The attention's staging reuses the selection's buffers.
template <int G>
__global__ void __launch_bounds__(kWcThreads, 2)
select_attend_kernel(const float* __restrict__ scores, const float* __restrict__ wmax, Geo g,
                     int32_t* __restrict__ idx, int64_t idx_stride, int32_t* __restrict__ count,
                     const uint16_t* __restrict__ q, const uint16_t* __restrict__ K,
                     const uint16_t* __restrict__ V, int Hq, int Hkv, int64_t n_tok,
                     int64_t ncap, int max_count, float scale, float* __restrict__ out,
                     float* __restrict__ lse) {
  static_assert(sizeof(AtChunk<G>) <= sizeof(WcSmem::gb) && sizeof(AtState<G>) <= sizeof(WcSmem::lc),
                "attention buffers must fit in the selection's");
  extern __shared__ __align__(16) uint8_t smem_raw[];
  WcSmem& S = *reinterpret_cast<WcSmem*>(smem_raw);
  wc_select<kAtCS>(S, scores, wmax, g, idx, idx_stride, count);
  cg::cluster_group cl = cg::this_cluster();
  cl.sync();  // every CTA's idx and count writes are visible cluster-wide
  if (threadIdx.x < 128) {
    at_cluster_row<G>(*reinterpret_cast<AtChunk<G>*>(&S.gb[0]),
                      *reinterpret_cast<AtState<G>*>(&S.lc[0]), blockIdx.y, q, K, V, idx,
                      idx_stride, count, Hq, Hkv, n_tok, ncap, max_count, scale, out, lse,
                      [] { asm volatile("bar.sync 5, 128;\n" ::: "memory"); });
  } else {  // the body's two cluster barriers
    cl.sync();
    cl.sync();
  }
}

// Resident clusters of CS CTAs of topk_wmax_cluster_kernel (0: cannot run), per device.
template <int CS>
static int wmax_cluster_capacity() {
  if (fallback_forced()) return 0;
  static std::atomic<int> cap[kMaxDev];
  return per_device_cached(cap, [] {
    auto kern = topk_wmax_cluster_kernel<CS>;
    int nc = 0;
    bool yes = set_smem_limit((const void*)kern, sizeof(WcSmem), "topk_wmax cluster") == SD_OK;
    if (yes && CS > 8)
      yes = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess;
    if (yes) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(CS, 1, 1);
      cfg.blockDim = dim3(kWcThreads, 1, 1);
      cfg.dynamicSmemBytes = sizeof(WcSmem);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = CS;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess) nc = 0;
    }
    cudaGetLastError();
    return nc;
  });
}

template <int CS>
static int launch_wmax_cluster(const float* scores, const float* wmax, int64_t rows,
                               const Geo& g, int32_t* idx, int64_t idx_stride, int32_t* count,
                               cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS, (unsigned)rows, 1);
  cfg.blockDim = dim3(kWcThreads, 1, 1);
  cfg.dynamicSmemBytes = sizeof(WcSmem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, topk_wmax_cluster_kernel<CS>, scores, wmax, g, idx, idx_stride,
                         count) != cudaSuccess)
    return check_launch("topk_wmax cluster");
  note_launches(1);
  return check_launch("topk_wmax cluster");
}

int launch_topk_wmax(const float* scores, const float* wmax, int64_t rows, int64_t n,
                     const sd_select& sel, int32_t* idx, int64_t idx_stride, int32_t* count,
                     void* ws, size_t ws_bytes, cudaStream_t st) {
  Geo g = make_geo(n, n, sel);
  const int64_t W = g.M > 0 ? ((g.tail - 1) >> 5) - (g.lead >> 5) + 1 : 0;
  if (!(n > kSmallRow && g.M > g.k && g.k <= kWmMaxK && W <= kWmWords &&
        (uintptr_t)scores % 16 == 0))
    return launch_topk(SD_SCORE_F32, scores, rows, n, n, sel, idx, idx_stride, count, ws,
                       ws_bytes, st);
  g.r_sample = sample_rank(g.k, imin64(W, kWmSample), W);
  // few rows: a cluster per row spreads the row's reads over CS SMs
  if (n <= (1 << 21) && W > g.k && W >= 64 * 16 && rows <= 65535) {
    if (rows <= wmax_cluster_capacity<16>())
      return launch_wmax_cluster<16>(scores, wmax, rows, g, idx, idx_stride, count, st);
    if (rows <= wmax_cluster_capacity<8>())
      return launch_wmax_cluster<8>(scores, wmax, rows, g, idx, idx_stride, count, st);
  }
  if (int rc = set_smem_limit((const void*)topk_wmax_kernel, sizeof(WmSmem), "topk_wmax"))
    return rc;
  topk_wmax_kernel<<<(unsigned)rows, kWmThreads, sizeof(WmSmem), st>>>(scores, wmax, g, idx,
                                                                        idx_stride, count);
  note_launches(1);
  return check_launch("topk_wmax");
}

// =====================================================================================
// Fused bit-plane scan + top-k (sd_score_topk).
//
// Filtering 32 MB of scores after the scan costs a full read per step.  Instead,
// a short kernel first scores a sample of every row -- kSmpRuns runs of 32
// consecutive tokens (one word of each planned plane), spread evenly over the
// competing tokens, with the scan's folded weights -- and takes a threshold key
// below the row's k-th score with high probability (the r-th largest sample key,
// r from the same margin as the other estimates, widened because the 32 tokens of
// a run are not independent: mu = k S / M, r = mu + 5 sqrt(8 mu) + 2).  The scan
// then appends every competing token whose key reaches the threshold to the row's
// candidate list (and still writes all scores), and the cluster top-k draws the
// exact top k from that list.  A row whose list holds fewer than k entries,
// overflows, or holds a NaN is selected again from its full score row, so the
// result is always that of sd_score followed by sd_topk.
// =====================================================================================
constexpr int kSmpRuns = 256;                   // sampled runs of 32 tokens per row
constexpr int kSmpSplit = 16;                   // CTAs per row
constexpr int kSmpRunsCta = kSmpRuns / kSmpSplit;  // 16
constexpr int kSmpPer = 8;                      // threads per run (adjacent lanes)
constexpr int kSmpThreads = kSmpRunsCta * kSmpPer;  // 128
constexpr int kSmpTok = kSmpRuns * 32;          // sampled tokens per row
constexpr int kFusedCap = kCap;                 // candidates the selecting CTA holds
constexpr int64_t kFusedMinM = 65536;           // shorter rows: scan, then sd_topk

struct SmpSmem {
  PsRow row;
  uint32_t wsum[kSmpThreads / 32];
  uint32_t last;
};

// The largest key T with at least r of the calling CTA's keys (K per thread, in
// registers) >= T: a bitwise search, one CTA-wide count per bit.  (r is small and
// the keys of a row's scores crowd a few high-order digits, so this beats a radix
// histogram with its serialised shared-memory atomics.)
template <int NT, int K>
__device__ uint32_t kth_largest_bits(const uint32_t (&key)[K], uint32_t r, uint32_t* wsum) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t T = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t cand = T | (1u << bit);
    uint32_t c = 0;
#pragma unroll
    for (int i = 0; i < K; ++i) c += key[i] >= cand;
    c = __reduce_add_sync(0xFFFFFFFFu, c);
    if (lane == 0) wsum[warp] = c;
    __syncthreads();
    uint32_t tot = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) tot += wsum[w];
    __syncthreads();
    if (tot >= r) T = cand;
  }
  return T;
}

// Sample keys of a row's runs [32 b, 32 b + 32), b = blockIdx.x: keys[row][...] in
// the workspace; the row's last CTA to finish (ticket) selects the threshold.
template <int G>
__global__ void __launch_bounds__(kSmpThreads)
plane_sample_kernel(const uint32_t* __restrict__ planes, const uint16_t* __restrict__ scales,
                    const uint8_t* __restrict__ plan, const uint16_t* __restrict__ q, int Hq,
                    int Hkv, int64_t ncap, int64_t lead, int64_t tail, int r,
                    uint32_t* __restrict__ skeys, uint32_t* __restrict__ ticket,
                    uint32_t* __restrict__ thr, uint32_t* __restrict__ cnan) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SmpSmem& S = *reinterpret_cast<SmpSmem*>(smem_raw);
  const int t = threadIdx.x;
  const int row = blockIdx.y;
  ps_build_row<G>(S.row, t, q, plan, row / Hkv, row % Hkv, Hq, (int64_t)row,
                  [] { __syncthreads(); });
  const int run = blockIdx.x * kSmpRunsCta + t / kSmpPer, eg = t % kSmpPer;
  // the run's word, evenly spaced over the words that hold competing tokens
  const int64_t w0 = lead / 32, w1 = (tail + 31) / 32;
  const int64_t w = w0 + ((2 * (int64_t)run + 1) * (w1 - w0)) / (2 * kSmpRuns);
  const uint32_t wstride = (uint32_t)(ncap / 32), sstride = (uint32_t)(ncap / 64);
  const uint32_t* prow = planes + (int64_t)row * kD * 4 * wstride + w;
  const uint16_t* srow = scales + (int64_t)row * kD * sstride + (w >> 1);
  const int nact = S.row.nact, nch = S.row.nch;
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
  float cp = 0.0f;
  // this thread's planes e = eg + 8u and slots sl = eg + 8u: loads issued 8 planes
  // and 8 slots at a time, then the bits and the block constant's terms
  const int nb = max(nact, nch);
  for (int e0 = eg; e0 < nb; e0 += 8 * kSmpPer) {
    uint32_t wv[8];
    float sv[8], cv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + u * kSmpPer;
      if (e < nact) {
        const int ent = S.row.act[e];
        wv[u] = __ldg(prow + (int64_t)ent * wstride);
        sv[u] = __half2float(__ushort_as_half(__ldg(srow + (int64_t)(ent >> 2) * sstride)));
      }
      if (e < nch)
        cv[u] = __half2float(__ushort_as_half(__ldg(srow + (int64_t)S.row.chan[e] * sstride)));
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + u * kSmpPer;
      if (e < nact) ps_bits(acc, wv[u], __fmul_rn(S.row.qp[e], sv[u]));
      if (e < nch) cp = __fadd_rn(cp, __fmul_rn(S.row.qo[e], cv[u]));
    }
  }
  // the run's eight partial sums meet by shuffles: each round halves what a lane
  // keeps; lane eg ends with the totals of 4 tokens
  float h16[16], h8[8], h4[4];
  {
    const bool b = eg & 1;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float keep = b ? acc[16 + i] : acc[i], give = b ? acc[i] : acc[16 + i];
      h16[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, give, 1);
    }
  }
  {
    const bool b = eg & 2;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float keep = b ? h16[8 + i] : h16[i], give = b ? h16[i] : h16[8 + i];
      h8[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, give, 2);
    }
  }
  {
    const bool b = eg & 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float keep = b ? h8[4 + i] : h8[i], give = b ? h8[i] : h8[4 + i];
      h4[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, give, 4);
    }
  }
  cp += __shfl_xor_sync(0xFFFFFFFFu, cp, 1);
  cp += __shfl_xor_sync(0xFFFFFFFFu, cp, 2);
  cp += __shfl_xor_sync(0xFFFFFFFFu, cp, 4);
  const int tk0 = ((eg & 1) ? 16 : 0) + ((eg & 2) ? 8 : 0) + ((eg & 4) ? 4 : 0);
  uint32_t* krow = skeys + (int64_t)row * kSmpTok;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float v = h4[i] + cp;
    const int64_t tok = w * 32 + tk0 + i;
    const bool in = tok >= lead && tok < tail && v == v;  // competing, not NaN
    krow[run * 32 + tk0 + i] = in ? key_of_f32(v) : 0u;
  }
  // the row's last CTA selects
  __threadfence();
  __syncthreads();
  if (t == 0) S.last = atomicAdd(ticket + row, 1u) == kSmpSplit - 1;
  __syncthreads();
  if (!S.last) return;
  __threadfence();
  constexpr int KPT = kSmpTok / kSmpThreads;  // keys per thread
  uint32_t key[KPT];
#pragma unroll
  for (int i = 0; i < KPT; ++i) key[i] = __ldcg(krow + i * kSmpThreads + t);
  const uint32_t T = kth_largest_bits<kSmpThreads, KPT>(key, (uint32_t)r, S.wsum);
  if (t == 0) {
    thr[row] = (uint32_t)T;
    cnan[row] = 0u;
    ticket[row] = 0u;  // ready for the next call
  }
}

static int fused_rank(int64_t k, int64_t S, int64_t M) {
  const double mu = (double)k * (double)S / (double)M;
  const double r = std::ceil(mu + 5.0 * std::sqrt(8.0 * mu) + 2.0);
  return (int)(r < (double)S ? r : (double)S);
}

size_t score_topk_workspace_bytes(int64_t rows, int64_t n, const sd_select& sel) {
  return align256(topk_workspace_bytes(rows, n, sel)) + align256(sizeof(uint32_t) * 3 * rows) +
         align256(sizeof(uint32_t) * rows * kSmpTok) + align256(sizeof(uint32_t) * rows * (n / 32));
}

template <int G>
static int sample_t(const Dims& s, const uint32_t* planes, const uint16_t* scales,
                    const uint8_t* plan, const uint16_t* q, const Geo& g, int r, uint32_t* skeys,
                    uint32_t* ticket, uint32_t* thr, uint32_t* cnan, cudaStream_t st) {
  auto kern = plane_sample_kernel<G>;
  if (int rc = set_smem_limit((const void*)kern, sizeof(SmpSmem), "plane sample: smem attribute"))
    return rc;
  const int64_t rows = (int64_t)s.B * s.Hkv;
  if (cudaMemsetAsync(ticket, 0, sizeof(uint32_t) * rows, st) != cudaSuccess)
    return check_launch("plane sample: ticket clear");
  kern<<<dim3(kSmpSplit, (unsigned)rows), kSmpThreads, sizeof(SmpSmem), st>>>(
      planes, scales, plan, q, s.Hq, s.Hkv, s.ncap, (int64_t)g.lead, (int64_t)g.tail, r, skeys,
      ticket, thr, cnan);
  note_launches(1);
  return check_launch("plane sample");
}

int launch_score_topk(const Dims& s, const uint32_t* planes, const uint16_t* scales,
                      const uint8_t* plan, const uint16_t* q, const sd_select& sel, float* scores,
                      int32_t* idx, int64_t idx_stride, int32_t* count, void* ws,
                      cudaStream_t st) {
  const int64_t rows = (int64_t)s.B * s.Hkv;
  Geo g = make_geo(s.n, s.n, sel);
  if (g.M > 0) {
    g.r_sample = sample_rank(g.k, sample_size(g), g.M);
    g.r_cluster = sample_rank(g.k, cluster_sample_size(g), g.M);
  }
  // fused where the threshold keeps the expected candidates within 3/5 of what the
  // selecting CTA holds (the count's spread is about sqrt of it)
  int r = 0;
  bool fused = false;
  if (sel.block == 1 && g.M >= kFusedMinM && g.M > g.k && planes_aligned(s, planes, scales)) {
    r = fused_rank(g.k, kSmpTok, g.M);
    fused = (int64_t)r * (g.M / kSmpTok) <= kFusedCap * 3 / 5;
  }
  if (!fused) {  // scan, then the standalone top-k
    if (int rc = launch_score_planes(s, planes, scales, plan, q, scores, st)) return rc;
    return topk_t<true>(scores, rows, g, idx, idx_stride, count, ws, st);
  }
  uint8_t* p = static_cast<uint8_t*>(ws) + align256(topk_workspace_bytes(rows, s.n, sel));
  uint32_t* thr = reinterpret_cast<uint32_t*>(p);
  uint32_t* cnan = thr + rows;
  uint32_t* ticket = cnan + rows;
  p += align256(sizeof(uint32_t) * 3 * rows);
  uint32_t* skeys = reinterpret_cast<uint32_t*>(p);
  uint32_t* hits = reinterpret_cast<uint32_t*>(p + align256(sizeof(uint32_t) * rows * kSmpTok));
  int rc;
  switch (s.G) {
    case 1: rc = sample_t<1>(s, planes, scales, plan, q, g, r, skeys, ticket, thr, cnan, st); break;
    case 2: rc = sample_t<2>(s, planes, scales, plan, q, g, r, skeys, ticket, thr, cnan, st); break;
    case 4: rc = sample_t<4>(s, planes, scales, plan, q, g, r, skeys, ticket, thr, cnan, st); break;
    default: rc = sample_t<8>(s, planes, scales, plan, q, g, r, skeys, ticket, thr, cnan, st); break;
  }
  if (rc) return rc;
  const PsCand cd{thr, hits, cnan, s.n / 32, (int64_t)g.lead, (int64_t)g.tail};
  if ((rc = launch_score_planes(s, planes, scales, plan, q, scores, st, &cd))) return rc;
  auto sel_k = topk_marked_kernel<true>;
  if ((rc = set_smem_limit((const void*)sel_k, sizeof(FinSmem), "topk marked: smem attribute")))
    return rc;
  sel_k<<<(unsigned)rows, kMarkThreads, sizeof(FinSmem), st>>>(scores, g, hits, cnan, s.n / 32,
                                                                idx, idx_stride, count);
  note_launches(1);
  return check_launch("topk marked");
}

}  // namespace sd

namespace sd {

// Resident 16-CTA clusters of select_attend_kernel<G> (0: cannot run), per device.
template <int G>
static int select_attend_capacity() {
  if (fallback_forced()) return 0;
  static std::atomic<int> cap[kMaxDev];
  return per_device_cached(cap, [] {
    auto kern = select_attend_kernel<G>;
    int nc = 0;
    bool yes = set_smem_limit((const void*)kern, sizeof(WcSmem), "select_attend") == SD_OK &&
               cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                   cudaSuccess;
    if (yes) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(kAtCS, 1, 1);
      cfg.blockDim = dim3(kWcThreads, 1, 1);
      cfg.dynamicSmemBytes = sizeof(WcSmem);
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
    return nc;
  });
}

template <int G>
static int launch_select_attend_g(const Dims& s, const float* scores, const float* wmax, Geo g,
                                  const uint16_t* q, const uint16_t* K, const uint16_t* V,
                                  float scale, int32_t* idx, int64_t idx_stride, int32_t* count,
                                  int64_t max_count, float* out, float* lse, int64_t rows,
                                  bool* launched, cudaStream_t st) {
  *launched = false;
  if (rows > select_attend_capacity<G>()) return SD_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kAtCS, (unsigned)rows, 1);
  cfg.blockDim = dim3(kWcThreads, 1, 1);
  cfg.dynamicSmemBytes = sizeof(WcSmem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kAtCS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  *launched = true;
  if (cudaLaunchKernelEx(&cfg, select_attend_kernel<G>, scores, wmax, g, idx, idx_stride, count,
                         q, K, V, s.Hq, s.Hkv, s.n, s.ncap, (int)max_count, scale, out,
                         lse) != cudaSuccess)
    return check_launch("select_attend");
  note_launches(1);
  return check_launch("select_attend");
}

size_t select_attend_workspace_bytes(const Dims& s, const sd_select& sel, int64_t max_count) {
  const size_t t = topk_workspace_bytes((int64_t)s.B * s.Hkv, s.n, sel);
  return ((t + 255) & ~(size_t)255) + attend_workspace_bytes(s, max_count);
}

int launch_select_attend(const Dims& s, const float* scores, const float* wmax,
                         const sd_select& sel, const uint16_t* q, const uint16_t* K,
                         const uint16_t* V, float scale, int32_t* idx, int64_t idx_stride,
                         int32_t* count, int64_t max_count, float* out, float* lse, void* ws,
                         size_t ws_bytes, cudaStream_t st) {
  const int64_t rows = (int64_t)s.B * s.Hkv, n = s.n;
  Geo g = make_geo(n, n, sel);
  const int64_t W = g.M > 0 ? ((g.tail - 1) >> 5) - (g.lead >> 5) + 1 : 0;
  if (n > kSmallRow && g.M > g.k && g.k <= kWmMaxK && W <= kWmWords && W > g.k &&
      W >= 64 * 16 && n <= (1 << 21) && rows <= 65535 && max_count <= (1 << 30) &&
      (uintptr_t)scores % 16 == 0) {
    g.r_sample = sample_rank(g.k, imin64(W, kWmSample), W);
    bool launched = false;
    int rc = SD_OK;
    switch (s.G) {
      case 1: rc = launch_select_attend_g<1>(s, scores, wmax, g, q, K, V, scale, idx, idx_stride, count, max_count, out, lse, rows, &launched, st); break;
      case 2: rc = launch_select_attend_g<2>(s, scores, wmax, g, q, K, V, scale, idx, idx_stride, count, max_count, out, lse, rows, &launched, st); break;
      case 4: rc = launch_select_attend_g<4>(s, scores, wmax, g, q, K, V, scale, idx, idx_stride, count, max_count, out, lse, rows, &launched, st); break;
      default: rc = launch_select_attend_g<8>(s, scores, wmax, g, q, K, V, scale, idx, idx_stride, count, max_count, out, lse, rows, &launched, st); break;
    }
    if (launched || rc != SD_OK) return rc;
  }
  // the two calls
  const size_t t = topk_workspace_bytes(rows, n, sel), ta = (t + 255) & ~(size_t)255;
  if (int rc = launch_topk_wmax(scores, wmax, rows, n, sel, idx, idx_stride, count, ws, t, st))
    return rc;
  return launch_gather_attend(s, q, K, V, idx, idx_stride, count, max_count, scale, out, lse,
                              ws ? (uint8_t*)ws + ta : nullptr, ws_bytes > ta ? ws_bytes - ta : 0,
                              st);
}

}  // namespace sd
