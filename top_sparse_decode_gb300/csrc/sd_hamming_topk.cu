// Hamming scan and exact top-k in two passes over the signatures (HashAttention:
// Semantic Sparsity for Faster Inference, 2.1 SCORE -> TOPK, 2.2 SCORE =
// -Hamming, summed here over the GQA group; 3.1 the first and last tokens kept,
// the budget counted apart).  The same idx and count as sd_score(SD_IDX_SIG)
// followed by sd_topk(SD_SCORE_I32): the k competing tokens of largest score,
// lowest index first among equal scores, ascending.
//
// A token's score v = -sum_g popcount(h_i ^ h_q,g) takes one of 32 G + 1 values, so
// u = -v in [0, 32 G] indexes a small histogram and the k-th largest score is found
// exactly from counts:
//   pass 1 (hist): CTA p of a row scores its range of 8192 competing tokens (128-bit
//     loads) and writes its histogram of u, also added into the row's; the row's
//     last CTA to finish (a ticket) finds u* (the k-th best value: fewer than k
//     tokens have u < u*, at least k have u <= u*) and need = k - #{u < u*}, and
//     from the ranges' histograms every range's count of ties (u = u*) and of
//     selected tokens before it (ties taken in token order);
//   pass 2 (pick): CTA p scores its range again from the signatures (4 B per token:
//     cheaper than writing and re-reading 4 B scores), takes every token with
//     u < u* and its first max(0, min(ties in range, need - ties before)) tokens
//     with u = u*, and writes them ascending from its offset (a block-wide scan in
//     token order: no sort).
#include "sd_internal.cuh"

namespace sd {

constexpr int kHtThreads = 256;
constexpr int kHtPer = 8;                          // 128-bit loads per thread
constexpr int kHtRange = kHtThreads * 4 * kHtPer;  // tokens per CTA (8192)
constexpr int kHtBins = 32 * 8 + 1;                // u in [0, 32 G], G <= 8
constexpr uint32_t kHtOut = 1023;                  // u of a token outside [lead, tail)

struct HtGeo {
  int64_t n, ncap;
  int lead, tail, k, P;  // competing tokens [lead, tail); P ranges per row
  int Hq, Hkv;
};

// Scores of the range's tokens for lane-strided 128-bit groups: token t0 + 4 (256 j
// + tid) + e for j < kHtPer, e < 4.  Tokens outside [lead, tail) get u = kHtOut.
template <int G>
__device__ __forceinline__ void ht_scores(const uint32_t* __restrict__ srow, const uint32_t (&qs)[G],
                                          int64_t t0, const HtGeo& g, bool vec,
                                          uint32_t (&u)[kHtPer][4]) {
  const int tid = threadIdx.x;
  if (vec) {
    uint4 s4[kHtPer];
#pragma unroll
    for (int j = 0; j < kHtPer; ++j) {
      const int64_t i = t0 + 4 * (j * kHtThreads + tid);
      s4[j] = i + 4 <= g.tail ? __ldg(reinterpret_cast<const uint4*>(srow + i))
                              : make_uint4(0u, 0u, 0u, 0u);
      if (i + 4 > g.tail) {  // the range's last, partial group: scalar loads in bounds
        uint32_t v[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (i + e < g.tail) v[e] = __ldg(srow + i + e);
        s4[j] = make_uint4(v[0], v[1], v[2], v[3]);
      }
    }
#pragma unroll
    for (int j = 0; j < kHtPer; ++j) {
      const uint32_t sv[4] = {s4[j].x, s4[j].y, s4[j].z, s4[j].w};
      const int64_t i = t0 + 4 * (j * kHtThreads + tid);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t acc = 0;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) acc += __popc(sv[e] ^ qs[gg]);
        u[j][e] = (i + e >= g.lead && i + e < g.tail) ? acc : kHtOut;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < kHtPer; ++j) {
      const int64_t i = t0 + 4 * (j * kHtThreads + tid);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t acc = kHtOut;
        if (i + e >= g.lead && i + e < g.tail) {
          const uint32_t sv = __ldg(srow + i + e);
          acc = 0;
#pragma unroll
          for (int gg = 0; gg < G; ++gg) acc += __popc(sv ^ qs[gg]);
        }
        u[j][e] = acc;
      }
    }
  }
}

// The range of CTA p: tokens [t0, t0 + kHtRange) of the competing span, aligned down
// to a 4-token group so that 128-bit loads stay aligned.
__device__ __forceinline__ int64_t ht_range0(const HtGeo& g, int p) {
  return ((int64_t)g.lead & ~(int64_t)3) + (int64_t)p * kHtRange;
}

// Per-row results of pass 1, in the workspace.
struct HtWs {
  uint32_t* hist;    // [rows][P][kHtBins]: each range's histogram of u
  uint32_t* total;   // [rows][kHtBins]: the row's histogram (zeroed by the call)
  uint32_t* ticket;  // [rows]: ranges done (zeroed by the call)
  int32_t* pick;     // [rows][2]: u*, need
  int32_t* before;   // [rows][P][2]: ties before the range, selected tokens before it
};

template <int G>
__global__ void __launch_bounds__(kHtThreads)
hamming_hist_kernel(const uint32_t* __restrict__ sig, const uint32_t* __restrict__ qsig, HtGeo g,
                    bool vec, HtWs w) {
  __shared__ uint32_t h[kHtBins + 1];
  __shared__ uint32_t wsum[kHtThreads / 32];
  __shared__ int last, ustar, need;
  const int p = blockIdx.x, tid = threadIdx.x;
  const int64_t row = blockIdx.y;
  const int b = (int)(row / g.Hkv), hh = (int)(row % g.Hkv);
  constexpr int nb = 32 * G + 1;
  uint32_t qs[G];
#pragma unroll
  for (int gg = 0; gg < G; ++gg) qs[gg] = __ldg(qsig + (int64_t)b * g.Hq + hh * G + gg);
  for (int i = tid; i <= kHtBins; i += kHtThreads) h[i] = 0;
  __syncthreads();
  uint32_t u[kHtPer][4];
  ht_scores<G>(sig + row * g.ncap, qs, ht_range0(g, p), g, vec, u);
#pragma unroll
  for (int j = 0; j < kHtPer; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      atomicAdd(&h[min(u[j][e], (uint32_t)kHtBins)], 1u);  // outside tokens: the spare bin
    }
  __syncthreads();
  uint32_t* hrow = w.hist + (row * g.P + p) * kHtBins;
  for (int i = tid; i < nb; i += kHtThreads) {
    hrow[i] = h[i];
    if (h[i]) atomicAdd(w.total + row * kHtBins + i, h[i]);
  }
  __threadfence();  // this range's counts are visible before its ticket
  __syncthreads();
  if (tid == 0) last = atomicAdd(w.ticket + row, 1u) == (uint32_t)(g.P - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  // the last range of the row: u* and the ties to take, then every range's offsets
  const uint32_t* tot = w.total + row * kHtBins;
  if (tid < 32) {  // one warp scans the row histogram from the best value (u = 0) up
    const int M = g.tail - g.lead;
    int us = nb, nd = 0;  // all competing tokens fit: none is cut
    if (M > g.k) {
      uint32_t run = 0;
      for (int u0 = 0; u0 < nb; u0 += 32) {
        const uint32_t c = u0 + tid < nb ? __ldcg(tot + u0 + tid) : 0u;
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (tid >= o) incl += y;
        }
        const uint32_t reach = __ballot_sync(0xFFFFFFFFu, run + incl >= (uint32_t)g.k);
        if (reach) {
          const int l = __ffs((int)reach) - 1;
          us = u0 + l;
          nd = g.k - (int)(run + __shfl_sync(0xFFFFFFFFu, incl - c, l));
          break;
        }
        run += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
    }
    if (tid == 0) { ustar = us; need = nd; }
  }
  __syncthreads();
  const int us = ustar, nd = need;
  // per range: ties (u = u*) and sure tokens (u < u*); ranges ascending.  The P x u*
  // counts below u* are summed by all threads at once (independent loads, shared
  // atomics per range); h serves as the per-range sums.
  const int nbu = min(us, nb);
  for (int i = tid; i < g.P; i += kHtThreads) h[i] = 0;
  __syncthreads();
  const uint32_t* hrow0 = w.hist + row * g.P * kHtBins;
  for (int e = tid; e < g.P * nbu; e += kHtThreads) {
    const int pp = e / nbu, i = e - pp * nbu;
    const uint32_t v = __ldcg(hrow0 + pp * kHtBins + i);
    if (v) atomicAdd(&h[pp], v);
  }
  __syncthreads();
  uint32_t ties = 0, sure = 0;
  if (tid < g.P) {
    sure = h[tid];
    ties = us < nb ? __ldcg(hrow0 + tid * kHtBins + us) : 0u;
  }
  // exclusive prefixes over the ranges (P <= kHtThreads), taking ties in order
  auto scan = [&](uint32_t v) {
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    uint32_t before = incl - v;
    for (int x = 0; x < warp; ++x) before += wsum[x];
    __syncthreads();
    return before;
  };
  const uint32_t ties_before = scan(ties);
  const uint32_t taken = (uint32_t)min(max(nd - (int)ties_before, 0), (int)ties);
  const uint32_t sel_before = scan(sure + taken);
  if (tid < g.P) {
    int32_t* bp = w.before + (row * g.P + tid) * 2;
    bp[0] = (int32_t)ties_before;
    bp[1] = (int32_t)sel_before;
  }
  if (tid == 0) {
    w.pick[row * 2] = us;
    w.pick[row * 2 + 1] = nd;
    w.ticket[row] = 0;  // ready for the next call
  }
  for (int i = tid; i < nb; i += kHtThreads) w.total[row * kHtBins + i] = 0;
}

// Exclusive prefix, in token order, of per-token flags held as c[j] = the count of
// the thread's four tokens of group j (token order: j, then thread, then e); the
// result, for each j, is the number of flagged tokens before the thread's group j.
// Uses tab[kHtPer][kHtThreads / 32]; contains two __syncthreads.
__device__ __forceinline__ void ht_order_scan(const uint32_t (&c)[kHtPer], uint32_t (&before)[kHtPer],
                                              uint32_t (*tab)[kHtThreads / 32], uint32_t& total) {
  constexpr int NW = kHtThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncwarp();  // the warp's reads of tab from a previous call come first
#pragma unroll
  for (int j = 0; j < kHtPer; ++j) {
    uint32_t incl = c[j];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    before[j] = incl - c[j];
    if (lane == 31) tab[j][warp] = incl;
  }
  __syncthreads();
  if (warp == 0) {  // (j, warp) entries in order: lane l takes entries 2l, 2l + 1
    static_assert(kHtPer * NW == 64, "one warp scans 64 entries");
    uint32_t* t = &tab[0][0];
    const uint32_t a = t[2 * lane], b = t[2 * lane + 1];
    uint32_t incl = a + b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t ex = incl - a - b;
    t[2 * lane] = ex;
    t[2 * lane + 1] = ex + a;
    if (lane == 31) t[64] = incl;  // the total, in the slot past the table
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kHtPer; ++j) before[j] += tab[j][warp];
  total = (&tab[0][0])[64];
}

template <int G>
__global__ void __launch_bounds__(kHtThreads)
hamming_pick_kernel(const uint32_t* __restrict__ sig, const uint32_t* __restrict__ qsig, HtGeo g,
                    bool vec, HtWs w, int32_t* __restrict__ idx, int64_t idx_stride,
                    int32_t* __restrict__ count) {
  __shared__ uint32_t tab[kHtPer + 1][kHtThreads / 32];  // + the total's slot
  const int p = blockIdx.x, tid = threadIdx.x;
  const int64_t row = blockIdx.y;
  const int b = (int)(row / g.Hkv), hh = (int)(row % g.Hkv);
  uint32_t qs[G];
#pragma unroll
  for (int gg = 0; gg < G; ++gg) qs[gg] = __ldg(qsig + (int64_t)b * g.Hq + hh * G + gg);
  const int64_t t0 = ht_range0(g, p);
  uint32_t u[kHtPer][4];
  ht_scores<G>(sig + row * g.ncap, qs, t0, g, vec, u);
  const uint32_t us = (uint32_t)__ldcg(w.pick + row * 2);
  const int nd = __ldcg(w.pick + row * 2 + 1);
  const int ties_before = __ldcg(w.before + (row * g.P + p) * 2);
  const int sel_before = __ldcg(w.before + (row * g.P + p) * 2 + 1);
  // ties in token order: the first (need - ties before) of the row are taken
  uint32_t c[kHtPer], tb[kHtPer], tot;
#pragma unroll
  for (int j = 0; j < kHtPer; ++j) {
    c[j] = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) c[j] += u[j][e] == us;
  }
  ht_order_scan(c, tb, tab, tot);
  const int budget = nd - ties_before;  // ties of this range to take, in order
  uint32_t sel[kHtPer];                 // bit e: token e of group j selected
#pragma unroll
  for (int j = 0; j < kHtPer; ++j) {
    uint32_t m = 0, r = tb[j];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool tie = u[j][e] == us;
      if (u[j][e] < us || (tie && (int)r < budget)) m |= 1u << e;
      r += tie;
    }
    sel[j] = m;
    c[j] = __popc(m);
  }
  uint32_t sb[kHtPer];
  ht_order_scan(c, sb, tab, tot);
  int32_t* irow = idx + row * idx_stride;
  const int lead = g.lead;
#pragma unroll
  for (int j = 0; j < kHtPer; ++j) {
    const int64_t i = t0 + 4 * (j * kHtThreads + tid);
    int pos = lead + sel_before + (int)sb[j];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (sel[j] & (1u << e)) irow[pos++] = (int32_t)(i + e);
  }
  if (p == 0) {  // the windows and the count
    const int M = g.tail - g.lead, kk = min(g.k, M), ntail = (int)(g.n - g.tail);
    for (int x = tid; x < lead; x += kHtThreads) irow[x] = x;
    for (int x = tid; x < ntail; x += kHtThreads) irow[lead + kk + x] = g.tail + x;
    if (tid == 0) count[row] = lead + kk + ntail;
  }
}

// ---------------------------------------------------------------------------------
struct HtLayout {
  size_t hist, total, ticket, pick, before, bytes;
};
static HtLayout ht_layout(int64_t rows, int P) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  HtLayout L;
  L.hist = 0;
  L.total = L.hist + al(sizeof(uint32_t) * rows * P * kHtBins);
  L.ticket = L.total + al(sizeof(uint32_t) * rows * kHtBins);
  L.pick = L.ticket + al(sizeof(uint32_t) * rows);
  L.before = L.pick + al(sizeof(int32_t) * rows * 2);
  L.bytes = L.before + al(sizeof(int32_t) * rows * P * 2);
  return L;
}

static HtGeo ht_geo(const Dims& s, const sd_select& sel) {
  HtGeo g;
  g.n = s.n;
  g.ncap = s.ncap;
  g.lead = (int)imin64(sel.sink, s.n);
  g.tail = (int)imax64(s.n - sel.local, g.lead);
  g.k = sel.k;
  const int64_t span = g.tail - (g.lead & ~3);
  g.P = (int)imax64(1, (span + kHtRange - 1) / kHtRange);
  g.Hq = s.Hq;
  g.Hkv = s.Hkv;
  return g;
}

size_t hamming_topk_workspace_bytes(const Dims& s, const sd_select& sel) {
  return ht_layout((int64_t)s.B * s.Hkv, ht_geo(s, sel).P).bytes;
}

bool hamming_topk_supported(const Dims& s, const sd_select& sel) {
  return sel.block == 1 && s.n < (1 << 30) && ht_geo(s, sel).P <= kHtThreads &&
         (int64_t)s.B * s.Hkv <= 65535;
}

template <int G>
static int ht_launch(const uint32_t* sig, const uint32_t* qsig, const HtGeo& g, bool vec, HtWs w,
                     int64_t rows, int32_t* idx, int64_t idx_stride, int32_t* count,
                     cudaStream_t st) {
  const dim3 grid((unsigned)g.P, (unsigned)rows);
  hamming_hist_kernel<G><<<grid, kHtThreads, 0, st>>>(sig, qsig, g, vec, w);
  hamming_pick_kernel<G><<<grid, kHtThreads, 0, st>>>(sig, qsig, g, vec, w, idx, idx_stride, count);
  note_launches(2);
  return check_launch("hamming_topk");
}

int launch_hamming_topk(const Dims& s, const uint32_t* sig, const uint32_t* qsig,
                        const sd_select& sel, int32_t* idx, int64_t idx_stride, int32_t* count,
                        void* ws, cudaStream_t st) {
  const int64_t rows = (int64_t)s.B * s.Hkv;
  const HtGeo g = ht_geo(s, sel);
  const HtLayout L = ht_layout(rows, g.P);
  uint8_t* base = (uint8_t*)ws;
  HtWs w;
  w.hist = (uint32_t*)(base + L.hist);
  w.total = (uint32_t*)(base + L.total);
  w.ticket = (uint32_t*)(base + L.ticket);
  w.pick = (int32_t*)(base + L.pick);
  w.before = (int32_t*)(base + L.before);
  // the row histograms and tickets start at zero (the last range of each row also
  // leaves them zero; this makes every call independent of the previous one)
  if (cudaMemsetAsync(base + L.total, 0, L.pick - L.total, st) != cudaSuccess)
    return check_launch("hamming_topk: workspace reset");
  const bool vec = (s.ncap % 4 == 0) && ((uintptr_t)sig % 16 == 0);
  switch (s.G) {
    case 1: return ht_launch<1>(sig, qsig, g, vec, w, rows, idx, idx_stride, count, st);
    case 2: return ht_launch<2>(sig, qsig, g, vec, w, rows, idx, idx_stride, count, st);
    case 4: return ht_launch<4>(sig, qsig, g, vec, w, rows, idx, idx_stride, count, st);
    default: return ht_launch<8>(sig, qsig, g, vec, w, rows, idx, idx_stride, count, st);
  }
}

}  // namespace sd
