// Bit-plane prefix scan fed by bulk copies (Fathom: Per-Query Read Depth for Sparse
// Decoding over Offloaded KV Caches, "bit planes per channel"): the kernel behind
// sd_score(SD_IDX_PLANES), sd_plan_score and sd_score_topk on 16-byte aligned
// layouts (n_cap % 512 == 0, 16-byte aligned planes and scales), for any n (a
// partial last 64-token block included).
//
// A token's score is
//   C_blk + sum over planned planes (j, p < t_j) of fl(qp_e * s_j,blk) * bit_jpi,
//   qp_e = q~_j * 2^(3-p),  C_blk = sum over active channels (slots, j ascending)
//   of fl(qo_j * s_j,blk),  qo_j = q~_j * (h(t_j) - 8),
// with q~ the group-summed query and s the channel's fp16 scale of the token's
// 64-token block: one bit test and one predicated add per planned plane and token.
//
// Work split: every CTA takes an equal contiguous range of 512-token units, walked
// as tiles that end at row ends; a tile's planned planes are consumed in chunks, in
// entry order (j ascending, then p).  Two geometries share one 20 KB slot:
//   WPL = 2 (the plain scan): a compute lane owns one 64-token scale block -- two
//     plane words and 64 accumulators -- so a warp's every plane step is 64
//     independent bit-test/add pairs behind one weight fold; tiles of 16,384
//     tokens, chunks of 8 planes;
//   WPL = 1 (the fused scan + top-k's candidate marks): a lane owns one word;
//     tiles of 8,192 tokens, chunks of 16 planes.
//
// Warp roles (288 threads, 2 CTAs per SM).  The producer warp builds a row's
// tables as it reaches the row -- the water-filled plan when it is computed here,
// the planned entries, the folded query values, each chunk's channels -- and posts
// every chunk into a ring of four slots: the lanes issue one bulk copy per planned
// plane's words and one per chunk channel's scales, all completing on the slot's
// mbarrier.  Eight compute warps work independently: per plane of each chunk they
// run the weight fold fl(qp_e * s), the bit tests and the predicated adds, and at a
// channel's first plane the constant's term fl(qo_j * s) (so C_blk adds up in
// channel order); at the tile's end they write their scores (and word maxima, or
// the fused top-k's hit masks).  Slots go back to the producer through "empty"
// mbarriers.  Every wait is bounded: one that runs out sets the library's device
// error word and ends the CTA's work.
#include <cuda_fp16.h>

#include "sd_planes.cuh"

namespace sd {

__device__ unsigned int g_scan_timeout = 0;  // set when a bounded wait of the scan ran out

namespace {

constexpr int kPtUnit = 512;             // tokens per unit of the work split
constexpr int kPtSlots = 4;
constexpr int kPtCompute = 256;
constexpr int kPtThreads = kPtCompute + 32;
constexpr int kPtCtasPerSm = 2;
constexpr int kPtRows = 2;               // rows one CTA's range may meet
constexpr uint32_t kPtSpin = 1u << 22;   // try_wait rounds before a wait gives up
constexpr int kInfoFirst = 1, kInfoLast = 2, kInfoEnd = 4;

template <int WPL>  // plane words per compute lane
struct PtGeo {
  static constexpr int kTile = 8192 * WPL;      // tokens per tile
  static constexpr int kWords = kTile / 32;     // words per plane and tile
  static constexpr int kBlocks = kTile / 64;    // scale blocks per tile
  static constexpr int kChunk = 16 / WPL;       // planned planes per slot
};

template <int WPL>
struct PtRow {  // one row's tables, padded to whole chunks
  // per planned entry e (j ascending, then p): (q~_j 2^(3-p), q~_j (h(t_j) - 8) at p = 0
  // else 0); entries past nact up to the chunk's end: (0, 0)
  float2 qq[4 * kD + PtGeo<WPL>::kChunk];
  // per entry: j * 4 + p; past nact: the last entry's (a real plane, copied with weight 0)
  uint16_t act[4 * kD + PtGeo<WPL>::kChunk];
  int nact;
};

struct PtInfo {  // a chunk, as the producer posts it
  int row;       // (sequence, KV head) row
  int tok0;      // the tile's first token
  int nwv;       // the tile's words holding tokens (even: whole 64-token blocks)
  int k;         // the chunk's index in the tile
  int ne;        // the chunk's entries
  int flags;     // kInfoFirst / kInfoLast / kInfoEnd
};

template <int WPL>
struct PtSlot {
  uint32_t words[PtGeo<WPL>::kChunk][PtGeo<WPL>::kWords];  // 16 KB: the planes' words
  uint16_t sc[PtGeo<WPL>::kChunk][PtGeo<WPL>::kBlocks];    // 4 KB: the chunk channels' scales
};

template <int WPL>
struct PtSmem {
  PtSlot<WPL> slot[kPtSlots];  // 80 KB
  PtRow<WPL> rows[kPtRows];
  int tbs[kPtRows][kD];        // the rows' plans (bits per channel), the producer's scratch
  PtInfo info[kPtSlots];
  unsigned long long full[kPtSlots], empty[kPtSlots];
  int abort;
};

__device__ __forceinline__ uint32_t su32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mb_init(unsigned long long* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mb_arrive(unsigned long long* b) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void mb_arrive_tx(unsigned long long* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n" ::"r"(su32(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mb_try(unsigned long long* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase of the given parity to complete; false once kPtSpin rounds ran
// out or another warp of the CTA gave up.
__device__ __forceinline__ bool mb_wait(int* abort, unsigned long long* b, uint32_t parity) {
  for (uint32_t i = 0; i < kPtSpin; ++i) {
    if (mb_try(b, parity)) return true;
    if (*(volatile int*)abort) return false;
  }
  *(volatile int*)abort = 1;
  atomicOr(&g_scan_timeout, 1u);
  return false;
}
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes,
                                          unsigned long long* b) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          su32(dst)),
      "l"(src), "r"(bytes), "r"(su32(b))
      : "memory");
}

// The CTA's range of units [u_begin, u_end) and its first row.
struct PtRange {
  int64_t u_begin, u_end;
  int bh0;
};
__device__ __forceinline__ PtRange pt_range(int upr, int64_t total_units) {
  PtRange r;
  r.u_begin = (int64_t)blockIdx.x * total_units / gridDim.x;
  r.u_end = (int64_t)(blockIdx.x + 1) * total_units / gridDim.x;
  r.bh0 = (int)(r.u_begin / upr);
  return r;
}

// The producer warp builds row bh's tables into D (lane l: channels 4 l .. 4 l + 3):
// the plan (computed here, ps_plan_row_warp, or read), the group-summed query q~_j
// (g ascending), the planned entries (j ascending, then p) with qp_e = q~_j 2^(3-p)
// and, at p = 0, qo = q~_j (h(t_j) - 8) -- the arithmetic of ps_build_row -- and
// the padding of the last chunk.  The plan is written when write_plan.  Later posts
// of the row's chunks publish the tables to the compute warps (the slots' barriers
// order the writes before them).
template <int G, int WPL>
__device__ __forceinline__ void pt_build_warp(PtRow<WPL>& D, int* tbs, int bh,
                                              const uint16_t* __restrict__ q,
                                              const uint8_t* __restrict__ plan, int Hq, int Hkv,
                                              const PsPlanIn& pl, bool write_plan) {
  constexpr int kChunk = PtGeo<WPL>::kChunk;
  const int lane = threadIdx.x & 31;
  const int b = bh / Hkv, h = bh % Hkv;
  float qt[4], mass[4], s2[4];  // q and sigma2 are loaded once, for the plan and the tables
  ps_load_row<G>(lane, q, pl.sigma2, b, h, Hq,
                 pl.on && (pl.mode == SD_PLAN_WATERFILL || pl.mode == SD_PLAN_FIXED), qt, mass, s2);
  if (pl.on) {
    ps_plan_lane(lane, mass, s2, pl.mode, pl.budget, tbs);
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c) tbs[lane * 4 + c] = min((int)plan[(int64_t)bh * kD + lane * 4 + c], 4);
  }
  __syncwarp();
  int tb[4], tot = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int j = lane * 4 + c;
    tb[c] = tbs[j];
    tot += tb[c];
    if (write_plan && pl.out) pl.out[(int64_t)bh * kD + j] = (uint8_t)tb[c];
  }
  int incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  int pos = incl - tot;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int j = lane * 4 + c;
    const float qo = __fmul_rn(qt[c], tb[c] < 4 ? (float)((1 << (3 - tb[c])) - 8) : -8.0f);
    for (int p = 0; p < tb[c]; ++p, ++pos) {
      D.act[pos] = (uint16_t)(j * 4 + p);
      D.qq[pos] = make_float2(ldexpf(qt[c], 3 - p), p == 0 ? qo : 0.0f);
    }
  }
  const int nact = __shfl_sync(0xFFFFFFFFu, incl, 31);
  __syncwarp();
  // padding to whole chunks: weight 0 on a real plane (the last entry's)
  const int npad = ((nact + kChunk - 1) / kChunk) * kChunk;
  if (nact > 0 && lane < npad - nact) {
    D.act[nact + lane] = D.act[nact - 1];
    D.qq[nact + lane] = make_float2(0.0f, 0.0f);
  }
  if (lane == 0) D.nact = nact;
  __syncwarp();
}

// The producer warp: posts every chunk of the CTA's range, then the end marker.
// Lane 0 waits for a free slot and posts its byte count and metadata; then lanes
// 0 .. kChunk-1 copy the chunk's planes and lanes 16 .. 16+kChunk-1 its channels'
// scales, side by side.  A tile holds the whole 64-token blocks of its units that
// hold tokens (nblk = ceil(n / 64) per row); copies are rounded up to 16 bytes
// inside the row's n_cap (a multiple of 512).
template <int G, int WPL>
__device__ __forceinline__ void pt_produce(PtSmem<WPL>& S, const uint32_t* __restrict__ planes,
                                           const uint16_t* __restrict__ scales, int64_t n,
                                           int64_t ncap, int upr, const PtRange& rg,
                                           const uint16_t* __restrict__ q,
                                           const uint8_t* __restrict__ plan, int Hq, int Hkv,
                                           const PsPlanIn& pl) {
  using Geo = PtGeo<WPL>;
  const int lane = threadIdx.x & 31;
  const uint32_t wstride = (uint32_t)(ncap / 32), sstride = (uint32_t)(ncap / 64);
  const int nblk = (int)((n + 63) / 64);  // blocks per row holding tokens
  int left = (int)(rg.u_end - rg.u_begin);
  int bh = rg.bh0;
  int ur = (int)(rg.u_begin - (int64_t)bh * upr);
  int c = 0;  // chunks posted
  int built = rg.bh0 - 1;  // the last row whose tables are built
  bool ok = true;
  auto wait0 = [&](unsigned long long* b, uint32_t parity) {  // lane 0 waits, the warp learns
    int r = 1;
    if (lane == 0) r = mb_wait(&S.abort, b, parity) ? 1 : 0;
    return __shfl_sync(0xFFFFFFFFu, r, 0) != 0;
  };
  while (left > 0 && ok) {
    const int nu = min(min(Geo::kTile / kPtUnit, upr - ur), left);
    const int tok0 = ur * kPtUnit;
    const int nbv = min(nu * (kPtUnit / 64), nblk - ur * (kPtUnit / 64));  // blocks with tokens
    const int nwv = 2 * nbv;
    const uint32_t wbytes = (uint32_t)((nwv + 3) & ~3) * 4;  // 16-byte multiples
    const uint32_t sbytes = (uint32_t)((nbv + 7) & ~7) * 2;
    if (bh != built) {  // a new row: its tables first (the row starts inside the range
      built = bh;       // when its first unit is the tile's)
      pt_build_warp<G, WPL>(S.rows[bh - rg.bh0], S.tbs[bh - rg.bh0], bh, q, plan, Hq, Hkv, pl,
                            ur == 0);
    }
    const PtRow<WPL>& R = S.rows[bh - rg.bh0];
    const int nact = R.nact;
    const uint32_t* pl_row = planes + (int64_t)bh * kD * 4 * wstride + tok0 / 32;
    const uint16_t* sc_row = scales + (int64_t)bh * kD * sstride + tok0 / 64;
    const int nck = max(1, (nact + Geo::kChunk - 1) / Geo::kChunk);
    for (int k = 0; k < nck; ++k, ++c) {
      const int s = c % kPtSlots;
      if (c >= kPtSlots && !(ok = wait0(&S.empty[s], ((c / kPtSlots) - 1) & 1))) break;
      const int ne = nact > 0 ? Geo::kChunk : 0;  // whole chunks (padded) or nothing
      if (lane == 0) {
        PtInfo& I = S.info[s];
        I.row = bh;
        I.tok0 = tok0;
        I.nwv = nwv;
        I.k = k;
        I.ne = ne;
        I.flags = (k == 0 ? kInfoFirst : 0) | (k == nck - 1 ? kInfoLast : 0);
        mb_arrive_tx(&S.full[s], ne * (wbytes + sbytes));
      }
      __syncwarp();
      const int ent = R.act[k * Geo::kChunk + (lane & 15)];
      if (lane < ne)  // the entry's plane words
        bulk_copy(&S.slot[s].words[lane][0], pl_row + (int64_t)ent * wstride, wbytes, &S.full[s]);
      else if (lane >= 16 && lane - 16 < ne)  // the entry's channel scales
        bulk_copy(&S.slot[s].sc[lane - 16][0], sc_row + (int64_t)(ent >> 2) * sstride, sbytes,
                  &S.full[s]);
    }
    left -= nu;
    ur += nu;
    if (ur == upr) { ur = 0; ++bh; }
  }
  if (ok) {  // the end marker
    const int s = c % kPtSlots;
    if (c < kPtSlots || wait0(&S.empty[s], ((c / kPtSlots) - 1) & 1)) {
      if (lane == 0) {
        S.info[s].flags = kInfoEnd;
        mb_arrive(&S.full[s]);
      }
    } else {
      ok = false;
    }
  }
  if (!ok && lane == 0) {
    // a wait ran out: let the copies already issued land before the CTA's shared
    // memory goes away (each slot's last posted phase)
    for (int x = max(0, c - kPtSlots); x < c; ++x)
      for (uint32_t i = 0; i < kPtSpin && !mb_try(&S.full[x % kPtSlots], (x / kPtSlots) & 1); ++i) {
      }
  }
}

// Writes a lane's 32 WPL scores of tokens tok .. (those < n) and, with wmax, the
// maxima of its WPL words (tokens >= n excluded; NaN if one of them is NaN).
template <int WPL>
__device__ __forceinline__ void pt_store(float (&acc)[32 * WPL], int row, int64_t tok, int64_t n,
                                         float* __restrict__ scores, float* __restrict__ wmax) {
  float* orow = scores + (int64_t)row * n + tok;
  if (tok + 32 * WPL <= n && (n & 3) == 0) {
    float4* o4 = reinterpret_cast<float4*>(orow);
#pragma unroll
    for (int k = 0; k < 8 * WPL; ++k)
      o4[k] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
  } else {
#pragma unroll
    for (int k = 0; k < 32 * WPL; ++k)
      if (tok + k < n) orow[k] = acc[k];
  }
  if (!wmax) return;
  const int64_t nw_out = (n + 31) / 32;
#pragma unroll
  for (int k = 0; k < 32 * WPL; ++k)
    if (tok + k >= n) acc[k] = -INFINITY;
#pragma unroll
  for (int hw = 0; hw < WPL; ++hw) {  // a tree of depth 5 in place: acc is reset by the next tile
    float* a = acc + 32 * hw;
#pragma unroll
    for (int w = 16; w > 0; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) a[i] = fmax_nan(a[i], a[i + w]);
    const int64_t word = tok / 32 + hw;
    if (word < nw_out) wmax[(int64_t)row * nw_out + word] = a[0];
  }
}

// The compute warps: every posted chunk until the end marker; lane l of warp w owns
// the tile's words (32 w + l) WPL .. + WPL - 1, i.e. scale block ((32 w + l) WPL) / 2.
template <bool CAND, int WPL>
__device__ __forceinline__ void pt_compute(PtSmem<WPL>& S, float* __restrict__ scores, int64_t n,
                                           const PsCand& cd, float* __restrict__ wmax, int bh0) {
  using Geo = PtGeo<WPL>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wl = (warp * 32 + lane) * WPL;  // the lane's first word of the tile
  const int blk = wl >> 1;                  // its scale block
  float acc[32 * WPL];
  float cb = 0.0f;  // C_blk of the lane's block
#pragma unroll
  for (int k = 0; k < 32 * WPL; ++k) acc[k] = 0.0f;
  for (int c = 0;; ++c) {
    const int s = c % kPtSlots;
    if (!mb_wait(&S.abort, &S.full[s], (c / kPtSlots) & 1)) return;
    const PtInfo I = S.info[s];
    if (I.flags & kInfoEnd) break;
    if (I.flags & kInfoFirst) {
#pragma unroll
      for (int k = 0; k < 32 * WPL; ++k) acc[k] = 0.0f;
      cb = 0.0f;
    }
    const bool active = warp * 32 * WPL < I.nwv;  // warps whose words all lie past the end idle
    if (active && I.ne) {
      const float2* qq = S.rows[I.row - bh0].qq + I.k * Geo::kChunk;
      const PtSlot<WPL>& sl = S.slot[s];
#pragma unroll
      for (int e = 0; e < Geo::kChunk; ++e) {  // whole chunks: padding entries weigh 0
        const float2 w = qq[e];
        const float sf = __half2float(reinterpret_cast<const __half*>(&sl.sc[e][0])[blk]);
        cb = __fadd_rn(cb, __fmul_rn(w.y, sf));  // fl(qo s) at a channel's first plane, else + 0
        const float wt = __fmul_rn(w.x, sf);
        if (WPL == 2) {
          const uint2 w2 = *reinterpret_cast<const uint2*>(&sl.words[e][wl]);
          ps_bits(*reinterpret_cast<float(*)[32]>(&acc[0]), w2.x, wt);
          ps_bits(*reinterpret_cast<float(*)[32]>(&acc[32 * (WPL - 1)]), w2.y, wt);
        } else {
          ps_bits(*reinterpret_cast<float(*)[32]>(&acc[0]), sl.words[e][wl], wt);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mb_arrive(&S.empty[s]);
    if ((I.flags & kInfoLast) && active) {
      const bool valid = wl < I.nwv;
#pragma unroll
      for (int k = 0; k < 32 * WPL; ++k) acc[k] += cb;
      if (valid)
        pt_store<WPL>(acc, I.row, (int64_t)I.tok0 + (int64_t)wl * 32, n, scores, CAND ? nullptr : wmax);
      if (CAND)  // warp-collective: every lane of an active warp takes part
        ps_mark(cd, I.row, __ldg(cd.thr + I.row), (int64_t)I.tok0 + wl * 32, valid,
                *reinterpret_cast<float(*)[32]>(&acc[0]));
    }
  }
}

template <int G, bool CAND, int WPL>
__global__ void __launch_bounds__(kPtThreads, kPtCtasPerSm)
score_planes_tma_kernel(const uint32_t* __restrict__ planes, const uint16_t* __restrict__ scales,
                        const uint8_t* __restrict__ plan, const uint16_t* __restrict__ q, int Hq,
                        int Hkv, int64_t n, int64_t ncap, int upr, int64_t total_units,
                        float* __restrict__ scores, PsCand cd, PsPlanIn pl,
                        float* __restrict__ wmax) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  PtSmem<WPL>& S = *reinterpret_cast<PtSmem<WPL>*>(smem_raw);
  const PtRange rg = pt_range(upr, total_units);  // meets <= kPtRows rows (host-checked)
  if (threadIdx.x == kPtCompute) {
    for (int s = 0; s < kPtSlots; ++s) {
      mb_init(&S.full[s], 1);
      mb_init(&S.empty[s], kPtCompute / 32);
    }
    S.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();  // the barriers are initialised
  if (threadIdx.x >= kPtCompute) {
    pt_produce<G, WPL>(S, planes, scales, n, ncap, upr, rg, q, plan, Hq, Hkv, pl);
    return;
  }
  pt_compute<CAND, WPL>(S, scores, n, cd, wmax, rg.bh0);
}

template <int G, bool CAND, int WPL>
int pt_launch(const Dims& s, const uint32_t* planes, const uint16_t* scales, const uint8_t* plan,
              const uint16_t* q, float* scores, const PsCand& cd, const PsPlanIn& pl, float* wmax,
              int grid, int upr, int64_t total, cudaStream_t st) {
  auto kern = score_planes_tma_kernel<G, CAND, WPL>;
  if (int rc = set_smem_limit((const void*)kern, sizeof(PtSmem<WPL>),
                              "score_planes_tma: smem attribute"))
    return rc;
  kern<<<(unsigned)grid, kPtThreads, sizeof(PtSmem<WPL>), st>>>(
      planes, scales, plan, q, s.Hq, s.Hkv, s.n, s.ncap, upr, total, scores, cd, pl, wmax);
  note_launches(1);
  return check_launch("score_planes_tma");
}

}  // namespace

// Reads this GPU's scan error word after the work on `st`, then clears it (both
// ordered on `st`; the host waits for the stream).
int scan_error_take(cudaStream_t st, unsigned* word) {
  *word = 0;
  unsigned zero = 0;
  if (cudaMemcpyFromSymbolAsync(word, g_scan_timeout, sizeof(unsigned), 0,
                                cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return check_launch("device status: read");
  if (*word &&
      (cudaMemcpyToSymbolAsync(g_scan_timeout, &zero, sizeof(unsigned), 0,
                               cudaMemcpyHostToDevice, st) != cudaSuccess ||
       cudaStreamSynchronize(st) != cudaSuccess))
    return check_launch("device status: clear");
  return SD_OK;
}

// Sets the word as a scan whose bounded wait ran out would (for testing the report).
int scan_error_set(unsigned word, cudaStream_t st) {
  if (cudaMemcpyToSymbolAsync(g_scan_timeout, &word, sizeof(unsigned), 0, cudaMemcpyHostToDevice,
                              st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return check_launch("device status: set");
  return SD_OK;
}

// The bulk-copy scan applies when every CTA's range meets at most two rows; returns
// 1 (not launched) otherwise.  Layouts must be 16-byte aligned (planes_aligned).
int launch_score_planes_tma(const Dims& s, const uint32_t* planes, const uint16_t* scales,
                            const uint8_t* plan, const uint16_t* q, float* scores,
                            const PsCand* cand, const PsPlanIn* plan_in, float* wmax, int sms,
                            cudaStream_t st) {
  const int upr = (int)((s.n + kPtUnit - 1) / kPtUnit);  // units per row (n < 2^31)
  const int64_t total = (int64_t)upr * s.B * s.Hkv;
  int grid = (int)imin64(total, (int64_t)sms * kPtCtasPerSm);
  // whole CTAs per row where that gives up at most a tenth of the grid: then no range
  // meets two rows, whose second row's tables a CTA would build in mid-range while
  // its compute warps wait
  const int64_t rows = (int64_t)s.B * s.Hkv;
  if (rows < grid) {
    const int64_t per = grid / rows;
    if (per * rows * 10 >= (int64_t)grid * 9 && per <= upr) grid = (int)(per * rows);
  }
  for (int b = 0; b < grid; ++b) {  // rows met by each CTA's range
    const int64_t u0 = (int64_t)b * total / grid, u1 = (int64_t)(b + 1) * total / grid;
    if (u1 > u0 && (u1 - 1) / upr - u0 / upr + 1 > kPtRows) return 1;
  }
  const PsPlanIn pl = plan_in ? *plan_in : PsPlanIn{};
  const PsCand none{};
  if (cand) {
    switch (s.G) {
      case 1: return pt_launch<1, true, 1>(s, planes, scales, plan, q, scores, *cand, pl, nullptr, grid, upr, total, st);
      case 2: return pt_launch<2, true, 1>(s, planes, scales, plan, q, scores, *cand, pl, nullptr, grid, upr, total, st);
      case 4: return pt_launch<4, true, 1>(s, planes, scales, plan, q, scores, *cand, pl, nullptr, grid, upr, total, st);
      default: return pt_launch<8, true, 1>(s, planes, scales, plan, q, scores, *cand, pl, nullptr, grid, upr, total, st);
    }
  }
  // a CTA whose range is under one 16K-token tile keeps every lane busy with one
  // word per lane (8K-token tiles); longer ranges take a block per lane
  if (total * kPtUnit / grid < PtGeo<2>::kTile) {
    switch (s.G) {
      case 1: return pt_launch<1, false, 1>(s, planes, scales, plan, q, scores, none, pl, wmax, grid, upr, total, st);
      case 2: return pt_launch<2, false, 1>(s, planes, scales, plan, q, scores, none, pl, wmax, grid, upr, total, st);
      case 4: return pt_launch<4, false, 1>(s, planes, scales, plan, q, scores, none, pl, wmax, grid, upr, total, st);
      default: return pt_launch<8, false, 1>(s, planes, scales, plan, q, scores, none, pl, wmax, grid, upr, total, st);
    }
  }
  switch (s.G) {
    case 1: return pt_launch<1, false, 2>(s, planes, scales, plan, q, scores, none, pl, wmax, grid, upr, total, st);
    case 2: return pt_launch<2, false, 2>(s, planes, scales, plan, q, scores, none, pl, wmax, grid, upr, total, st);
    case 4: return pt_launch<4, false, 2>(s, planes, scales, plan, q, scores, none, pl, wmax, grid, upr, total, st);
    default: return pt_launch<8, false, 2>(s, planes, scales, plan, q, scores, none, pl, wmax, grid, upr, total, st);
  }
}

}  // namespace sd
