// Bit-plane prefix scan fed by bulk copies (Fathom: Per-Query Read Depth for Sparse
// Decoding over Offloaded KV Caches, "bit planes per channel"): the kernel behind
// sd_score(SD_IDX_PLANES), sd_plan_score and sd_score_topk on 16-byte aligned
// layouts (n_cap % 512 == 0, 16-byte aligned planes and scales).
//
// A token's score is
//   C_blk + sum over planned planes (j, p < t_j) of fl(qp_e * s_j,blk) * bit_jpi,
//   qp_e = q~_j * 2^(3-p),  C_blk = sum over active channels (slots, j ascending)
//   of fl(qo_j * s_j,blk),  qo_j = q~_j * (h(t_j) - 8),
// with q~ the group-summed query and s the channel's fp16 scale of the token's
// 64-token block: one bit test and one predicated add per planned plane and token.
//
// Work split as the cp.async kernel: every CTA takes an equal contiguous range of
// 512-token units, walked as tiles of at most 8192 tokens that end at row ends; a
// tile's planned planes are consumed in chunks of up to 16, in entry order (j
// ascending, then p).
//
// Warp roles (288 threads, 2 CTAs per SM).  Before the pipeline starts, two groups
// of 128 threads build the tables of the (at most two) rows the range meets -- the
// water-filled plan when it is computed here, the planned entries, the folded
// query values, each chunk's channels -- in parallel.  Then the producer warp
// posts every chunk into a ring of four slots: the lanes issue one bulk copy per
// planned plane's words and one per chunk channel's scales, all completing on the
// slot's mbarrier.  Eight compute warps work independently: warp w owns words
// 32 w .. 32 w + 31 of the tile (lane l one word, 32 tokens of one scale block) and
// runs, per plane of each chunk, the weight fold fl(qp_e * s), the bit tests and
// the predicated adds, and at a channel's first plane the constant's term
// fl(qo_j * s) (so C_blk adds up in channel order); at the tile's end it writes
// its scores (and word maxima, or the fused top-k's hit masks).  Slots go back to
// the producer through "empty" mbarriers.  Every wait is bounded: one that runs
// out sets the library's device error word and ends the CTA's work.
#include <cuda_fp16.h>

#include "sd_planes.cuh"

namespace sd {

__device__ unsigned int g_scan_timeout = 0;  // set when a bounded wait of the scan ran out

namespace {

constexpr int kPtTile = 8192;
constexpr int kPtUnit = 512;
constexpr int kPtWords = kPtTile / 32;   // 256
constexpr int kPtBlocks = kPtTile / 64;  // 128
constexpr int kPtChunk = 16;             // planned planes per slot
constexpr int kPtMaxChunks = 4 * kD / kPtChunk;
constexpr int kPtSlots = 4;
constexpr int kPtCompute = 256;
constexpr int kPtThreads = kPtCompute + 32;
constexpr int kPtCtasPerSm = 2;
constexpr int kPtRows = 2;               // rows one CTA's range may meet
constexpr uint32_t kPtSpin = 1u << 22;   // try_wait rounds before a wait gives up
constexpr int kInfoFirst = 1, kInfoLast = 2, kInfoEnd = 4;

struct PtRow {                       // one row's tables
  float qp[4 * kD];                  // per planned entry e: q~_j * 2^(3-p)
  float qo[4 * kD];                  // per entry with p = 0: q~_j * (h(t_j) - 8)
  uint16_t act[4 * kD];              // per entry: j * 4 + p (j ascending, then p)
  uint8_t cs[4 * kD];                // per entry: its channel's place in the chunk's list
  uint8_t chl[kPtMaxChunks][kPtChunk];  // per chunk: its distinct channels, ascending
  uint8_t nchl[kPtMaxChunks];
  int nact;
};

struct PtInfo {  // a chunk, as the producer posts it
  int row;       // (sequence, KV head) row
  int tok0;      // the tile's first token
  int nwv;       // the tile's valid words
  int k;         // the chunk's index in the tile (entries 16 k ..)
  int ne;        // the chunk's entries
  int flags;     // kInfoFirst / kInfoLast / kInfoEnd
};

struct PtSlot {
  uint32_t words[kPtChunk][kPtWords];  // 16 KB: the planes' words
  uint16_t sc[kPtChunk][kPtBlocks];    // 4 KB: the chunk channels' scales
};

struct PtSmem {
  PtSlot slot[kPtSlots];  // 80 KB
  PtRow rows[kPtRows];
  int tbs[kD];            // the producer's plan scratch
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
__device__ __forceinline__ bool mb_wait(PtSmem& S, unsigned long long* b, uint32_t parity) {
  for (uint32_t i = 0; i < kPtSpin; ++i) {
    if (mb_try(b, parity)) return true;
    if (*(volatile int*)&S.abort) return false;
  }
  *(volatile int*)&S.abort = 1;
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
// and, at p = 0, qo = q~_j (h(t_j) - 8), and each chunk's distinct channels -- the
// arithmetic of ps_build_row.  The plan is written when write_plan.  Later posts
// of the row's chunks publish the tables to the compute warps (the slots' barriers
// order the writes before them).
template <int G>
__device__ __forceinline__ void pt_build_warp(PtRow& D, int* tbs, int bh,
                                              const uint16_t* __restrict__ q,
                                              const uint8_t* __restrict__ plan, int Hq, int Hkv,
                                              const PsPlanIn& pl, bool write_plan) {
  const int lane = threadIdx.x & 31;
  const int b = bh / Hkv, h = bh % Hkv;
  if (pl.on) {
    ps_plan_row_warp<G>(lane, q, pl.sigma2, b, h, Hq, pl.mode, pl.budget, tbs);
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c) tbs[lane * 4 + c] = min((int)plan[(int64_t)bh * kD + lane * 4 + c], 4);
  }
  __syncwarp();
  int tb[4], tot = 0;
  float qt[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int j = lane * 4 + c;
    tb[c] = tbs[j];
    tot += tb[c];
    float a = 0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g)
      a = __fadd_rn(a, bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + j]));
    qt[c] = a;
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
      D.qp[pos] = ldexpf(qt[c], 3 - p);
      D.qo[pos] = p == 0 ? qo : 0.0f;
    }
  }
  const int nact = __shfl_sync(0xFFFFFFFFu, incl, 31);
  __syncwarp();
  // each chunk's distinct channels (entries of one channel are consecutive)
  for (int k = lane; k * kPtChunk < nact; k += 32) {
    int nc = 0, prev = -1;
    for (int e = k * kPtChunk; e < min(nact, (k + 1) * kPtChunk); ++e) {
      const int j = D.act[e] >> 2;
      if (j != prev) {
        D.chl[k][nc++] = (uint8_t)j;
        prev = j;
      }
      D.cs[e] = (uint8_t)(nc - 1);
    }
    D.nchl[k] = (uint8_t)nc;
  }
  if (lane == 0) D.nact = nact;
  __syncwarp();
}

// The producer warp: posts every chunk of the CTA's range, then the end marker.
// Lane 0 waits for a free slot and posts its byte count and metadata; then lanes
// 0-15 copy the chunk's planes and lanes 16-31 its channels' scales, side by side.
template <int G>
__device__ __forceinline__ void pt_produce(PtSmem& S, const uint32_t* __restrict__ planes,
                                           const uint16_t* __restrict__ scales, int64_t n,
                                           int64_t ncap, int upr, const PtRange& rg,
                                           const uint16_t* __restrict__ q,
                                           const uint8_t* __restrict__ plan, int Hq, int Hkv,
                                           const PsPlanIn& pl) {
  const int lane = threadIdx.x & 31;
  const uint32_t wstride = (uint32_t)(ncap / 32), sstride = (uint32_t)(ncap / 64);
  const int n32 = (int)(n / 32);
  int left = (int)(rg.u_end - rg.u_begin);
  int bh = rg.bh0;
  int ur = (int)(rg.u_begin - (int64_t)bh * upr);
  int c = 0;  // chunks posted
  int built = rg.bh0 - 1;  // the last row whose tables are built
  bool ok = true;
  auto wait0 = [&](unsigned long long* b, uint32_t parity) {  // lane 0 waits, the warp learns
    int r = 1;
    if (lane == 0) r = mb_wait(S, b, parity) ? 1 : 0;
    return __shfl_sync(0xFFFFFFFFu, r, 0) != 0;
  };
  while (left > 0 && ok) {
    const int nu = min(min(kPtTile / kPtUnit, upr - ur), left);
    const int tok0 = ur * kPtUnit;
    const int nwv = min(nu * (kPtUnit / 32), n32 - ur * (kPtUnit / 32));  // valid words (even)
    const uint32_t wbytes = (uint32_t)((nwv + 3) & ~3) * 4;           // 16-byte multiples
    const uint32_t sbytes = (uint32_t)(((nwv / 2) + 7) & ~7) * 2;
    if (bh != built) {  // a new row: its tables first (the row starts inside the range
      built = bh;       // when its first unit is the tile's)
      pt_build_warp<G>(S.rows[bh - rg.bh0], S.tbs, bh, q, plan, Hq, Hkv, pl, ur == 0);
    }
    const PtRow& R = S.rows[bh - rg.bh0];
    const int nact = R.nact;
    const uint32_t* pl_row = planes + (int64_t)bh * kD * 4 * wstride + tok0 / 32;
    const uint16_t* sc_row = scales + (int64_t)bh * kD * sstride + tok0 / 64;
    const int nck = max(1, (nact + kPtChunk - 1) / kPtChunk);
    for (int k = 0; k < nck; ++k, ++c) {
      const int s = c % kPtSlots;
      if (c >= kPtSlots && !(ok = wait0(&S.empty[s], ((c / kPtSlots) - 1) & 1))) break;
      const int ne = max(0, min(kPtChunk, nact - k * kPtChunk));
      const int nc = ne ? R.nchl[k] : 0;
      if (lane == 0) {
        PtInfo& I = S.info[s];
        I.row = bh;
        I.tok0 = tok0;
        I.nwv = nwv;
        I.k = k;
        I.ne = ne;
        I.flags = (k == 0 ? kInfoFirst : 0) | (k == nck - 1 ? kInfoLast : 0);
        mb_arrive_tx(&S.full[s], ne * wbytes + nc * sbytes);
      }
      __syncwarp();
      if (lane < ne)
        bulk_copy(&S.slot[s].words[lane][0],
                  pl_row + (int64_t)R.act[k * kPtChunk + lane] * wstride, wbytes, &S.full[s]);
      else if (lane >= kPtChunk && lane - kPtChunk < nc)
        bulk_copy(&S.slot[s].sc[lane - kPtChunk][0],
                  sc_row + (int64_t)R.chl[k][lane - kPtChunk] * sstride, sbytes, &S.full[s]);
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

// The compute warps: every posted chunk until the end marker; warp w owns the
// tile's words 32 w .. 32 w + 31.
template <bool CAND>
__device__ __forceinline__ void pt_compute(PtSmem& S, float* __restrict__ scores, int64_t n,
                                           const PsCand& cd, float* __restrict__ wmax, int bh0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wl = warp * 32 + lane;  // the lane's word of the tile
  const int blk = wl >> 1;          // its scale block
  float acc[32];
  float cb = 0.0f;  // C_blk of the lane's block
#pragma unroll
  for (int k = 0; k < 32; ++k) acc[k] = 0.0f;
  for (int c = 0;; ++c) {
    const int s = c % kPtSlots;
    if (!mb_wait(S, &S.full[s], (c / kPtSlots) & 1)) return;
    const PtInfo I = S.info[s];
    if (I.flags & kInfoEnd) break;
    if (I.flags & kInfoFirst) {
#pragma unroll
      for (int k = 0; k < 32; ++k) acc[k] = 0.0f;
      cb = 0.0f;
    }
    const bool active = warp * 32 < I.nwv;  // warps whose words all lie past the end idle
    if (active) {
      const PtRow& R = S.rows[I.row - bh0];
      const PtSlot& sl = S.slot[s];
      const int e0 = I.k * kPtChunk;
#pragma unroll 4  // 45.7 us at 1M tokens, against 49.8 (2) and 51.9 (1); 8, 16: 45.7
      for (int e = 0; e < I.ne; ++e) {
        const int ee = e0 + e;
        const float sf = __half2float(reinterpret_cast<const __half*>(&sl.sc[R.cs[ee]][0])[blk]);
        if ((R.act[ee] & 3) == 0) cb = __fadd_rn(cb, __fmul_rn(R.qo[ee], sf));
        ps_bits(acc, sl.words[e][wl], __fmul_rn(R.qp[ee], sf));
      }
    }
    __syncwarp();
    if (lane == 0) mb_arrive(&S.empty[s]);
    if ((I.flags & kInfoLast) && active) {
      const bool valid = wl < I.nwv;
      float4* orow = reinterpret_cast<float4*>(scores + (int64_t)I.row * n + I.tok0 + wl * 32);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        acc[4 * k] += cb;
        acc[4 * k + 1] += cb;
        acc[4 * k + 2] += cb;
        acc[4 * k + 3] += cb;
        if (valid) orow[k] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
      }
      if (CAND) {
        ps_mark(cd, I.row, __ldg(cd.thr + I.row), (int64_t)I.tok0 + wl * 32, valid, acc);
      } else if (wmax) {  // a tree of depth 5 in place: acc is reset by the next tile
#pragma unroll
        for (int w = 16; w > 0; w >>= 1)
#pragma unroll
          for (int i = 0; i < w; ++i) acc[i] = fmax_nan(acc[i], acc[i + w]);
        if (valid) wmax[(int64_t)I.row * (n >> 5) + (I.tok0 >> 5) + wl] = acc[0];
      }
    }
  }
}

template <int G, bool CAND>
__global__ void __launch_bounds__(kPtThreads, kPtCtasPerSm)
score_planes_tma_kernel(const uint32_t* __restrict__ planes, const uint16_t* __restrict__ scales,
                        const uint8_t* __restrict__ plan, const uint16_t* __restrict__ q, int Hq,
                        int Hkv, int64_t n, int64_t ncap, int upr, int64_t total_units,
                        float* __restrict__ scores, PsCand cd, PsPlanIn pl,
                        float* __restrict__ wmax) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  PtSmem& S = *reinterpret_cast<PtSmem*>(smem_raw);
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
    pt_produce<G>(S, planes, scales, n, ncap, upr, rg, q, plan, Hq, Hkv, pl);
    return;
  }
  pt_compute<CAND>(S, scores, n, cd, wmax, rg.bh0);
}

template <int G, bool CAND>
int pt_launch(const Dims& s, const uint32_t* planes, const uint16_t* scales, const uint8_t* plan,
              const uint16_t* q, float* scores, const PsCand& cd, const PsPlanIn& pl, float* wmax,
              int grid, int upr, int64_t total, cudaStream_t st) {
  auto kern = score_planes_tma_kernel<G, CAND>;
  if (int rc = set_smem_limit((const void*)kern, sizeof(PtSmem), "score_planes_tma: smem attribute"))
    return rc;
  kern<<<(unsigned)grid, kPtThreads, sizeof(PtSmem), st>>>(planes, scales, plan, q, s.Hq, s.Hkv, s.n,
                                                           s.ncap, upr, total, scores, cd, pl, wmax);
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
  const int grid = (int)imin64(total, (int64_t)sms * kPtCtasPerSm);
  for (int b = 0; b < grid; ++b) {  // rows met by each CTA's range
    const int64_t u0 = (int64_t)b * total / grid, u1 = (int64_t)(b + 1) * total / grid;
    if (u1 > u0 && (u1 - 1) / upr - u0 / upr + 1 > kPtRows) return 1;
  }
  const PsPlanIn pl = plan_in ? *plan_in : PsPlanIn{};
  const PsCand none{};
  if (cand) {
    switch (s.G) {
      case 1: return pt_launch<1, true>(s, planes, scales, plan, q, scores, *cand, pl, nullptr, grid, upr, total, st);
      case 2: return pt_launch<2, true>(s, planes, scales, plan, q, scores, *cand, pl, nullptr, grid, upr, total, st);
      case 4: return pt_launch<4, true>(s, planes, scales, plan, q, scores, *cand, pl, nullptr, grid, upr, total, st);
      default: return pt_launch<8, true>(s, planes, scales, plan, q, scores, *cand, pl, nullptr, grid, upr, total, st);
    }
  }
  switch (s.G) {
    case 1: return pt_launch<1, false>(s, planes, scales, plan, q, scores, none, pl, wmax, grid, upr, total, st);
    case 2: return pt_launch<2, false>(s, planes, scales, plan, q, scores, none, pl, wmax, grid, upr, total, st);
    case 4: return pt_launch<4, false>(s, planes, scales, plan, q, scores, none, pl, wmax, grid, upr, total, st);
    default: return pt_launch<8, false>(s, planes, scales, plan, q, scores, none, pl, wmax, grid, upr, total, st);
  }
}

}  // namespace sd
