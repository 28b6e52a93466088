// Bit-plane prefix scan, direct-streaming form (Fathom: Per-Query Read Depth for
// Sparse Decoding over Offloaded KV Caches, "bit planes per channel" and "per-query
// reverse water-filling"): the kernel behind sd_score(SD_IDX_PLANES) and
// sd_plan_score, for any n (a partial last 64-token block included).
//
// A token's score is
//   C_blk + sum over planned planes (j, p < t_j) of fl(qp_e * s_j,blk) * bit_jpi,
//   qp_e = q~_j * 2^(3-p),  C_blk = sum over active channels (j ascending) of
//   fl(qo_j * s_j,blk),  qo_j = q~_j * (h(t_j) - 8),
// with q~ the group-summed query and s the channel's fp16 scale of the token's
// 64-token block: one bit test and one predicated add per planned plane and token,
// in the same order as the bulk-copy kernel (so both give the same bits).
//
// Work split.  The (row, 64-token block) pairs of all rows are cut into equal
// contiguous ranges, one per CTA; the grid has at least as many CTAs as there are
// rows, so a range holds at most a row's worth of blocks and meets at most two rows.
// Warps take passes of up to 32 blocks of one row from a shared counter; lane l of
// a pass owns one block: its two plane words per planned plane (64 tokens) and its
// scale.  No warp waits for another after the prologue.
//
// Memory.  Right after the read plan is known, the CTA issues L2 bulk prefetches of
// every planned plane's words and every active channel's scales over its whole
// range, so HBM streams at its own rate while the warps compute.  Each lane keeps
// the words and scales of the next kDrDepth planned planes in flight in registers.
//
// Prologue.  Warps 0 and 1 build the tables of the (at most two) rows the range
// meets, in parallel: the read plan (computed here, ps_plan_row_warp, or read), the
// group-summed query, and per planned entry e (j ascending, then p) the word and
// scale offsets of its plane and channel, qp_e and (at p = 0) qo_j.
#include <cuda_fp16.h>

#include "sd_planes.cuh"

namespace sd {
namespace {

constexpr int kDrThreads = 512;  // 16 warps
constexpr int kDrDepth = 4;      // planned planes in flight per lane
constexpr int kDrPass = 32;      // blocks per pass (one per lane)

struct DrEnt {       // one planned entry (j, p)
  uint32_t poff;     // word offset of plane j * 4 + p within the row's planes
  uint32_t soff;     // element offset of channel j's scales within the row's scales
  float qp;          // q~_j * 2^(3-p)
  float qo;          // q~_j * (h(t_j) - 8) at p = 0, else 0
};

struct DrRow {
  DrEnt e[4 * kD];
  int nact;
};

struct DrSmem {
  DrRow rows[2];
  int tbs[2][kD];
  int next_pass;
};

// One warp builds row bh's tables (lane l: channels 4 l .. 4 l + 3), the arithmetic
// of pt_build_warp / ps_build_row: q~_j summed over g ascending, qp = ldexp(q~, 3-p),
// qo = fl(q~ (h(t) - 8)).  The plan is written to pl.out when write_plan.
template <int G>
__device__ __forceinline__ void dr_build_row(DrRow& D, int* tbs, int bh,
                                             const uint16_t* __restrict__ q,
                                             const uint8_t* __restrict__ plan, int Hq, int Hkv,
                                             uint32_t wstride, uint32_t sstride,
                                             const PsPlanIn& pl, bool write_plan) {
  const int lane = threadIdx.x & 31;
  const int b = bh / Hkv, h = bh % Hkv;
  if (pl.on) {
    ps_plan_row_warp<G>(lane, q, pl.sigma2, b, h, Hq, pl.mode, pl.budget, tbs);
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      tbs[lane * 4 + c] = min((int)plan[(int64_t)bh * kD + lane * 4 + c], 4);
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
      DrEnt E;
      E.poff = (uint32_t)(j * 4 + p) * wstride;
      E.soff = (uint32_t)j * sstride;
      E.qp = ldexpf(qt[c], 3 - p);
      E.qo = p == 0 ? qo : 0.0f;
      D.e[pos] = E;
    }
  }
  if (lane == 31) D.nact = incl;
  __syncwarp();
}

__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

// A byte range [lo, hi) of one buffer, rounded outward to 16 bytes and clamped to
// the buffer's 16-byte aligned interior [blo, bhi): what a bulk prefetch may name
// (its address and size must be multiples of 16) without leaving the buffer.
__device__ __forceinline__ void l2_prefetch_range(uintptr_t lo, uintptr_t hi, uintptr_t blo,
                                                  uintptr_t bhi) {
  lo = lo & ~(uintptr_t)15;
  hi = (hi + 15) & ~(uintptr_t)15;
  if (lo < blo) lo = blo;
  if (hi > bhi) hi = bhi;
  if (hi > lo) l2_prefetch((const void*)lo, (uint32_t)(hi - lo));
}

// Prefetches into L2 the planned planes' words and active channels' scales of row
// portion [blk0, blk1) (row-local blocks), entries e = first, first + step, ...
// [pb_lo, pb_hi) and [sb_lo, sb_hi) are the planes' and scales' aligned interiors.
__device__ __forceinline__ void dr_prefetch(const DrRow& R, const uint32_t* prow,
                                            const uint16_t* srow, int64_t blk0, int64_t blk1,
                                            int first, int step, uintptr_t pb_lo,
                                            uintptr_t pb_hi, uintptr_t sb_lo, uintptr_t sb_hi) {
  if (blk1 <= blk0) return;
  for (int e = first; e < R.nact; e += step) {
    const DrEnt E = R.e[e];
    const uintptr_t w = (uintptr_t)(prow + E.poff);
    l2_prefetch_range(w + 8 * blk0, w + 8 * blk1, pb_lo, pb_hi);  // words 2 blk0 .. 2 blk1
    if (e == 0 || R.e[e - 1].soff != E.soff) {                    // a channel's first entry
      const uintptr_t c = (uintptr_t)(srow + E.soff);
      l2_prefetch_range(c + 2 * blk0, c + 2 * blk1, sb_lo, sb_hi);
    }
  }
}

__device__ __forceinline__ uint2 ldg_u2(const uint32_t* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_u16(const uint16_t* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];\n" : "=h"(v) : "l"(p));
  return v;
}

template <int G>
__global__ void __launch_bounds__(kDrThreads, 1)
score_planes_direct_kernel(const uint32_t* __restrict__ planes, const uint16_t* __restrict__ scales,
                           const uint8_t* __restrict__ plan, const uint16_t* __restrict__ q,
                           int Hq, int Hkv, int64_t n, int64_t ncap, int64_t nbr,
                           int64_t total_blocks, float* __restrict__ scores, PsPlanIn pl,
                           float* __restrict__ wmax) {
  __shared__ DrSmem S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t b0 = (int64_t)blockIdx.x * total_blocks / gridDim.x;
  const int64_t b1 = (int64_t)(blockIdx.x + 1) * total_blocks / gridDim.x;
  if (b1 <= b0) return;
  const int r0 = (int)(b0 / nbr), r1 = (int)((b1 - 1) / nbr);  // r1 <= r0 + 1
  const uint32_t wstride = (uint32_t)(ncap / 32), sstride = (uint32_t)(ncap / 64);
  if (warp < 2 && r0 + warp <= r1) {
    const int bh = r0 + warp;
    // the plan is written by the CTA holding the row's first block
    dr_build_row<G>(S.rows[warp], S.tbs[warp], bh, q, plan, Hq, Hkv, wstride, sstride, pl,
                    b0 <= (int64_t)bh * nbr);
  }
  if (threadIdx.x == 0) S.next_pass = 0;
  __syncthreads();
  // the row portions: [s0, e0) of row r0, [e0, b1) of row r1 (empty when r1 == r0)
  const int64_t e0 = imin64(b1, (int64_t)(r0 + 1) * nbr);
  const int P0 = (int)((e0 - b0 + kDrPass - 1) / kDrPass);
  const int P1 = (int)((b1 - e0 + kDrPass - 1) / kDrPass);
  if (lane == 0) {  // L2 prefetch of the whole range: every warp takes every 16th entry
    const int64_t rows = total_blocks / nbr;
    const uintptr_t pb = (uintptr_t)planes, sb = (uintptr_t)scales;
    const uintptr_t pb_lo = (pb + 15) & ~(uintptr_t)15;
    const uintptr_t pb_hi = (pb + (uintptr_t)(rows * kD * 4 * wstride) * 4) & ~(uintptr_t)15;
    const uintptr_t sb_lo = (sb + 15) & ~(uintptr_t)15;
    const uintptr_t sb_hi = (sb + (uintptr_t)(rows * kD * sstride) * 2) & ~(uintptr_t)15;
    const int64_t rb0 = (int64_t)r0 * nbr;
    dr_prefetch(S.rows[0], planes + (int64_t)r0 * kD * 4 * wstride,
                scales + (int64_t)r0 * kD * sstride, b0 - rb0, e0 - rb0, warp, kDrThreads / 32,
                pb_lo, pb_hi, sb_lo, sb_hi);
    if (r1 != r0) {
      const int64_t rb1 = (int64_t)r1 * nbr;
      dr_prefetch(S.rows[1], planes + (int64_t)r1 * kD * 4 * wstride,
                  scales + (int64_t)r1 * kD * sstride, e0 - rb1, b1 - rb1, warp, kDrThreads / 32,
                  pb_lo, pb_hi, sb_lo, sb_hi);
    }
  }
  const int64_t nw_out = (n + 31) / 32;  // word maxima per row
  for (;;) {
    int p = 0;
    if (lane == 0) p = atomicAdd(&S.next_pass, 1);
    p = __shfl_sync(0xFFFFFFFFu, p, 0);
    if (p >= P0 + P1) break;
    const int ri = p < P0 ? 0 : 1;
    const int row = r0 + ri;
    const int64_t start = ri == 0 ? b0 + (int64_t)kDrPass * p : e0 + (int64_t)kDrPass * (p - P0);
    const int64_t end = imin64(start + kDrPass, ri == 0 ? e0 : b1);
    const bool valid = start + lane < end;
    // row-local block of the lane (a lane past the end reads the pass's first block)
    const int64_t blk = (valid ? start + lane : start) - (int64_t)row * nbr;
    const DrRow& R = S.rows[ri];
    const int nact = R.nact;
    const uint32_t* prow = planes + (int64_t)row * kD * 4 * wstride + 2 * blk;
    const uint16_t* srow = scales + (int64_t)row * kD * sstride + blk;
    float acc[64];
#pragma unroll
    for (int k = 0; k < 64; ++k) acc[k] = 0.0f;
    float cb = 0.0f;
    uint2 wb[kDrDepth];
    uint32_t sb[kDrDepth];
    float qpb[kDrDepth], qob[kDrDepth];
#pragma unroll
    for (int d = 0; d < kDrDepth; ++d) {
      if (d < nact) {
        const DrEnt E = R.e[d];
        wb[d] = ldg_u2(prow + E.poff);
        sb[d] = ldg_u16(srow + E.soff);
        qpb[d] = E.qp;
        qob[d] = E.qo;
      }
    }
    for (int e0p = 0; e0p < nact; e0p += kDrDepth) {
#pragma unroll
      for (int d = 0; d < kDrDepth; ++d) {
        const int e = e0p + d;
        if (e < nact) {  // uniform across the warp
          const float sf = __half2float(__ushort_as_half((unsigned short)sb[d]));
          cb = __fadd_rn(cb, __fmul_rn(qob[d], sf));
          const float wt = __fmul_rn(qpb[d], sf);
          const uint2 w = wb[d];
          const int en = e + kDrDepth;
          if (en < nact) {
            const DrEnt E = R.e[en];
            wb[d] = ldg_u2(prow + E.poff);
            sb[d] = ldg_u16(srow + E.soff);
            qpb[d] = E.qp;
            qob[d] = E.qo;
          }
          ps_bits(*reinterpret_cast<float(*)[32]>(&acc[0]), w.x, wt);
          ps_bits(*reinterpret_cast<float(*)[32]>(&acc[32]), w.y, wt);
        }
      }
    }
    if (!valid) continue;
    const int64_t tok0 = blk * 64;  // the lane's first token
#pragma unroll
    for (int k = 0; k < 64; ++k) acc[k] += cb;
    if (scores) {
      float* orow = scores + (int64_t)row * n + tok0;
      if (tok0 + 64 <= n && (n & 3) == 0) {
        float4* o4 = reinterpret_cast<float4*>(orow);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          o4[k] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
      } else {
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (tok0 + k < n) orow[k] = acc[k];
      }
    }
    if (wmax) {  // each 32-token word's maximum over its tokens < n (NaN if one is NaN)
#pragma unroll
      for (int k = 0; k < 64; ++k)
        if (tok0 + k >= n) acc[k] = -INFINITY;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float* a = acc + 32 * h;
#pragma unroll
        for (int w = 16; w > 0; w >>= 1)
#pragma unroll
          for (int i = 0; i < w; ++i) a[i] = fmax_nan(a[i], a[i + w]);
        const int64_t word = 2 * blk + h;
        if (word < nw_out) wmax[(int64_t)row * nw_out + word] = a[0];
      }
    }
  }
}

}  // namespace

// The direct-streaming scan: every layout with n_cap % 64 == 0 and any n >= 1;
// returns 1 (not launched) when the plane offsets would not fit 32 bits.
int launch_score_planes_direct(const Dims& s, const uint32_t* planes, const uint16_t* scales,
                               const uint8_t* plan, const uint16_t* q, float* scores,
                               const PsPlanIn* plan_in, float* wmax, int sms, cudaStream_t st) {
  const int64_t nbr = (s.n + 63) / 64;  // blocks per row
  const int64_t rows = (int64_t)s.B * s.Hkv;
  const int64_t total = nbr * rows;
  if ((int64_t)(4 * kD) * (s.ncap / 32) >= ((int64_t)1 << 32)) return 1;
  // at least one CTA per row's worth of blocks, so that a range meets at most two rows
  int64_t grid = imax64((int64_t)sms, (total + nbr - 1) / nbr);
  grid = imin64(grid, total);
  const PsPlanIn pl = plan_in ? *plan_in : PsPlanIn{};
  auto go = [&](auto kern) {
    kern<<<(unsigned)grid, kDrThreads, 0, st>>>(planes, scales, plan, q, s.Hq, s.Hkv, s.n, s.ncap,
                                                 nbr, total, scores, pl, wmax);
    note_launches(1);
    return check_launch("score_planes_direct");
  };
  switch (s.G) {
    case 1: return go(score_planes_direct_kernel<1>);
    case 2: return go(score_planes_direct_kernel<2>);
    case 4: return go(score_planes_direct_kernel<4>);
    default: return go(score_planes_direct_kernel<8>);
  }
}

}  // namespace sd
