// SCORE kernels: one cheap score per cached key (or 16-token block) of every
// (sequence, KV head).
//
//  * Hamming     -- HashAttention: Semantic Sparsity for Faster Inference, 2.2:
//                   SCORE = -popcount(h_i XOR h_q), summed over the GQA group.
//  * bit planes  -- Fathom: Per-Query Read Depth ..., "bit planes per channel" and
//                   "per-query reverse water-filling": only the planned planes
//                   of each channel are read.
//  * Quest bound -- OasisKV: Scaling In-Decode KV Cache Beyond HBM ...,
//                   prerequisites: block importance from per-channel min/max.
#include <cuda_fp16.h>

#include "sd_internal.cuh"
#include "sd_planes.cuh"

namespace sd {

// =====================================================================================
// Hamming scan: 4 B per token per KV head.  A thread takes 16 tokens as four 128-bit
// loads 1024 tokens apart, all issued before any is used, so every SM keeps enough
// bytes in flight to cover HBM latency; stores are 128-bit and coalesced alike.
// =====================================================================================
constexpr int kHmThreads = 256, kHmPer = 4;  // 128-bit loads per thread
constexpr int kHmTile = kHmThreads * 4 * kHmPer;  // tokens per CTA (4096)

template <int G>
__device__ __forceinline__ int4 hm_score4(uint4 s4, const uint32_t (&qs)[G]) {
  const uint32_t sv[4] = {s4.x, s4.y, s4.z, s4.w};
  int r[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    int acc = 0;
#pragma unroll
    for (int g = 0; g < G; ++g) acc += __popc(sv[k] ^ qs[g]);
    r[k] = -acc;
  }
  return make_int4(r[0], r[1], r[2], r[3]);
}

template <int G>
__global__ void __launch_bounds__(kHmThreads)
score_hamming_kernel(const uint32_t* __restrict__ sig, const uint32_t* __restrict__ qsig,
                     int Hq, int Hkv, int64_t n, int64_t ncap, bool vec,
                     int32_t* __restrict__ scores) {
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / Hkv), h = (int)(bh % Hkv);
  uint32_t qs[G];
#pragma unroll
  for (int g = 0; g < G; ++g) qs[g] = __ldg(qsig + (int64_t)b * Hq + h * G + g);
  const uint32_t* srow = sig + bh * ncap;
  int32_t* orow = scores + bh * n;
  const int64_t base = (int64_t)blockIdx.x * kHmTile + threadIdx.x * 4;
  if (vec && (int64_t)blockIdx.x * kHmTile + kHmTile <= n) {  // a whole tile
    uint4 s4[kHmPer];
#pragma unroll
    for (int j = 0; j < kHmPer; ++j)
      s4[j] = __ldg(reinterpret_cast<const uint4*>(srow + base + j * kHmThreads * 4));
#pragma unroll
    for (int j = 0; j < kHmPer; ++j)
      *reinterpret_cast<int4*>(orow + base + j * kHmThreads * 4) = hm_score4<G>(s4[j], qs);
    return;
  }
  for (int j = 0; j < kHmPer; ++j) {  // the row's last, partial tile
    const int64_t i0 = base + j * kHmThreads * 4;
    if (i0 >= n) break;
    if (vec && i0 + 4 <= n) {
      *reinterpret_cast<int4*>(orow + i0) =
          hm_score4<G>(__ldg(reinterpret_cast<const uint4*>(srow + i0)), qs);
    } else {
      for (int64_t i = i0; i < imin64(i0 + 4, n); ++i) {
        const uint32_t sv = __ldg(srow + i);
        int acc = 0;
#pragma unroll
        for (int g = 0; g < G; ++g) acc += __popc(sv ^ qs[g]);
        orow[i] = -acc;
      }
    }
  }
}

template <int G>
static void hamming_t(const Dims& s, const uint32_t* sig, const uint32_t* qsig, int32_t* out,
                      cudaStream_t st) {
  bool vec = (s.n % 4 == 0) && (s.ncap % 4 == 0);
  dim3 grid((unsigned)((s.n + kHmTile - 1) / kHmTile), (unsigned)(s.B * s.Hkv));
  score_hamming_kernel<G><<<grid, kHmThreads, 0, st>>>(sig, qsig, s.Hq, s.Hkv, s.n, s.ncap, vec,
                                                        out);
  note_launches(1);
}

int launch_score_hamming(const Dims& s, const uint32_t* sig, const uint32_t* qsig,
                         int32_t* scores, cudaStream_t st) {
  switch (s.G) {
    case 1: hamming_t<1>(s, sig, qsig, scores, st); break;
    case 2: hamming_t<2>(s, sig, qsig, scores, st); break;
    case 4: hamming_t<4>(s, sig, qsig, scores, st); break;
    default: hamming_t<8>(s, sig, qsig, scores, st); break;
  }
  return check_launch("score_hamming");
}

// =====================================================================================
// Bit-plane prefix scan.
//
// With q~_j = sum_g q_gj and W'_j = q~_j * s_j,blk, the score of token i is
//   sum_j W'_j * (prefix_ij + h(t_j) - 8)
//     = C_blk + sum over active planes (j, p < t_j) of (W'_j * 2^(3-p)) * bit_jpi,
//   C_blk = sum_j W'_j * (h(t_j) - 8),  h(t) = 2^(3-t) (t < 4), 0 (t = 4).
// So each planned plane costs one bit test and one predicated add per token --
// the in-HBM scan is bound by these operations, as the Fathom page notes.
//
// Work split.  The rows' tokens are cut into 512-token units and each CTA takes an
// equal contiguous range of units (every CTA has the same work to within one unit),
// walked as tiles of at most 8 units (4096 tokens: 128 words per plane, 64 scale
// blocks) that end at row ends.  A tile's active planes are consumed in chunks of
// up to 32.
//
// Warp roles (384 threads, 2 CTAs per SM).  Four helper warps stage each chunk's
// plane words with cp.async into a ring of three slots and write its folded
// weights (and, for a tile's first chunk, stage the tile's scales and form its
// per-block constants), then hand the slot over.  Eight compute warps only run the
// bit tests and adds: lane l of compute warp w owns word 32 (w mod 4) + l of the
// tile (32 tokens of one scale block), so per plane a warp reads 32 distinct words
// and 16 distinct weights and runs 32 bit tests and predicated adds on registers.
// Warps 0-3 take a chunk's even planes, warps 4-7 its odd ones; the two partial
// sums meet in shared memory at the tile's end.  Slots are handed over with named
// barriers: FULL[s] (helpers arrive, compute warps wait) and EMPTY[s] (compute warps
// arrive, helpers wait); a last FULL carries an end marker.
// =====================================================================================
constexpr int kPsTile = 4096;
constexpr int kPsUnit = 512;             // work split granularity (16-byte aligned copies)
constexpr int kPsWords = kPsTile / 32;   // 128
constexpr int kPsBlocks = kPsTile / 64;  // 64
constexpr int kPsChunk = 32;             // planes per slot
constexpr int kPsSlots = 3;
constexpr int kPsCompute = 256, kPsHelpers = 128;
constexpr int kPsThreads = kPsCompute + kPsHelpers;
constexpr int kPsCtasPerSm = 2;
// named barrier ids (0 is __syncthreads, which the kernel does not use)
constexpr int kBarFull = 1, kBarEmpty = kBarFull + kPsSlots, kBarHelp = kBarEmpty + kPsSlots,
              kBarComp = kBarHelp + 1;
constexpr int kSlotFirst = 1, kSlotLast = 2, kSlotEnd = 4;

struct PsSlot {
  int64_t tok0;  // the tile's first token
  int row;       // the tile's (sequence, KV head) row
  uint32_t thr;  // the row's candidate threshold key (fused scan + top-k)
  // planes in the chunk (bits 0-7; 0 for a tile with no active plane), the tile's
  // valid words (8-15), kSlotFirst / kSlotLast / kSlotEnd (16-19), the tile's
  // entry in the Cs ring (20-21)
  int info;
  __host__ __device__ int ne() const { return info & 255; }
  __host__ __device__ int nwv() const { return (info >> 8) & 255; }
  __host__ __device__ int flags() const { return (info >> 16) & 15; }
  __host__ __device__ int cs() const { return (info >> 20) & 3; }
};
__device__ __forceinline__ int slot_info(int ne, int nwv, int flags, int cs) {
  return ne | (nwv << 8) | (flags << 16) | (cs << 20);
}

struct PsSmem {
  uint32_t words[kPsSlots][kPsChunk][kPsWords];  // 48 KB
  float Wt[kPsSlots][kPsChunk][kPsBlocks];       // 24 KB
  float4 red[kPsWords * 8];                      // 16 KB: odd-plane partial sums
  uint16_t sc[kD][kPsBlocks];                    // 16 KB: active channels' scales by slot:
                                                 // two 64-slot halves (alternate tiles) or,
                                                 // past 64 active channels, one flat buffer
  float Cs[4][kPsBlocks];                        // per-block constants of 4 tiles in flight
  float hred[4][kPsBlocks];
  PsSlot slot[kPsSlots];
  PsRow row;                                     // the current row's tables
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }
__device__ __forceinline__ void nb_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void nb_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

// Compute warps: consume slots until the end marker; with CAND, also mark the
// row's candidates (see PsCand); with wmax, also write each 32-token word's
// maximum score (NaN if one of them is NaN) to wmax[row][word].
template <bool CAND>
__device__ __forceinline__ void ps_compute(PsSmem& S, float* __restrict__ scores, int64_t n,
                                           const PsCand& cd, float* __restrict__ wmax) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = warp >> 2, wl = (warp & 3) * 32 + lane;  // plane parity, word
  float4* red = &S.red[wl * 8];
  const int sw = lane & 7;
  float acc[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) acc[k] = 0.0f;
  for (int c = 0;; ++c) {
    const int s = c % kPsSlots;
    nb_sync(kBarFull + s, kPsThreads);
    const PsSlot m = S.slot[s];
    const int flags = m.flags(), nwv = m.nwv();
    if (flags & kSlotEnd) break;
    if (flags & kSlotFirst) {
#pragma unroll
      for (int k = 0; k < 32; ++k) acc[k] = 0.0f;
    }
    if ((warp & 3) * 32 < nwv) {  // warps whose words all lie past the end idle
      const uint32_t* wp = &S.words[s][half][wl];
      const float* tp = &S.Wt[s][half][wl >> 1];
#pragma unroll 2
      for (int e = half, ne = m.ne(); e < ne; e += 2, wp += 2 * kPsWords, tp += 2 * kPsBlocks)
        ps_bits(acc, *wp, *tp);
    }
    nb_arrive(kBarEmpty + s, kPsThreads);
    if (flags & kSlotLast) {
      // odd-plane partial sums: lane l's eight float4s go to 16-byte slots k ^ (l & 7),
      // so each quarter-warp hits 8 distinct bank groups.  (The next tile's writes to
      // red come after a FULL wait that every compute thread joins only once done
      // reading it here.)
      if (half == 1) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          red[k ^ sw] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
      }
      nb_sync(kBarComp, kPsCompute);
      if (half == 0) {
        const bool valid = wl < nwv;
        const float cb = S.Cs[m.cs()][wl >> 1];
        float4* orow = reinterpret_cast<float4*>(scores + (int64_t)m.row * n + m.tok0 + wl * 32);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float4 o = red[k ^ sw];
          acc[4 * k] = (acc[4 * k] + o.x) + cb;
          acc[4 * k + 1] = (acc[4 * k + 1] + o.y) + cb;
          acc[4 * k + 2] = (acc[4 * k + 2] + o.z) + cb;
          acc[4 * k + 3] = (acc[4 * k + 3] + o.w) + cb;
          if (valid) orow[k] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
        }
        if (CAND) {
          ps_mark(cd, m.row, m.thr, m.tok0 + wl * 32, valid, acc);
        } else if (wmax) {  // a tree of depth 5 in place: acc is reset by the next tile
#pragma unroll
          for (int w = 16; w > 0; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) acc[i] = fmax_nan(acc[i], acc[i + w]);
          if (valid) wmax[(int64_t)m.row * (n >> 5) + (m.tok0 >> 5) + wl] = acc[0];
        }
      }
    }
  }
}

// Helper-side record of a chunk whose copies are in flight.
struct PsPending {
  PsSlot m;
  int e0;  // first entry of the chunk
  int sb;  // scale buffer: 0 / 1 (halves) or 2 (flat)
};

__device__ __forceinline__ const uint16_t* ps_scales(const PsSmem& S, int sb) {
  return sb == 1 ? &S.sc[kD / 2][0] : &S.sc[0][0];
}

// Finishes the oldest pending chunk (slot d % kPsSlots): waits for its copies (the
// `newer` chunks issued after it may stay in flight), forms the tile's per-block
// constants if it is the tile's first chunk, writes its folded weights and hands
// the slot to the compute warps.
__device__ __forceinline__ void ps_finish(PsSmem& S, const PsPending& pd, int d, int newer) {
  const int ht = threadIdx.x - kPsCompute, hw = ht >> 5, lane = threadIdx.x & 31;
  if (newer > 0)
    asm volatile("cp.async.wait_group 1;\n" ::: "memory");
  else
    cp_async_wait_all();
  nb_sync(kBarHelp, kPsHelpers);  // every helper's copies of the chunk have landed
  const int s = d % kPsSlots;
  const uint16_t* scb = ps_scales(S, pd.sb);
  const int nbv = pd.m.nwv() / 2;
  // blocks b4..b4+3 (a group that reaches past nbv holds blocks past the end: their
  // values are read only by lanes whose sums are not stored)
  const int b4 = (lane & 15) * 4;
  if (pd.m.flags() & kSlotFirst) {
    // per-block constants C_blk: half-warps take alternate slots, a shuffle joins
    // the halves, then the four warps' partial sums are added
    float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (b4 < nbv) {
      for (int sl = 2 * hw + (lane >> 4); sl < S.row.nch; sl += 2 * (kPsHelpers / 32)) {
        const uint2 raw = *reinterpret_cast<const uint2*>(scb + sl * kPsBlocks + b4);
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        const float qo = S.row.qo[sl];
        a.x = __fadd_rn(a.x, __fmul_rn(qo, f0.x));
        a.y = __fadd_rn(a.y, __fmul_rn(qo, f0.y));
        a.z = __fadd_rn(a.z, __fmul_rn(qo, f1.x));
        a.w = __fadd_rn(a.w, __fmul_rn(qo, f1.y));
      }
    }
    a.x = __fadd_rn(a.x, __shfl_xor_sync(0xFFFFFFFFu, a.x, 16));
    a.y = __fadd_rn(a.y, __shfl_xor_sync(0xFFFFFFFFu, a.y, 16));
    a.z = __fadd_rn(a.z, __shfl_xor_sync(0xFFFFFFFFu, a.z, 16));
    a.w = __fadd_rn(a.w, __shfl_xor_sync(0xFFFFFFFFu, a.w, 16));
    if (lane < 16) *reinterpret_cast<float4*>(&S.hred[hw][b4]) = a;
    nb_sync(kBarHelp, kPsHelpers);
    if (ht < kPsBlocks)
      S.Cs[pd.m.cs()][ht] = __fadd_rn(__fadd_rn(S.hred[0][ht], S.hred[1][ht]),
                                    __fadd_rn(S.hred[2][ht], S.hred[3][ht]));
  }
  // folded weights Wt = (q~_j * 2^(3-p)) * s_j,blk, which equals
  // fl(q~_j * s_j,blk) * 2^(3-p) exactly (power-of-two scaling commutes with rounding);
  // half-warps take alternate planes, each lane four blocks
  if (b4 < nbv) {
#pragma unroll 2
    for (int e = 2 * hw + (lane >> 4), ne = pd.m.ne(); e < ne; e += 2 * (kPsHelpers / 32)) {
      const float qv = S.row.qp[pd.e0 + e];
      const uint2 raw = *reinterpret_cast<const uint2*>(scb + S.row.eslot[pd.e0 + e] * kPsBlocks + b4);
      const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
      const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
      *reinterpret_cast<float4*>(&S.Wt[s][e][b4]) =
          make_float4(__fmul_rn(qv, f0.x), __fmul_rn(qv, f0.y), __fmul_rn(qv, f1.x),
                      __fmul_rn(qv, f1.y));
    }
  }
  if (ht == 0) S.slot[s] = pd.m;
  nb_arrive(kBarFull + s, kPsThreads);
}

// Helper warps: walk the CTA's tiles and keep up to two chunks' copies in flight:
// chunk c is issued once the compute warps release its slot, right after chunk
// c - 2 is finished and handed over.  The pipeline drains before a row change
// (the row tables are rebuilt) and, past 64 active channels, before each tile
// (one flat scale buffer); then the end marker is posted.
template <int G, bool A16, bool CAND>
__device__ __forceinline__ void ps_help(PsSmem& S, const uint32_t* __restrict__ planes,
                                        const uint16_t* __restrict__ scales,
                                        const uint8_t* __restrict__ plan,
                                        const uint16_t* __restrict__ q, int Hq, int Hkv, int64_t n,
                                        int64_t ncap, int upr, int64_t total_units,
                                        const PsCand& cd, const PsPlanIn& pl) {
  const int ht = threadIdx.x - kPsCompute, hw = ht >> 5, lane = threadIdx.x & 31;
  const uint32_t wstride = (uint32_t)(ncap / 32), sstride = (uint32_t)(ncap / 64);
  // this CTA's units, walked as (row bh, unit ur) without dividing; rows <= 65535
  // and a CTA holds fewer than 2^30 units, so 32-bit counters suffice
  const int64_t u_begin = (int64_t)blockIdx.x * total_units / gridDim.x;
  const int64_t u_end = (int64_t)(blockIdx.x + 1) * total_units / gridDim.x;
  int left = (int)(u_end - u_begin);
  int bh = (int)(u_begin / upr);
  int ur = (int)(u_begin - (int64_t)bh * upr);
  int cur_bh = -1;
  uint32_t row_thr = 0;
  int c = 0, d = 0;  // chunks issued, chunks handed over
  PsPending p0, p1;  // pending chunks, oldest first (registers: indexed statically)
  int np = 0;
  const int n32 = (int)(n / 32);  // words per row (n < 2^31)
  for (int tcount = 0; left > 0; ++tcount) {
    const int nu = min(min(kPsTile / kPsUnit, upr - ur), left);
    const int64_t tok0 = (int64_t)ur * kPsUnit;
    const int nwv = min(nu * (kPsUnit / 32), n32 - ur * (kPsUnit / 32));  // valid words (even)
    const int nbv = nwv / 2;                                             // valid scale blocks
    if (bh != cur_bh) {  // per-row tables: drain, then rebuild
      for (; np > 0; --np, ++d) {
        ps_finish(S, p0, d, np - 1);
        p0 = p1;
      }
      nb_sync(kBarHelp, kPsHelpers);  // every helper is done with the old tables
      cur_bh = bh;
      // (the CTA whose range holds the row's first unit writes a computed plan)
      ps_build_row<G>(S.row, ht, q, plan, bh / Hkv, bh % Hkv, Hq, (int64_t)bh,
                      [] { nb_sync(kBarHelp, kPsHelpers); }, pl, ur == 0);
      if (CAND) row_thr = __ldg(cd.thr + bh);
    }
    const int nact = S.row.nact, nch = S.row.nch;
    const int nck = max(1, (nact + kPsChunk - 1) / kPsChunk);
    const int sb = nch <= kD / 2 ? (tcount & 1) : 2;
    if (sb == 2) {  // one flat scale buffer: drain first
      for (; np > 0; --np, ++d) {
        ps_finish(S, p0, d, np - 1);
        p0 = p1;
      }
    }
    uint16_t* scb = const_cast<uint16_t*>(ps_scales(S, sb));
    const uint32_t* pl_tile = planes + (int64_t)bh * kD * 4 * wstride + tok0 / 32;
    const uint16_t* sc_tile = scales + (int64_t)bh * kD * sstride + tok0 / 64;
    for (int k = 0; k < nck; ++k, ++c) {
      if (np == 2) {  // hand over chunk c - 2 before waiting for a slot
        ps_finish(S, p0, d, 1);
        p0 = p1;
        --np;
        ++d;
      }
      const int s = c % kPsSlots;
      if (c >= kPsSlots) nb_sync(kBarEmpty + s, kPsThreads);  // compute is done with slot s
      const int e0 = k * kPsChunk, ne = max(0, min(kPsChunk, nact - e0));
      if (k == 0) {  // the tile's active-channel scales
        nb_sync(kBarHelp, kPsHelpers);  // every helper is done reading this scale buffer
        if (A16) {
          // whole 16-byte segments (8 blocks) inside the valid blocks, the rest singly
          for (int x = ht; x < nch * 8; x += kPsHelpers) {
            const int sl = x >> 3, sg = x & 7;
            const uint16_t* src = sc_tile + (uint64_t)S.row.chan[sl] * sstride + sg * 8;
            uint16_t* dst = scb + sl * kPsBlocks + sg * 8;
            if (sg * 8 + 8 <= nbv) {
              cp_async16(smem_u32(dst), src);
            } else {
              for (int i = 0; sg * 8 + i < nbv; ++i) dst[i] = src[i];
            }
          }
        } else {
          for (int x = ht; x < nch * kPsBlocks; x += kPsHelpers) {
            const int sl = x / kPsBlocks, blk = x % kPsBlocks;
            if (blk < nbv) scb[sl * kPsBlocks + blk] = sc_tile[(uint64_t)S.row.chan[sl] * sstride + blk];
          }
        }
      }
      // the chunk's plane words: one warp per plane row
      const uint32_t wdst = smem_u32(&S.words[s][0][0]);
      if (A16) {
        // whole 16-byte segments inside the valid words, then an 8-byte remainder
        // (nwv is even): no copy reads past the last valid word of a plane row
        const int seg = lane * 4 + 4 <= nwv ? 16 : (lane * 4 + 2 == nwv ? 8 : 0);
        if (seg) {
          for (int e = hw; e < ne; e += kPsHelpers / 32) {
            const uint32_t* src = pl_tile + (uint64_t)S.row.act[e0 + e] * wstride + lane * 4;
            const uint32_t dd = wdst + e * (kPsWords * 4) + lane * 16;
            if (seg == 16) cp_async16(dd, src);
            else cp_async8(dd, src);
          }
        }
      } else {
        for (int e = hw; e < ne; e += kPsHelpers / 32) {
          const uint32_t* src = pl_tile + (uint64_t)S.row.act[e0 + e] * wstride;
          for (int sg = lane; sg * 2 < nwv; sg += 32)
            cp_async8(wdst + e * (kPsWords * 4) + sg * 8, src + sg * 2);
        }
      }
      cp_async_commit();
      PsPending pd;
      pd.m.info = slot_info(ne, nwv, (k == 0 ? kSlotFirst : 0) | (k == nck - 1 ? kSlotLast : 0),
                            tcount & 3);
      pd.m.tok0 = tok0;
      pd.m.row = bh;
      pd.m.thr = row_thr;
      pd.e0 = e0;
      pd.sb = sb;
      if (np == 0) p0 = pd;
      else p1 = pd;
      ++np;
    }
    // the next tile of the range
    left -= nu;
    ur += nu;
    if (ur == upr) { ur = 0; ++bh; }
  }
  for (; np > 0; --np, ++d) {
    ps_finish(S, p0, d, np - 1);
    p0 = p1;
  }
  // end marker, then wait out the compute warps' releases of the last slots
  {
    const int s = c % kPsSlots;
    if (c >= kPsSlots) nb_sync(kBarEmpty + s, kPsThreads);
    if (ht == 0) S.slot[s].info = slot_info(0, 0, kSlotEnd, 0);
    nb_arrive(kBarFull + s, kPsThreads);
  }
  for (int x = max(0, c - kPsSlots + 1); x < c; ++x) nb_sync(kBarEmpty + x % kPsSlots, kPsThreads);
}

template <int G, bool A16, bool CAND>
__global__ void __launch_bounds__(kPsThreads, kPsCtasPerSm)
score_planes_kernel(const uint32_t* __restrict__ planes, const uint16_t* __restrict__ scales,
                    const uint8_t* __restrict__ plan, const uint16_t* __restrict__ q, int Hq,
                    int Hkv, int64_t n, int64_t ncap, int upr, int64_t total_units,
                    float* __restrict__ scores, PsCand cd, PsPlanIn pl,
                    float* __restrict__ wmax) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  PsSmem& S = *reinterpret_cast<PsSmem*>(smem_raw);
  if (threadIdx.x < kPsCompute)
    ps_compute<CAND>(S, scores, n, cd, wmax);
  else
    ps_help<G, A16, CAND>(S, planes, scales, plan, q, Hq, Hkv, n, ncap, upr, total_units, cd, pl);
}

static int sm_count() {
  static int cnt[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (!cnt[dev]) {
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0)
      c = 152;
    cnt[dev] = c;
  }
  return cnt[dev];
}

template <int G, bool A16, bool CAND>
static int planes_t(const Dims& s, const uint32_t* planes, const uint16_t* scales,
                    const uint8_t* plan, const uint16_t* q, float* scores, const PsCand& cd,
                    const PsPlanIn& pl, float* wmax, cudaStream_t st) {
  auto kern = score_planes_kernel<G, A16, CAND>;
  if (int rc = set_smem_limit((const void*)kern, sizeof(PsSmem), "score_planes: smem attribute"))
    return rc;
  const int upr = (int)((s.n + kPsUnit - 1) / kPsUnit);  // units per row (n < 2^31)
  const int64_t total = (int64_t)upr * s.B * s.Hkv;
  const int64_t grid = imin64(total, (int64_t)sm_count() * kPsCtasPerSm);
  kern<<<(unsigned)grid, kPsThreads, sizeof(PsSmem), st>>>(planes, scales, plan, q, s.Hq, s.Hkv,
                                                          s.n, s.ncap, upr, total, scores, cd, pl,
                                                          wmax);
  note_launches(1);
  return check_launch("score_planes");
}

bool planes_aligned(const Dims& s, const void* planes, const void* scales) {
  return (s.ncap % 512 == 0) && ((uintptr_t)planes % 16 == 0) && ((uintptr_t)scales % 16 == 0);
}

int launch_score_planes(const Dims& s, const uint32_t* planes, const uint16_t* scales,
                        const uint8_t* plan, const uint16_t* q, float* scores, cudaStream_t st,
                        const PsCand* cand, const PsPlanIn* plan_in, float* wmax) {
  const bool a16 = planes_aligned(s, planes, scales) && !fallback_forced();
  const PsPlanIn pl = plan_in ? *plan_in : PsPlanIn{};
  if (a16) {  // the bulk-copy kernel (any n), when every CTA's range meets at most two rows
    const int rc = launch_score_planes_tma(s, planes, scales, plan, q, scores, cand, plan_in,
                                           wmax, sm_count(), st);
    if (rc != 1) return rc;
  }
  if (s.n % 64) {  // a partial last block outside the bulk-copy kernel: the direct kernel
    if (cand) return fail(SD_ERR_UNSUPPORTED, "score_planes: candidates need n %% 64 == 0");
    const int rc = launch_score_planes_direct(s, planes, scales, plan, q, scores, plan_in, wmax,
                                              sm_count(), st);
    if (rc != 1) return rc;
    return fail(SD_ERR_UNSUPPORTED, "score_planes: n_cap too large for n %% 64 != 0");
  }
  if (cand) {  // the fused scan + top-k path (16-byte aligned layouts only)
    if (!a16) return fail(SD_ERR_INVALID_ARG, "score_planes: candidates need n_cap %% 512 == 0 "
                                              "and 16-byte aligned planes and scales");
    switch (s.G) {
      case 1: return planes_t<1, true, true>(s, planes, scales, plan, q, scores, *cand, pl, nullptr, st);
      case 2: return planes_t<2, true, true>(s, planes, scales, plan, q, scores, *cand, pl, nullptr, st);
      case 4: return planes_t<4, true, true>(s, planes, scales, plan, q, scores, *cand, pl, nullptr, st);
      default: return planes_t<8, true, true>(s, planes, scales, plan, q, scores, *cand, pl, nullptr, st);
    }
  }
  const PsCand none{};
  switch (s.G) {
    case 1: return a16 ? planes_t<1, true, false>(s, planes, scales, plan, q, scores, none, pl, wmax, st) : planes_t<1, false, false>(s, planes, scales, plan, q, scores, none, pl, wmax, st);
    case 2: return a16 ? planes_t<2, true, false>(s, planes, scales, plan, q, scores, none, pl, wmax, st) : planes_t<2, false, false>(s, planes, scales, plan, q, scores, none, pl, wmax, st);
    case 4: return a16 ? planes_t<4, true, false>(s, planes, scales, plan, q, scores, none, pl, wmax, st) : planes_t<4, false, false>(s, planes, scales, plan, q, scores, none, pl, wmax, st);
    default: return a16 ? planes_t<8, true, false>(s, planes, scales, plan, q, scores, none, pl, wmax, st) : planes_t<8, false, false>(s, planes, scales, plan, q, scores, none, pl, wmax, st);
  }
}

// =====================================================================================
// Quest block bound.  max(q*mn, q*mx) = q*mx if q >= 0 else q*mn (mn <= mx), so
//   U = sum_j (P_j * max_j + N_j * min_j),  P_j = sum_g max(q_gj, 0),
//                                           N_j = sum_g min(q_gj, 0):
// two FMAs per channel per block instead of 4G operations.  A warp scores 4 blocks
// (512 B each), lane l owning channels 4l..4l+3; a CTA scores 32 blocks.
// =====================================================================================
template <int G>
__global__ void __launch_bounds__(256)
score_quest_kernel(const uint16_t* __restrict__ summ, const uint16_t* __restrict__ q, int Hq,
                   int Hkv, int64_t n, int64_t ncap, float* __restrict__ scores) {
  __shared__ float Ps[kD], Ns[kD];
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / Hkv), h = (int)(bh % Hkv);
  if (threadIdx.x < kD) {
    float p = 0.0f, m = 0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float x = bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + threadIdx.x]);
      p = __fadd_rn(p, fmaxf(x, 0.0f));
      m = __fadd_rn(m, fminf(x, 0.0f));
    }
    Ps[threadIdx.x] = p;
    Ns[threadIdx.x] = m;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nblk = (n + 15) / 16, nblk_cap = (ncap + 15) / 16;
  float P[4], N[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) { P[k] = Ps[lane * 4 + k]; N[k] = Ns[lane * 4 + k]; }
  const int64_t c0 = (int64_t)blockIdx.x * 32 + warp * 4;
  float acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    acc[k] = 0.0f;
    const int64_t c = c0 + k;
    if (c < nblk) {
      const uint16_t* base = summ + (bh * nblk_cap + c) * 2 * kD + lane * 4;
      uint2 lo = __ldg(reinterpret_cast<const uint2*>(base));
      uint2 hi = __ldg(reinterpret_cast<const uint2*>(base + kD));
      float a = 0.0f;
      a = __fmaf_rn(P[0], bf16_lo(hi.x), a);
      a = __fmaf_rn(N[0], bf16_lo(lo.x), a);
      a = __fmaf_rn(P[1], bf16_hi(hi.x), a);
      a = __fmaf_rn(N[1], bf16_hi(lo.x), a);
      a = __fmaf_rn(P[2], bf16_lo(hi.y), a);
      a = __fmaf_rn(N[2], bf16_lo(lo.y), a);
      a = __fmaf_rn(P[3], bf16_hi(hi.y), a);
      a = __fmaf_rn(N[3], bf16_hi(lo.y), a);
      acc[k] = a;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] += __shfl_xor_sync(0xFFFFFFFFu, acc[k], o);
  if (lane < 4 && c0 + lane < nblk) {
    float r = lane == 0 ? acc[0] : lane == 1 ? acc[1] : lane == 2 ? acc[2] : acc[3];
    scores[bh * nblk + c0 + lane] = r;
  }
}

int launch_score_quest(const Dims& s, const uint16_t* summ, const uint16_t* q, float* scores,
                       cudaStream_t st) {
  int64_t nblk = (s.n + 15) / 16;
  dim3 grid((unsigned)((nblk + 31) / 32), (unsigned)(s.B * s.Hkv));
  switch (s.G) {
    case 1: score_quest_kernel<1><<<grid, 256, 0, st>>>(summ, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
    case 2: score_quest_kernel<2><<<grid, 256, 0, st>>>(summ, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
    case 4: score_quest_kernel<4><<<grid, 256, 0, st>>>(summ, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
    default: score_quest_kernel<8><<<grid, 256, 0, st>>>(summ, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
  }
  note_launches(1);
  return check_launch("score_quest");
}

// =====================================================================================
// Block landmark scan: U = sum_j q~_j L_j, q~ the group-summed query (fp32, g
// ascending).  A warp scores 4 blocks (256 B each), lane l owning channels 4l..4l+3;
// a CTA scores 32 blocks.
// =====================================================================================
template <int G>
__global__ void __launch_bounds__(256)
score_landmark_kernel(const uint16_t* __restrict__ L, const uint16_t* __restrict__ q, int Hq,
                      int Hkv, int64_t n, int64_t ncap, float* __restrict__ scores) {
  __shared__ float Qs[kD];
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / Hkv), h = (int)(bh % Hkv);
  if (threadIdx.x < kD) {
    float a = 0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g)
      a = __fadd_rn(a, bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + threadIdx.x]));
    Qs[threadIdx.x] = a;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nblk = (n + kLmBlock - 1) / kLmBlock, nblk_cap = (ncap + kLmBlock - 1) / kLmBlock;
  float Q[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) Q[k] = Qs[lane * 4 + k];
  const int64_t c0 = (int64_t)blockIdx.x * 32 + warp * 4;
  float acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    acc[k] = 0.0f;
    const int64_t c = c0 + k;
    if (c < nblk) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(L + (bh * nblk_cap + c) * kD + lane * 4));
      float a = 0.0f;
      a = __fmaf_rn(Q[0], bf16_lo(v.x), a);
      a = __fmaf_rn(Q[1], bf16_hi(v.x), a);
      a = __fmaf_rn(Q[2], bf16_lo(v.y), a);
      a = __fmaf_rn(Q[3], bf16_hi(v.y), a);
      acc[k] = a;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] += __shfl_xor_sync(0xFFFFFFFFu, acc[k], o);
  if (lane < 4 && c0 + lane < nblk) {
    float r = lane == 0 ? acc[0] : lane == 1 ? acc[1] : lane == 2 ? acc[2] : acc[3];
    scores[bh * nblk + c0 + lane] = r;
  }
}

int launch_score_landmark(const Dims& s, const uint16_t* L, const uint16_t* q, float* scores,
                          cudaStream_t st) {
  const int64_t nblk = (s.n + kLmBlock - 1) / kLmBlock;
  dim3 grid((unsigned)((nblk + 31) / 32), (unsigned)(s.B * s.Hkv));
  switch (s.G) {
    case 1: score_landmark_kernel<1><<<grid, 256, 0, st>>>(L, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
    case 2: score_landmark_kernel<2><<<grid, 256, 0, st>>>(L, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
    case 4: score_landmark_kernel<4><<<grid, 256, 0, st>>>(L, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
    default: score_landmark_kernel<8><<<grid, 256, 0, st>>>(L, q, s.Hq, s.Hkv, s.n, s.ncap, scores); break;
  }
  note_launches(1);
  return check_launch("score_landmark");
}

}  // namespace sd
