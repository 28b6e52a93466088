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

namespace sd {

// =====================================================================================
// Hamming scan: 4 B per token per KV head, four tokens per thread (128-bit loads).
// =====================================================================================
template <int G>
__global__ void __launch_bounds__(256)
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
  const int64_t i0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i0 >= n) return;
  if (vec && i0 + 4 <= n) {
    uint4 s4 = __ldg(reinterpret_cast<const uint4*>(srow + i0));
    uint32_t sv[4] = {s4.x, s4.y, s4.z, s4.w};
    int r[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      int acc = 0;
#pragma unroll
      for (int g = 0; g < G; ++g) acc += __popc(sv[k] ^ qs[g]);
      r[k] = -acc;
    }
    *reinterpret_cast<int4*>(orow + i0) = make_int4(r[0], r[1], r[2], r[3]);
  } else {
    for (int64_t i = i0; i < imin64(i0 + 4, n); ++i) {
      uint32_t sv = __ldg(srow + i);
      int acc = 0;
#pragma unroll
      for (int g = 0; g < G; ++g) acc += __popc(sv ^ qs[g]);
      orow[i] = -acc;
    }
  }
}

template <int G>
static void hamming_t(const Dims& s, const uint32_t* sig, const uint32_t* qsig, int32_t* out,
                      cudaStream_t st) {
  bool vec = (s.n % 4 == 0) && (s.ncap % 4 == 0);
  dim3 grid((unsigned)((s.n + 1023) / 1024), (unsigned)(s.B * s.Hkv));
  score_hamming_kernel<G><<<grid, 256, 0, st>>>(sig, qsig, s.Hq, s.Hkv, s.n, s.ncap, vec, out);
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
// A CTA scores tiles of up to 4096 tokens (128 words per plane, 64 scale blocks) of
// one (sequence, KV head); the grid is persistent (3 CTAs per SM).  The rows' tokens
// are cut into 512-token units and each CTA takes an equal contiguous range of
// units (so every CTA has the same work to within one unit), walked as tiles of at
// most 8 units that end at row ends; the per-row prologue (group-summed query,
// active plane list) is paid once per row change.  Per tile: the active channels' scales
// are staged once; planes are staged 32 at a time with cp.async into a double
// buffer while the previous 32 are consumed; folded weights are built per stage.
// Each lane owns one word (32 tokens, one scale block) of the tile: lane l of warp
// w holds word 32 (w mod 4) + l, so per plane a warp reads 32 distinct words and
// 16 distinct weights (one shared-memory wavefront each) and then runs 32 bit
// tests and predicated adds on registers.  Warps 0-3 take the even planes of each
// stage, warps 4-7 the odd ones; the two partial sums meet in shared memory once
// per tile.
// =====================================================================================
constexpr int kPsTile = 4096;
constexpr int kPsUnit = 512;             // work split granularity (16-byte aligned copies)
constexpr int kPsWords = kPsTile / 32;   // 128
constexpr int kPsBlocks = kPsTile / 64;  // 64
constexpr int kPsChunk = 32;             // planes per stage
constexpr int kPsThreads = 256;
constexpr int kPsCtasPerSm = 3;

struct PsSmem {
  uint32_t words[2][kPsChunk][kPsWords];  // 32 KB
  float Wt[2][kPsChunk][kPsBlocks];       // 16 KB
  uint16_t sc[2][kD / 2][kPsBlocks];      // 16 KB: active channels' scales by slot: two
                                          // 64-slot halves (current / prefetched tile),
                                          // or one flat 128-slot buffer
  float red[8][kPsBlocks];
  float Cs[kPsBlocks];
  float qt[kD];
  float qo[kD];                           // q~_j * (h(t_j) - 8) per slot
  int tb[kD];
  int slot_of[kD];
  int chan[kD];                           // channel of each slot
  uint16_t act[4 * kD];                   // active entries j * 4 + p, j ascending
  uint8_t eslot[4 * kD];                  // slot of each entry's channel
  float qp[4 * kD];                       // q~_j * 2^(3-p) per entry (exact scaling)
  int nact, nch;
};

// The tile starting at unit u of a CTA's range [.., u_end): its row, first token
// and unit count.
struct PsTile {
  int64_t bh, tok0;
  int nu;
};
__device__ __forceinline__ PsTile ps_tile_at(int64_t u, int64_t u_end, int64_t upr) {
  PsTile t;
  t.bh = u / upr;
  const int64_t ur = u - t.bh * upr;
  t.tok0 = ur * kPsUnit;
  t.nu = (int)imin64(imin64(kPsTile / kPsUnit, upr - ur), u_end - u);
  return t;
}
// valid words of a tile (even: n is a multiple of 64)
__device__ __forceinline__ int ps_valid_words(const PsTile& t, int64_t n) {
  return (int)imin64(t.nu * (kPsUnit / 32), (n - t.tok0) / 32);
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  unsigned d = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem));
}
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
  unsigned d = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(d), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// Issues the copies of planes [e0, e0 + ne) of the tile into words[buf].
template <bool A16>
__device__ __forceinline__ void ps_stage_words(PsSmem& S, int buf, int e0, int ne,
                                               const uint32_t* pl_tile, int64_t wstride,
                                               int nwv) {
  // one warp per plane row
  const int lane = threadIdx.x & 31;
  for (int e = threadIdx.x >> 5; e < ne; e += kPsThreads / 32) {
    const uint32_t* src = pl_tile + (int64_t)S.act[e0 + e] * wstride;
    uint32_t* dst = &S.words[buf][e][0];
    if (A16) {
      // whole 16-byte segments inside the valid words, then an 8-byte remainder
      // (nwv is even): no copy reads past the last valid word of a plane row
      if (lane * 4 + 4 <= nwv)
        cp_async16(dst + lane * 4, src + lane * 4);
      else if (lane * 4 + 2 == nwv)
        cp_async8(dst + lane * 4, src + lane * 4);
    } else {
      for (int sg = lane; sg * 2 < nwv; sg += 32) cp_async8(dst + sg * 2, src + sg * 2);
    }
  }
  cp_async_commit();
}

// Folded weights of planes [e0, e0 + ne): Wt = (q~_j * 2^(3-p)) * s_j,blk, which
// equals fl(q~_j * s_j,blk) * 2^(3-p) exactly (power-of-two scaling commutes with
// rounding).
// Only valid blocks are written: the other weights are read only by lanes whose
// words lie past the tile's end, whose sums are never stored.
__device__ __forceinline__ void ps_weights(PsSmem& S, const uint16_t* scb, int buf, int e0, int ne,
                                           int nbv) {
  // blocks b2, b2 + 1; for odd nbv the last pair's second weight is not valid (and
  // is read only by lanes past the end)
  const int b2 = (threadIdx.x & 31) * 2;
  if (b2 >= nbv) return;
  for (int e = threadIdx.x >> 5; e < ne; e += kPsThreads / 32) {
    const float qp = S.qp[e0 + e];
    const __half2 sv = *reinterpret_cast<const __half2*>(&scb[S.eslot[e0 + e] * kPsBlocks + b2]);
    const float2 f = __half22float2(sv);
    *reinterpret_cast<float2*>(&S.Wt[buf][e][b2]) = make_float2(__fmul_rn(qp, f.x), __fmul_rn(qp, f.y));
  }
}

// Issues the copies of a tile's active-channel scales into scb (one group with
// the tile's first chunk of planes, which the caller stages).
template <bool A16>
__device__ __forceinline__ void ps_stage_scales(PsSmem& S, uint16_t* scb, const uint16_t* sc_tile,
                                                int64_t sstride, int nch, int nbv) {
  if (A16) {
    // whole 16-byte segments (8 blocks) inside the valid blocks, the rest singly
    for (int x = threadIdx.x; x < nch * 8; x += kPsThreads) {
      const int sl = x >> 3, seg = x & 7;
      const uint16_t* src = sc_tile + (int64_t)S.chan[sl] * sstride + seg * 8;
      uint16_t* dst = scb + sl * kPsBlocks + seg * 8;
      if (seg * 8 + 8 <= nbv) {
        cp_async16(dst, src);
      } else {
        for (int k = 0; seg * 8 + k < nbv; ++k) dst[k] = src[k];
      }
    }
  } else {
    for (int x = threadIdx.x; x < nch * kPsBlocks; x += kPsThreads) {
      const int sl = x / kPsBlocks, blk = x % kPsBlocks;
      if (blk < nbv) scb[sl * kPsBlocks + blk] = sc_tile[(int64_t)S.chan[sl] * sstride + blk];
    }
  }
}

template <int G, bool A16>
__global__ void __launch_bounds__(kPsThreads, kPsCtasPerSm)
score_planes_kernel(const uint32_t* __restrict__ planes, const uint16_t* __restrict__ scales,
                    const uint8_t* __restrict__ plan, const uint16_t* __restrict__ q, int Hq,
                    int Hkv, int64_t n, int64_t ncap, int64_t units_per_row, int64_t total_units,
                    float* __restrict__ scores) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  PsSmem& S = *reinterpret_cast<PsSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t wstride = ncap / 32, sstride = ncap / 64;
  const int64_t u_begin = (int64_t)blockIdx.x * total_units / gridDim.x;
  const int64_t u_end = (int64_t)(blockIdx.x + 1) * total_units / gridDim.x;
  int64_t cur_bh = -1;
  bool staged = false;  // this tile's scales and first chunk are already in flight
  int sbuf = 0;         // scale half of this tile (double-buffered mode)
  int wb0 = 0;          // words buffer holding this tile's first chunk

  for (int64_t u = u_begin; u < u_end;) {
    const PsTile T = ps_tile_at(u, u_end, units_per_row);
    const int64_t bh = T.bh, tok0 = T.tok0, u_next = u + T.nu;
    if (bh != cur_bh) {  // per-row prologue
      cur_bh = bh;
      staged = false;
      const int b = (int)(bh / Hkv), h = (int)(bh % Hkv);
      if (threadIdx.x < kD) {
        const int j = threadIdx.x;
        float acc = 0.0f;
#pragma unroll
        for (int g = 0; g < G; ++g)
          acc = __fadd_rn(acc, bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + j]));
        S.qt[j] = acc;
        S.tb[j] = min((int)plan[bh * kD + j], 4);  // a plan holds 0..4 bits per channel
      }
      __syncthreads();
      if (warp == 0) {  // active entries and channel slots, j ascending
        int c[4], tot = 0, chs = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          c[k] = S.tb[lane * 4 + k];
          tot += c[k];
          chs += c[k] > 0;
        }
        int incl = tot, inclc = chs;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
          const int yc = __shfl_up_sync(0xFFFFFFFFu, inclc, off);
          if (lane >= off) { incl += y; inclc += yc; }
        }
        int pos = incl - tot, slot = inclc - chs;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = lane * 4 + k;
          for (int p = 0; p < c[k]; ++p) S.act[pos++] = (uint16_t)(j * 4 + p);
          if (c[k] > 0) {
            S.slot_of[j] = slot;
            S.chan[slot] = j;
            S.qo[slot] = __fmul_rn(S.qt[j], c[k] < 4 ? (float)((1 << (3 - c[k])) - 8) : -8.0f);
            ++slot;
          } else {
            S.slot_of[j] = 0;
          }
        }
        if (lane == 31) { S.nact = incl; S.nch = inclc; }
      }
      __syncthreads();
      for (int e = threadIdx.x; e < S.nact; e += kPsThreads) {
        const int ent = S.act[e], j = ent >> 2, p = ent & 3;
        S.eslot[e] = (uint8_t)S.slot_of[j];
        S.qp[e] = ldexpf(S.qt[j], 3 - p);
      }
      __syncthreads();
    }
    const int nact = S.nact, nch = S.nch;
    const bool dbl = nch <= kD / 2;  // scales fit one half: prefetch the next tile
    uint16_t* scb = dbl ? &S.sc[sbuf][0][0] : &S.sc[0][0][0];
    const int nwv = ps_valid_words(T, n);  // valid words (even)
    const int nbv = nwv / 2;               // valid scale blocks
    const uint32_t* pl_tile = planes + bh * kD * 4 * wstride + tok0 / 32;
    const int ne0 = min(kPsChunk, nact);
    if (!staged) {
      ps_stage_scales<A16>(S, scb, scales + bh * kD * sstride + tok0 / 64, sstride, nch, nbv);
      ps_stage_words<A16>(S, wb0, 0, ne0, pl_tile, wstride, nwv);
    }
    cp_async_wait_all();
    __syncthreads();
    // per-block constants C_blk (four partial sums per block) and the first weights
    {
      const int b2 = (threadIdx.x & 31) * 2, part = threadIdx.x >> 5;
      float a0 = 0.0f, a1 = 0.0f;
      if (b2 < nbv)
        for (int sl = part; sl < nch; sl += kPsThreads / 32) {
          const float2 f =
              __half22float2(*reinterpret_cast<const __half2*>(&scb[sl * kPsBlocks + b2]));
          const float qo = S.qo[sl];
          a0 = __fadd_rn(a0, __fmul_rn(qo, f.x));
          a1 = __fadd_rn(a1, __fmul_rn(qo, f.y));
        }
      *reinterpret_cast<float2*>(&S.red[part][b2]) = make_float2(a0, a1);
    }
    ps_weights(S, scb, wb0, 0, ne0, nbv);
    __syncthreads();
    if (threadIdx.x < kPsBlocks) {
      float c = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k) c = __fadd_rn(c, S.red[k][threadIdx.x]);
      S.Cs[threadIdx.x] = c;
    }

    // the next tile of the same row can be staged during this tile's last chunk
    const bool pref = dbl && u_next < u_end && u_next / units_per_row == bh;
    bool staged_next = false;
    int next_wb0 = 0;
    const int half = warp >> 2, wl = (warp & 3) * 32 + lane;  // plane parity, word
    float acc[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) acc[k] = 0.0f;
    int buf = wb0;
    for (int e0 = 0; e0 < nact; e0 += kPsChunk, buf ^= 1) {
      const int ne = min(kPsChunk, nact - e0);
      const int e1 = e0 + kPsChunk;
      const int ne1 = min(kPsChunk, nact - e1);
      if (ne1 > 0) {
        ps_stage_words<A16>(S, buf ^ 1, e1, ne1, pl_tile, wstride, nwv);
      } else if (pref) {
        const PsTile NT = ps_tile_at(u_next, u_end, units_per_row);
        const int64_t ntok0 = NT.tok0;
        const int nnwv = ps_valid_words(NT, n);
        ps_stage_scales<A16>(S, &S.sc[sbuf ^ 1][0][0], scales + bh * kD * sstride + ntok0 / 64,
                             sstride, nch, nnwv / 2);
        ps_stage_words<A16>(S, buf ^ 1, 0, ne0, planes + bh * kD * 4 * wstride + ntok0 / 32,
                            wstride, nnwv);
        staged_next = true;
        next_wb0 = buf ^ 1;
      }
      const uint32_t* wp = &S.words[buf][half][wl];
      const float* tp = &S.Wt[buf][half][wl >> 1];
      const int ne_w = (warp & 3) * 32 < nwv ? ne : 0;  // warps past the tile's end idle
#pragma unroll 2
      for (int e = half; e < ne_w; e += 2, wp += 2 * kPsWords, tp += 2 * kPsBlocks) {
        const uint32_t w = *wp;
        const float wt = *tp;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (w & (1u << i)) acc[i] += wt;
      }
      if (ne1 > 0) {
        ps_weights(S, scb, buf ^ 1, e1, ne1, nbv);
        cp_async_wait_all();  // the next chunk (nothing else is in flight)
      }
      __syncthreads();
    }
    if (nact == 0) {
      if (pref) {  // nothing to prefetch but the (empty) tile bookkeeping
        staged_next = false;
      }
      __syncthreads();  // Cs written above must be visible
    }
    // odd-plane partial sums through the (now idle) weight buffers: lane l's eight
    // float4s go to 16-byte slots k ^ (l & 7), so each quarter-warp hits 8 distinct
    // bank groups
    float4* red = reinterpret_cast<float4*>(&S.Wt[0][0][0]) + ((warp & 3) * 32 + lane) * 8;
    const int sw = lane & 7;
    if (half == 1) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        red[k ^ sw] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
    }
    __syncthreads();
    if (half == 0 && wl < nwv) {
      const float c = S.Cs[wl >> 1];
      float4* orow = reinterpret_cast<float4*>(scores + bh * n + tok0 + wl * 32);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 o = red[k ^ sw];
        orow[k] = make_float4((acc[4 * k] + o.x) + c, (acc[4 * k + 1] + o.y) + c,
                              (acc[4 * k + 2] + o.z) + c, (acc[4 * k + 3] + o.w) + c);
      }
    }
    __syncthreads();  // buffers are reused by the next tile
    u = u_next;
    staged = staged_next;
    if (staged_next) {
      sbuf ^= 1;
      wb0 = next_wb0;
    } else {
      wb0 = 0;
    }
  }
  cp_async_wait_all();  // nothing may be left in flight at exit
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

template <int G, bool A16>
static int planes_t(const Dims& s, const uint32_t* planes, const uint16_t* scales,
                    const uint8_t* plan, const uint16_t* q, float* scores, cudaStream_t st) {
  auto kern = score_planes_kernel<G, A16>;
  if (int rc = set_smem_limit((const void*)kern, sizeof(PsSmem), "score_planes: smem attribute"))
    return rc;
  const int64_t units_per_row = (s.n + kPsUnit - 1) / kPsUnit;
  const int64_t total = units_per_row * s.B * s.Hkv;
  const int64_t grid = imin64(total, (int64_t)sm_count() * kPsCtasPerSm);
  kern<<<(unsigned)grid, kPsThreads, sizeof(PsSmem), st>>>(planes, scales, plan, q, s.Hq, s.Hkv,
                                                          s.n, s.ncap, units_per_row, total,
                                                          scores);
  return check_launch("score_planes");
}

int launch_score_planes(const Dims& s, const uint32_t* planes, const uint16_t* scales,
                        const uint8_t* plan, const uint16_t* q, float* scores, cudaStream_t st) {
  const bool a16 = (s.ncap % 512 == 0) && ((uintptr_t)planes % 16 == 0) &&
                   ((uintptr_t)scales % 16 == 0);
  switch (s.G) {
    case 1: return a16 ? planes_t<1, true>(s, planes, scales, plan, q, scores, st) : planes_t<1, false>(s, planes, scales, plan, q, scores, st);
    case 2: return a16 ? planes_t<2, true>(s, planes, scales, plan, q, scores, st) : planes_t<2, false>(s, planes, scales, plan, q, scores, st);
    case 4: return a16 ? planes_t<4, true>(s, planes, scales, plan, q, scores, st) : planes_t<4, false>(s, planes, scales, plan, q, scores, st);
    default: return a16 ? planes_t<8, true>(s, planes, scales, plan, q, scores, st) : planes_t<8, false>(s, planes, scales, plan, q, scores, st);
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
  return check_launch("score_quest");
}

}  // namespace sd
