// GATHER-ATT for many long rows at once (HashAttention: Semantic Sparsity for Faster
// Inference, 2.1: o = sum_{i in I} e^{z_i} v_i / sum_{j in I} e^{z_j}, z_i = <q, k_i>
// scaled by 1/sqrt(d); 2.5: page size 1, the selected rows read in place; the
// block-sparse Quest decode of OasisKV / Quest gathers 16-token blocks the same way).
//
// Every warp is an independent online softmax over a contiguous range of 16-token
// groups (the rows' selected tokens in row-major order; warp w of NW takes groups
// [w T / NW, (w + 1) T / NW)), so every warp moves the same number of bytes.
//  * The K and V rows come from HBM straight into registers by 16-byte loads, laid
//    out as the tensor cores' operands: lane (gid, tig) loads chunks tig, tig + 4,
//    tig + 8, tig + 12 of the K rows of positions gid and 8 + gid (q's fragments
//    take the same channel order; a dot product does not depend on it), and chunks
//    gid, 8 + gid of the V rows of positions 2tig, 2tig + 1, 2tig + 8, 2tig + 9
//    (paired per dimension by byte permutes into V^T's fragments).  Each 4-lane (K)
//    or 8-lane (V) set reads whole 32-byte sectors.
//  * S = Q K^T as m16n8k16 bf16 MMAs (M: the G query heads, zero-padded to 16; N: 8
//    positions; K: 16 channels).  p = 2^(z log2 e - m) in fp32 with the reference
//    max m raised only when a group's max exceeds it by more than 2^8 (then O and l
//    are rescaled).  O^T += V^T P^T with P^T split into bf16 hi and lo parts (B
//    columns, summed at the end), so P keeps ~16 significant bits.
//  * The next group's K rows are requested as soon as S is computed, its V rows
//    after the P V product; the group three ahead is prefetched into L2 and the
//    indices run four groups ahead, so a warp waits on little but the HBM stream.
//  * At the end of its part of a row each warp writes its (m, l, O) as one partial;
//    the warp that completes the row's count of partials (a ticket) combines them in
//    slot order and writes out and lse.
// Registers bound the design (8 warps per SM at up to 255 registers).  Staging the
// rows through shared memory with cp.async, bulk copies or loader warps measured
// slower on this gather.
#include "sd_internal.cuh"
#include "sd_mma.cuh"

namespace sd {
namespace {

constexpr int kAsGrp = 16;     // tokens per group (one k-step of the P V product)
constexpr int kAsWarps = 4;    // warps per CTA
constexpr int kAsThreads = 32 * kAsWarps;
constexpr int kAsCtasPerSm = 2;
constexpr float kAsLog2e = 1.4426950408889634f;
constexpr float kAsLn2 = 0.6931471805599453f;
constexpr float kAsSlack = 8.0f;  // log2 headroom before the reference max is raised

struct AsArgs {
  const uint16_t* q;
  const uint16_t* K;
  const uint16_t* V;
  const int32_t* idx;
  int64_t idx_stride;
  const int32_t* count;
  int Hq, Hkv;
  int64_t n, ncap, rows;
  int max_count;
  float sl2;        // scale * log2(e)
  int64_t gpr;      // groups per row, ceil(max_count / 16)
  int64_t total;    // rows * gpr
  int slots;        // partial slots per row in the workspace
  uint32_t* ticket; // [rows], zero at launch
  float* part_o;    // [rows][slots][G][kD]
  float2* part_ml;  // [rows][slots][G]: (m in log2 units, l)
  float* out;
  float* lse;
};

// The warp whose range holds group g (ranges [w T / NW, (w + 1) T / NW)).
__device__ __forceinline__ int64_t as_warp_of(int64_t g, int64_t T, int64_t NW) {
  return ((g + 1) * NW - 1) / T;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Row counts 32 rows at a time: lane j holds row rb + j's (clamped to max_count).
struct AsCounts {
  int64_t rb;
  int cnt;
  __device__ __forceinline__ int of(const AsArgs& a, int64_t r, int lane) {
    if (r >= rb + 32) {
      rb = r;
      cnt = r + lane < a.rows ? min(a.count[r + lane], a.max_count) : 0;
    }
    return __shfl_sync(0xFFFFFFFFu, cnt, (int)(r - rb));
  }
};

// A group's position: row r, group gi of the row (no divisions in the loop).
struct AsPos {
  int64_t r;
  int gi;
};
// The warp's range [begin, end) of groups, as positions.
struct AsRange {
  AsPos end;
  __device__ __forceinline__ bool in(const AsPos& p) const {
    return p.r < end.r || (p.r == end.r && p.gi < end.gi);
  }
};

// The first position >= p in the range whose group holds selected tokens; past the
// range: p.r = end row + 1 (or beyond), which `in` rejects.
__device__ __forceinline__ AsPos as_next(AsCounts& cn, const AsArgs& a, AsPos p,
                                         const AsRange& rg, int lane) {
  while (rg.in(p)) {
    const int c = cn.of(a, p.r, lane);
    const int held = c > 0 ? (c + kAsGrp - 1) / kAsGrp : 0;
    if (p.gi < held) return p;
    ++p.r;
    p.gi = 0;
  }
  return p;
}

// Group p's indices: lane l < 16 holds position l's token (-1 past the count).
struct AsIdx {
  int tok;
};
__device__ __forceinline__ AsIdx as_idx(AsCounts& cn, const AsArgs& a, const AsPos& p,
                                        const AsRange& rg, int lane) {
  AsIdx x;
  x.tok = -1;
  if (rg.in(p)) {
    const int t0 = p.gi * kAsGrp;
    const int c = cn.of(a, p.r, lane);
    if (lane < kAsGrp && t0 + lane < c) x.tok = a.idx[p.r * a.idx_stride + t0 + lane];
  }
  return x;
}
__device__ __forceinline__ uint32_t as_mask(const AsArgs& a, int tok, int lane) {
  return __ballot_sync(0xFFFFFFFFu, lane < kAsGrp && tok >= 0 && tok < a.n) & 0xFFFFu;
}

// 16 bytes from global memory (streaming), or zeros where v is false; volatile, so
// that the loads stay where the loop issues them (after the registers' last use).
__device__ __forceinline__ uint4 as_ld(const uint4* ptr, bool v) {
  uint4 x;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %5, 0;\n\t"
      "mov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\tmov.b32 %3, 0;\n\t"
      "@p ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];\n\t}\n"
      : "=&r"(x.x), "=&r"(x.y), "=&r"(x.z), "=&r"(x.w)
      : "l"(ptr), "r"((uint32_t)v));
  return x;
}

__device__ __forceinline__ uint4 as_ld_all(const uint4* ptr) {
  uint4 x;
  asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
               : "l"(ptr));
  return x;
}

// Issues the loads of a group's K rows: lane (gid, tig) takes 16-byte chunks tig,
// tig + 4, tig + 8, tig + 12 of the rows of positions gid and 8 + gid.
__device__ __forceinline__ void as_load_k(uint4 (&kr)[2][4], const AsArgs& a, int64_t row,
                                          int tok_lane, uint32_t mask, int gid, int tig) {
  const uint4* Kr = reinterpret_cast<const uint4*>(a.K + row * a.ncap * kD);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int p = gid + 8 * h;
    const int t = __shfl_sync(0xFFFFFFFFu, tok_lane, p);
    const bool v = (mask >> p) & 1u;
    const uint4* src = Kr + (int64_t)(v ? t : 0) * 16 + tig;
    if (mask == 0xFFFFu) {  // every position holds a token: plain loads
#pragma unroll
      for (int j = 0; j < 4; ++j) kr[h][j] = as_ld_all(src + 4 * j);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) kr[h][j] = as_ld(src + 4 * j, v);
    }
  }
}
// ... of its V rows: lane (gid, tig) takes positions 2tig, 2tig + 1, 2tig + 8, 2tig + 9,
// 16-byte chunks gid and 8 + gid (dimensions 8gid .. 8gid + 7 and 64 + 8gid ..).
__device__ __forceinline__ void as_load_v(uint4 (&vr)[4][2], const AsArgs& a, int64_t row,
                                          int tok_lane, uint32_t mask, int gid, int tig) {
  const uint4* Vr = reinterpret_cast<const uint4*>(a.V + row * a.ncap * kD);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int p = 2 * tig + (w & 1) + 8 * (w >> 1);
    const int t = __shfl_sync(0xFFFFFFFFu, tok_lane, p);
    const bool v = (mask >> p) & 1u;
    const uint4* src = Vr + (int64_t)(v ? t : 0) * 16 + gid;
    if (mask == 0xFFFFu) {
#pragma unroll
      for (int h = 0; h < 2; ++h) vr[w][h] = as_ld_all(src + 8 * h);
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) vr[w][h] = as_ld(src + 8 * h, v);
    }
  }
}

__device__ __forceinline__ uint32_t u4_at(const uint4& x, int i) {
  return i == 0 ? x.x : i == 1 ? x.y : i == 2 ? x.z : x.w;
}

// Row r's slot for warp wg and the row's count of partials.
__device__ __forceinline__ void as_slot(const AsArgs& a, int64_t r, int64_t wg, int64_t NW,
                                        int& slot, int& np) {
  const int64_t wf = as_warp_of(r * a.gpr, a.total, NW);
  const int64_t wl = as_warp_of((r + 1) * a.gpr - 1, a.total, NW);
  np = (int)(wl - wf + 1);
  slot = (int)(wg - wf);
}

// After the warp's partial for row r is written: the ticket; the warp that brings
// the row's count of partials combines them (slot order) into out and lse.
template <int G>
__device__ __noinline__ void as_finish(const AsArgs& a, int64_t r, int np, int lane) {
  __threadfence();
  __syncwarp();
  uint32_t t = 0;
  if (lane == 0) t = atomicAdd(&a.ticket[r], 1u);
  t = __shfl_sync(0xFFFFFFFFu, t, 0);
  if (t != (uint32_t)(np - 1)) return;
  __threadfence();
  const int b = (int)(r / a.Hkv), h = (int)(r % a.Hkv);
  const float2* ml = a.part_ml + r * a.slots * G;
  const float* po = a.part_o + r * a.slots * G * kD;
  for (int g = 0; g < G; ++g) {
    float m = -INFINITY;
    for (int p = 0; p < np; ++p) m = fmaxf(m, __ldcg(&ml[p * G + g].x));
    float ls = 0.0f;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int p = 0; p < np; ++p) {
      const float2 x = __ldcg(&ml[p * G + g]);
      if (x.x == -INFINITY) continue;  // empty: its O was not written
      const float wgt = exp2f(x.x - m);
      ls = fmaf(x.y, wgt, ls);
      const float4 v = __ldcg(reinterpret_cast<const float4*>(po + (p * G + g) * kD) + lane);
      acc.x = fmaf(v.x, wgt, acc.x);
      acc.y = fmaf(v.y, wgt, acc.y);
      acc.z = fmaf(v.z, wgt, acc.z);
      acc.w = fmaf(v.w, wgt, acc.w);
    }
    const float inv = ls > 0.0f ? 1.0f / ls : 0.0f;  // an empty set gives o = 0
    float* dst = a.out + ((int64_t)b * a.Hq + h * G + g) * kD + 4 * lane;
    dst[0] = acc.x * inv;
    dst[1] = acc.y * inv;
    dst[2] = acc.z * inv;
    dst[3] = acc.w * inv;
    if (a.lse && lane == 0)
      a.lse[(int64_t)b * a.Hq + h * G + g] = ls > 0.0f ? (m + log2f(ls)) * kAsLn2 : -INFINITY;
  }
}

// An empty partial for row r (no selected token in the warp's part of it).
template <int G>
__device__ __forceinline__ void as_flush_empty(const AsArgs& a, int64_t r, int64_t wg, int64_t NW,
                                               int lane) {
  int slot, np;
  as_slot(a, r, wg, NW, slot, np);
  if (lane < G) a.part_ml[(r * a.slots + slot) * G + lane] = make_float2(-INFINITY, 0.0f);
  as_finish<G>(a, r, np, lane);
}

// The per-warp state of the online softmax over the warp's part of a row.
template <int G>
struct AsState {
  static constexpr int NT = G == 8 ? 2 : 1;
  // O^T accumulators: m-tile mt, rows gid / gid + 8 <-> dimensions 8gid + mt /
  // 64 + 8gid + mt; columns: P^T's heads, bf16 hi and lo parts (NT n-tiles)
  float o[8][NT][4];
  float mref, l;  // reference max (log2 units) of the lane's head gid; its partial sum
};

// The warp's groups in flight: the K and V fragments of the group at `pos` (mask:
// its positions holding a token), and the positions and indices of the three groups
// after it -- the next one's rows load into these registers as they free up, the
// one three ahead is prefetched into L2.
struct AsSlot {
  uint4 k[2][4], v[4][2];
  AsPos pos, npos, ppos, fpos;  // this group and the three after it
  uint32_t mask;
  int ntok, ptok, ftok;         // the indices of those three (lanes < 16)
};

// L2 prefetch of a group's K and V rows (lane l: position l / 2, 128-byte line l % 2).
__device__ __forceinline__ void as_prefetch(const AsArgs& a, int64_t row, int tok_lane, int lane) {
  const int p = lane >> 1;
  const int t = __shfl_sync(0xFFFFFFFFu, tok_lane, p);
  if (t >= 0 && t < a.n) {
    const int64_t off = (row * a.ncap + t) * kD + 64 * (lane & 1);
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a.K + off));
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a.V + off));
  }
}

// Processes the group in slot X (next_pos: the group after it), requests the next
// group's rows into X's registers as they free up, prefetches the group three ahead
// into L2 and loads the indices of the group four ahead.
template <int G>
__device__ __forceinline__ void as_step(AsSlot& X, const AsPos next_pos, AsState<G>& St,
                                        const AsArgs& a, AsCounts& cn, AsPos& enum_pos,
                                        const AsRange& rg, int64_t r_last, int64_t wg,
                                        int64_t NW, uint32_t (&qa)[8][2], bool& fresh, int lane) {
  constexpr int NT = AsState<G>::NT;
  const int gid = lane >> 2, tig = lane & 3;
  const bool real = gid < G;
  const int64_t r = X.pos.r;
  if (fresh) {
    // q's A fragments into this warp's shared memory, channels permuted as the K
    // loads are: k-step kk, lane tig holds channels 8(tig + 4(kk >> 1)) + 4(kk & 1) +
    // {0, 1} and + {2, 3}
    const int b = (int)(r / a.Hkv), h = (int)(r % a.Hkv);
    const uint32_t* qr =
        reinterpret_cast<const uint32_t*>(a.q + ((int64_t)b * a.Hq + h * G + (real ? gid : 0)) * kD);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int c0 = 8 * (tig + 4 * (kk >> 1)) + 4 * (kk & 1);
      qa[kk][0] = real ? qr[c0 >> 1] : 0u;
      qa[kk][1] = real ? qr[(c0 >> 1) + 1] : 0u;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) St.o[mt][nt][0] = St.o[mt][nt][1] = St.o[mt][nt][2] = St.o[mt][nt][3] = 0.0f;
    St.mref = -INFINITY;
    St.l = 0.0f;
    fresh = false;
  }
  // S = Q K^T over the group's 16 positions (n-tile h: positions 8h .. 8h + 7)
  float sc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4& x = X.k[h][kk >> 1];
      mma_bf16(sc[h], qa[kk][0], 0u, qa[kk][1], 0u, (kk & 1) ? x.z : x.x, (kk & 1) ? x.w : x.y);
    }
  }
  // the group two ahead: its K rows into this slot (the registers are free now)
  const uint32_t nmask = as_mask(a, X.ntok, lane);
  const bool nin = rg.in(X.npos);
  if (nin) as_load_k(X.k, a, X.npos.r, X.ntok, nmask, gid, tig);
  float x[2][2];
  float mc = -INFINITY;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const bool ok = real && ((X.mask >> (8 * h + 2 * tig + e)) & 1u);
      x[h][e] = ok ? sc[h][e] * a.sl2 : -INFINITY;
      mc = fmaxf(mc, x[h][e]);
    }
  mc = fmaxf(mc, __shfl_xor_sync(0xFFFFFFFFu, mc, 1));
  mc = fmaxf(mc, __shfl_xor_sync(0xFFFFFFFFu, mc, 2));
  const bool need = mc > St.mref + kAsSlack;
  if (__any_sync(0xFFFFFFFFu, need)) {
    const float mnew = need ? mc : St.mref;
    const float al = need ? exp2f(St.mref - mnew) : 1.0f;  // mref = -inf: 0
    // this lane's O^T columns 2tig, 2tig + 1 belong to heads hA, hA + 1, whose
    // factors the lanes of rows hA, hA + 1 of S hold
    const int hA = G == 8 ? 2 * tig : (2 * tig) & 3;
    const float aA = __shfl_sync(0xFFFFFFFFu, al, 4 * hA);
    const float aB = __shfl_sync(0xFFFFFFFFu, al, 4 * (hA + 1));
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        St.o[mt][nt][0] *= aA;
        St.o[mt][nt][1] *= aB;
        St.o[mt][nt][2] *= aA;
        St.o[mt][nt][3] *= aB;
      }
    St.l *= al;
    St.mref = mnew;
  }
  const float mu = St.mref == -INFINITY ? 0.0f : St.mref;
  float p[2][2];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      p[h][e] = exp2f(x[h][e] - mu);
      St.l += p[h][e];
    }
  // P^T as bf16 hi + lo parts: b0 holds positions 2tig, 2tig + 1 of column gid,
  // b1 positions 2tig + 8, 2tig + 9.  G = 8: n-tile 0 the heads' hi parts, n-tile
  // 1 their lo parts; else columns 0..3 hi, 4..7 lo (head gid - 4, from lane - 16)
  uint32_t bh[NT][2];
  {
    const uint32_t h0 = pack_bf16(p[0][0], p[0][1]), h1 = pack_bf16(p[1][0], p[1][1]);
    const uint32_t l0 = pack_bf16(p[0][0] - bf16_lo(h0), p[0][1] - bf16_hi(h0));
    const uint32_t l1 = pack_bf16(p[1][0] - bf16_lo(h1), p[1][1] - bf16_hi(h1));
    if constexpr (G == 8) {
      bh[0][0] = h0;
      bh[0][1] = h1;
      bh[NT - 1][0] = l0;
      bh[NT - 1][1] = l1;
    } else {
      const uint32_t s0 = __shfl_xor_sync(0xFFFFFFFFu, l0, 16);
      const uint32_t s1 = __shfl_xor_sync(0xFFFFFFFFu, l1, 16);
      bh[0][0] = gid < 4 ? h0 : s0;
      bh[0][1] = gid < 4 ? h1 : s1;
    }
  }
  // O^T += V^T P^T: a0 pairs positions 2tig, 2tig + 1 of row gid's dimension, a1
  // row gid + 8's, a2 / a3 positions + 8
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int reg = mt >> 1;
    const uint32_t sel = (mt & 1) ? 0x7632u : 0x5410u;
    const uint32_t a0 = __byte_perm(u4_at(X.v[0][0], reg), u4_at(X.v[1][0], reg), sel);
    const uint32_t a1 = __byte_perm(u4_at(X.v[0][1], reg), u4_at(X.v[1][1], reg), sel);
    const uint32_t a2 = __byte_perm(u4_at(X.v[2][0], reg), u4_at(X.v[3][0], reg), sel);
    const uint32_t a3 = __byte_perm(u4_at(X.v[2][1], reg), u4_at(X.v[3][1], reg), sel);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma_bf16(St.o[mt][nt], a0, a1, a2, a3, bh[nt][0], bh[nt][1]);
  }
  if (nin) as_load_v(X.v, a, X.npos.r, X.ntok, nmask, gid, tig);
  // the group three ahead: its rows into L2; the one after that: its indices
  if (rg.in(X.fpos)) as_prefetch(a, X.fpos.r, X.ftok, lane);
  const AsPos far = enum_pos;
  const AsIdx fi = as_idx(cn, a, far, rg, lane);
  if (rg.in(enum_pos)) enum_pos = as_next(cn, a, AsPos{enum_pos.r, enum_pos.gi + 1}, rg, lane);
  // row r ends before the next group: its partial; rows between get empty ones
  const int64_t rn = rg.in(next_pos) ? next_pos.r : r_last + 1;
  if (rn != r) {
    int slot, np;
    as_slot(a, r, wg, NW, slot, np);
    float lr = St.l + __shfl_xor_sync(0xFFFFFFFFu, St.l, 1);
    lr += __shfl_xor_sync(0xFFFFFFFFu, lr, 2);
    // O^T columns 2tig, 2tig + 1: G = 8 heads 2tig, 2tig + 1 (hi in n-tile 0, lo in
    // 1); else tig < 2 the hi parts of heads 2tig, 2tig + 1 and lane + 2 their lo
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (G == 8) {
          St.o[mt][0][e] += St.o[mt][NT - 1][e];
        } else {
          St.o[mt][0][e] += __shfl_xor_sync(0xFFFFFFFFu, St.o[mt][0][e], 2);
        }
      }
    if (G == 8 || tig < 2) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if (2 * tig + e < G) {
          float* po = a.part_o + ((r * a.slots + slot) * G + 2 * tig + e) * kD;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            po[8 * gid + mt] = St.o[mt][0][e];
            po[64 + 8 * gid + mt] = St.o[mt][0][2 + e];
          }
        }
      }
    }
    if (real && tig == 0) a.part_ml[(r * a.slots + slot) * G + gid] = make_float2(St.mref, lr);
    as_finish<G>(a, r, np, lane);
    for (int64_t e2 = r + 1; e2 < rn; ++e2) as_flush_empty<G>(a, e2, wg, NW, lane);
    fresh = true;
  }
  X.pos = X.npos;
  X.mask = nmask;
  X.npos = X.ppos;
  X.ntok = X.ptok;
  X.ppos = X.fpos;
  X.ptok = X.ftok;
  X.fpos = far;
  X.ftok = fi.tok;
}

template <int G>
__global__ void __launch_bounds__(kAsThreads, kAsCtasPerSm) attend_stream_kernel(AsArgs a) {
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int64_t NW = (int64_t)gridDim.x * kAsWarps;
  const int64_t wg = (int64_t)blockIdx.x * kAsWarps + (threadIdx.x >> 5);
  const int64_t g0 = wg * a.total / NW, g1 = (wg + 1) * a.total / NW;
  if (g0 >= g1) return;
  uint32_t qa[8][2];
  AsCounts cn;
  const AsPos p0{g0 / a.gpr, (int)(g0 % a.gpr)};
  AsRange rg;
  rg.end = AsPos{g1 / a.gpr, (int)(g1 % a.gpr)};
  cn.rb = p0.r;
  cn.cnt = cn.rb + lane < a.rows ? min(a.count[cn.rb + lane], a.max_count) : 0;
  const int64_t r_last = (g1 - 1) / a.gpr;

  // the group being processed (its K and V in the slot's registers), the next one
  // (its indices in flight, its rows loaded into the slot as the current group's
  // registers free up) and the one after (its indices fetched meanwhile)
  AsSlot X;
  X.pos = as_next(cn, a, p0, rg, lane);
  const int64_t rc0 = rg.in(X.pos) ? X.pos.r : r_last + 1;
  for (int64_t rr = p0.r; rr < rc0; ++rr) as_flush_empty<G>(a, rr, wg, NW, lane);  // no tokens
  if (!rg.in(X.pos)) return;
  auto after = [&](const AsPos& q) {
    return rg.in(q) ? as_next(cn, a, AsPos{q.r, q.gi + 1}, rg, lane) : q;
  };
  X.npos = after(X.pos);
  X.ppos = after(X.npos);
  X.fpos = after(X.ppos);
  AsPos enum_pos = after(X.fpos);
  {
    const AsIdx ia = as_idx(cn, a, X.pos, rg, lane);
    X.mask = as_mask(a, ia.tok, lane);
    as_load_k(X.k, a, X.pos.r, ia.tok, X.mask, gid, tig);
    as_load_v(X.v, a, X.pos.r, ia.tok, X.mask, gid, tig);
    X.ntok = as_idx(cn, a, X.npos, rg, lane).tok;
    X.ptok = as_idx(cn, a, X.ppos, rg, lane).tok;
    X.ftok = as_idx(cn, a, X.fpos, rg, lane).tok;
    if (rg.in(X.npos)) as_prefetch(a, X.npos.r, X.ntok, lane);
    if (rg.in(X.ppos)) as_prefetch(a, X.ppos.r, X.ptok, lane);
  }
  AsState<G> St;
  bool fresh = true;  // the next group starts a row: its q and state
  while (rg.in(X.pos))
    as_step<G>(X, X.npos, St, a, cn, enum_pos, rg, r_last, wg, NW, qa, fresh, lane);
}

template <int G>
int as_launch(const AsArgs& a, int grid, cudaStream_t st) {
  attend_stream_kernel<G><<<(unsigned)grid, kAsThreads, 0, st>>>(a);
  note_launches(1);
  return check_launch("attend stream");
}

}  // namespace

// The streaming gather-attend applies when the rows hold at least kAsMinUnitsPerCta
// units per CTA of a full grid and the partial slots fit the workspace that
// sd_gather_attend_workspace_size() sizes; returns 1 (not launched) otherwise.
int launch_attend_stream(const Dims& s, const uint16_t* q, const uint16_t* K, const uint16_t* V,
                         const int32_t* idx, int64_t idx_stride, const int32_t* count,
                         int64_t max_count, float scale, float* out, float* lse,
                         uint32_t* ticket, float* part_o, float2* part_ml, int slots_avail,
                         cudaStream_t st) {
  constexpr int kAsMinGroupsPerWarp = 4;
  const int64_t rows = (int64_t)s.B * s.Hkv;
  const int64_t gpr = (max_count + kAsGrp - 1) / kAsGrp;
  const int64_t total = rows * gpr;
  const int64_t grid = (int64_t)device_sm_count() * kAsCtasPerSm;
  const int64_t NW = grid * kAsWarps;
  if (gpr == 0 || total < NW * kAsMinGroupsPerWarp || ((uintptr_t)q & 15u) != 0) return 1;
  const int64_t L = total / NW;  // the shortest range (>= 1)
  const int64_t segs = imin64(NW, 1 + (gpr - 1 + L - 1) / L);
  if (segs > slots_avail) return 1;
  if (cudaMemsetAsync(ticket, 0, sizeof(uint32_t) * rows, st) != cudaSuccess)
    return check_launch("attend stream: ticket clear");
  AsArgs a;
  a.q = q;
  a.K = K;
  a.V = V;
  a.idx = idx;
  a.idx_stride = idx_stride;
  a.count = count;
  a.Hq = s.Hq;
  a.Hkv = s.Hkv;
  a.n = s.n;
  a.ncap = s.ncap;
  a.rows = rows;
  a.max_count = (int)max_count;
  a.sl2 = scale * kAsLog2e;
  a.gpr = gpr;
  a.total = total;
  a.slots = slots_avail;
  a.ticket = ticket;
  a.part_o = part_o;
  a.part_ml = part_ml;
  a.out = out;
  a.lse = lse;
  switch (s.G) {
    case 1: return as_launch<1>(a, (int)grid, st);
    case 2: return as_launch<2>(a, (int)grid, st);
    case 4: return as_launch<4>(a, (int)grid, st);
    default: return as_launch<8>(a, (int)grid, st);
  }
}

}  // namespace sd
