// Per-row tables of the bit-plane scan, shared by the scan kernel and the
// threshold sample kernel (Fathom: Per-Query Read Depth for Sparse Decoding over
// Offloaded KV Caches, "bit planes per channel" and "per-query reverse
// water-filling").
//
// For one (sequence, KV head) row and its plan t_j (planned bits per channel):
//   q~_j = sum_g q_gj (fp32, g ascending);
//   the active entries (j, p), p < t_j, in order j ascending then p ascending,
//   stored as j * 4 + p; the active channels ("slots") j ascending;
//   qp_e = q~_j * 2^(3-p) per entry and qo = q~_j * (h(t_j) - 8) per slot, with
//   h(t) = 2^(3-t) (t < 4), 0 (t = 4): a token's score is
//   sum_slots fl(qo * s_j,blk) + sum_entries fl(qp_e * s_j,blk) * bit_e.
#pragma once

#include "sd_internal.cuh"

namespace sd {

struct PsRow {
  float qt[kD];           // group-summed query
  float qo[kD];           // q~_j * (h(t_j) - 8) per slot
  int tb[kD];             // planned bits per channel (0..4)
  int slot_of[kD];
  int chan[kD];           // channel of each slot
  uint16_t act[4 * kD];   // active entries j * 4 + p, j ascending
  uint8_t eslot[4 * kD];  // slot of each entry's channel
  float qp[4 * kD];       // q~_j * 2^(3-p) per entry (exact scaling)
  int nact, nch;
};

// The read plan of one row, computed by one warp with the same arithmetic and tie
// order as plan_kernel (sd_plan.cu): the budget largest pairs w_j * 4^-b, ties to
// the lower 4j + b (water-filling), the budget channels of largest sigma2 (fixed)
// or of largest query mass sum_g q_gj^2 (top-q), or 4 bits everywhere (full).  Lane
// l holds channels 4 l .. 4 l + 3 and their pairs (j, 0..3) -- pairs 16 l .. 16 l + 15
// in pair order -- with mass[c] = sum_g q_gj^2 (fp32, g ascending, no fused
// multiply-add) and s2[c] = sigma2 of channel 4 l + c.  Writes tb[j] (shared memory)
// for every channel.
__device__ __forceinline__ bool ps_plan_fixed(int mode) {
  return mode == SD_PLAN_FIXED || mode == SD_PLAN_TOPQ;  // one key per channel
}
// Whether the plan is all-4 or all-0 without a search; then *v is the bits.
__device__ __forceinline__ bool ps_plan_trivial(int mode, int budget, int* v) {
  const int nkeys = (ps_plan_fixed(mode) ? 1 : 4) * kD;
  if (mode == SD_PLAN_FULL || budget >= nkeys || budget <= 0) {
    *v = (mode == SD_PLAN_FULL || budget >= nkeys) ? 4 : 0;
    return true;
  }
  return false;
}
// The lane's 16 pair keys (slots 4c + p; with one key per channel only p = 0 counts).
__device__ __forceinline__ void ps_plan_keys(const float (&mass)[4], const float (&s2)[4], int mode,
                                             uint32_t (&key)[16]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (ps_plan_fixed(mode)) {  // its variance (fixed) or its query mass (top-q)
      key[4 * c] = key_of_f32(mode == SD_PLAN_FIXED ? s2[c] : mass[c]);
      key[4 * c + 1] = key[4 * c + 2] = key[4 * c + 3] = 0u;  // not counted
    } else {
      const float w = __fmul_rn(mass[c], s2[c]);
      const float scale4[4] = {1.0f, 0.25f, 0.0625f, 0.015625f};
#pragma unroll
      for (int p = 0; p < 4; ++p) key[4 * c + p] = key_of_f32(__fmul_rn(w, scale4[p]));
    }
  }
}
// Keys of the warp satisfying pred (every lane calls it).
template <class P>
__device__ __forceinline__ int ps_plan_count(const uint32_t (&key)[16], int per, P pred) {
  int n = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) n += ((i & 3) < per) && pred(key[i]);
  return __reduce_add_sync(0xFFFFFFFFu, n);
}
// Given T, the budget-th largest key: every key above T is taken and the keys equal
// to T in pair order until the budget is met; writes tb[j] for the lane's channels.
__device__ __forceinline__ void ps_plan_finish(int lane, const uint32_t (&key)[16], int mode,
                                               int budget, uint32_t T, int* tb) {
  const int per = ps_plan_fixed(mode) ? 1 : 4;
  const int above = ps_plan_count(key, per, [&](uint32_t k) { return k > T; });
  int eq = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) eq += ((i & 3) < per) && key[i] == T;
  int incl = eq;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  int before = incl - eq;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    int taken = 0;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      if (p >= per) break;
      const uint32_t k = key[4 * c + p];
      const bool e = k == T;
      if (k > T || (e && before < budget - above)) ++taken;
      before += e;
    }
    tb[lane * 4 + c] = ps_plan_fixed(mode) ? (taken ? 4 : 0) : taken;
  }
}

__device__ __forceinline__ void ps_plan_lane(int lane, const float (&mass)[4], const float (&s2)[4],
                                             int mode, int budget, int* tb) {
  int v;
  if (ps_plan_trivial(mode, budget, &v)) {
#pragma unroll
    for (int c = 0; c < 4; ++c) tb[lane * 4 + c] = v;
    return;
  }
  uint32_t key[16];
  ps_plan_keys(mass, s2, mode, key);
  const int per = ps_plan_fixed(mode) ? 1 : 4;
  // T: the largest key value with at least `budget` keys >= it
  uint32_t T = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t cand = T | (1u << bit);
    if (ps_plan_count(key, per, [&](uint32_t k) { return k >= cand; }) >= budget) T = cand;
  }
  ps_plan_finish(lane, key, mode, budget, T, tb);
}

// Loads lane l's query values for channels 4 l .. 4 l + 3 (g ascending) and returns
// their group sum q~ (fp32, g ascending) and mass sum_g q^2 (fp32, no fused
// multiply-add), plus sigma2 of those channels when the mode reads it.  All loads
// are issued before any arithmetic.
template <int G>
__device__ __forceinline__ void ps_load_row(int lane, const uint16_t* __restrict__ q,
                                            const float* __restrict__ sigma2, int b, int h, int Hq,
                                            bool need_s2, float (&qt)[4], float (&mass)[4],
                                            float (&s2)[4]) {
  float x[4][G];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int g = 0; g < G; ++g)
      x[c][g] = bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + lane * 4 + c]);
    s2[c] = need_s2 ? sigma2[(int64_t)h * kD + lane * 4 + c] : 0.0f;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float a = 0.0f, m = 0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      a = __fadd_rn(a, x[c][g]);
      m = __fadd_rn(m, __fmul_rn(x[c][g], x[c][g]));
    }
    qt[c] = a;
    mass[c] = m;
  }
}

// The plan of row (b, h) by one warp from q and sigma2 (see ps_plan_lane).
template <int G>
__device__ __forceinline__ void ps_plan_row_warp(int lane, const uint16_t* __restrict__ q,
                                                 const float* __restrict__ sigma2, int b, int h,
                                                 int Hq, int mode, int budget, int* tb) {
  float qt[4], mass[4], s2[4];
  ps_load_row<G>(lane, q, sigma2, b, h, Hq, mode == SD_PLAN_WATERFILL || mode == SD_PLAN_FIXED,
                 qt, mass, s2);
  ps_plan_lane(lane, mass, s2, mode, budget, tb);
}

// Builds R for row bh = b * Hkv + h.  Every thread of the calling group runs it
// and `bar()` synchronises exactly that group; threads t < kD (t = the thread's
// index within the group) do the per-channel work, warp t / 32 == 0 the scan.
// With pl.on set, the row's plan is computed here (ps_plan_row_warp) instead of
// read from `plan`, and written to pl.out when write_plan.
struct PsPlanIn {
  bool on;
  const float* sigma2;  // unused by the full and top-q modes
  int mode, budget;
  uint8_t* out;
};

template <int G, class Bar>
__device__ __noinline__ void ps_build_row(PsRow& R, int t, const uint16_t* __restrict__ q,
                                          const uint8_t* __restrict__ plan, int b, int h, int Hq,
                                          int64_t bh, Bar bar, const PsPlanIn& pl = PsPlanIn{},
                                          bool write_plan = false) {
  const int lane = t & 31;
  int tb = 0;
  if (pl.on) {  // the plan, by the group's first warp, through slot_of
    if ((t >> 5) == 0)
      ps_plan_row_warp<G>(lane, q, pl.sigma2, b, h, Hq, pl.mode, pl.budget, R.slot_of);
    bar();
    if (t < kD) tb = R.slot_of[t];
    if (write_plan && t < kD && pl.out) pl.out[bh * kD + t] = (uint8_t)tb;
  }
  if (t < kD) {
    const int j = t;
    float a = 0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g)
      a = __fadd_rn(a, bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + j]));
    R.qt[j] = a;
    R.tb[j] = pl.on ? tb : min((int)plan[bh * kD + j], 4);  // 0..4 bits per channel
  }
  bar();
  if ((t >> 5) == 0) {  // active entries and channel slots, j ascending
    int cnt[4], tot = 0, chs = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      cnt[k] = R.tb[lane * 4 + k];
      tot += cnt[k];
      chs += cnt[k] > 0;
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
      for (int p = 0; p < cnt[k]; ++p) R.act[pos++] = (uint16_t)(j * 4 + p);
      if (cnt[k] > 0) {
        R.slot_of[j] = slot;
        R.chan[slot] = j;
        R.qo[slot] = __fmul_rn(R.qt[j], cnt[k] < 4 ? (float)((1 << (3 - cnt[k])) - 8) : -8.0f);
        ++slot;
      } else {
        R.slot_of[j] = 0;
      }
    }
    if (lane == 31) { R.nact = incl; R.nch = inclc; }
  }
  bar();
  if (t < kD) {
    for (int e = t; e < R.nact; e += kD) {
      const int ent = R.act[e], j = ent >> 2, p = ent & 3;
      R.eslot[e] = (uint8_t)R.slot_of[j];
      R.qp[e] = ldexpf(R.qt[j], 3 - p);
    }
  }
  bar();
}

// acc[i] += wt for every set bit i of w (a bit test and a predicated add per bit)
__device__ __forceinline__ void ps_bits(float (&acc)[32], uint32_t w, float wt) {
#pragma unroll
  for (int i = 0; i < 32; ++i)
    asm("{\n\t.reg .pred p;\n\t.reg .b32 t;\n\tand.b32 t, %1, %2;\n\tsetp.ne.b32 p, t, 0;\n\t"
        "@p add.f32 %0, %0, %3;\n\t}"
        : "+f"(acc[i])
        : "r"(w), "r"(1u << i), "f"(wt));
}

// Candidates of the fused scan + top-k: per row, the threshold key thr[row] (from
// the sample kernel); the scan writes hits[row][w], bit i set when token 32 w + i
// competes (lead <= token < tail) and its score key reaches the threshold, for
// every word w of the row, and sets nan[row] when a competing score is NaN.
struct PsCand {
  const uint32_t* thr;
  uint32_t* hits;  // [rows][n32]
  uint32_t* nan;   // [rows]
  int64_t n32;     // words per row (n / 32)
  int64_t lead, tail;
};

// Marks this lane's competing scores that reach the row's threshold in the hit
// masks (warp-collective: every lane of the warp calls it).
__device__ __forceinline__ void ps_mark(const PsCand& cd, int row, uint32_t T, int64_t tok,
                                        bool valid, const float (&v)[32]) {
  const int lane = threadIdx.x & 31;
  const bool all = T == 0;  // key 0 lies below every score's key
  const float Tf = __uint_as_float((T & 0x80000000u) ? (T & 0x7FFFFFFFu) : ~T);
  float t[16];  // the maximum of the 32 scores as a tree (depth 5)
#pragma unroll
  for (int i = 0; i < 16; ++i) t[i] = fmax_nan(v[2 * i], v[2 * i + 1]);
#pragma unroll
  for (int w = 8; w > 0; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = fmax_nan(t[i], t[i + w]);
  const float mx = t[0];
  // almost every lane lies below the threshold: one compare screens its 32 scores
  const bool maybe = valid && (all || !(mx < Tf));  // reaches it, or holds a NaN
  uint32_t hit = 0;
  bool nan = false;
  if (maybe) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const bool in = tok + i >= cd.lead && tok + i < cd.tail;
      nan |= in && v[i] != v[i];
      if (in && (all || v[i] >= Tf)) hit |= 1u << i;
    }
  }
  if (valid) cd.hits[(int64_t)row * cd.n32 + tok / 32] = hit;  // every word, every call
  if (__any_sync(0xFFFFFFFFu, nan) && lane == 0) atomicOr(cd.nan + row, 1u);
}

}  // namespace sd
