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

// The read plan of one row computed by a group of kD threads (thread t: channel
// j = t and its pairs (j, 0..3)), with the same arithmetic and tie order as
// plan_kernel (sd_plan.cu): the budget largest pairs w_j * 4^-b, ties to the
// lower 4j + b (water-filling), the budget channels of largest sigma2 (fixed), or
// 4 bits everywhere (full).  Returns channel t's bits.  sums: 2 * (kD / 32) words
// of shared memory; bar() synchronises the group (threads t >= kD hold no keys).
template <int G, class Bar>
__device__ __forceinline__ int ps_plan_row(int t, const uint16_t* __restrict__ q,
                                           const float* __restrict__ sigma2, int b, int h,
                                           int Hq, int mode, int budget, int* sums, Bar bar) {
  constexpr int NW = kD / 32;
  const int lane = t & 31, warp = t >> 5;
  if (mode == SD_PLAN_FULL) return 4;
  const int nkeys = (mode == SD_PLAN_FIXED ? 1 : 4) * kD;
  if (budget >= nkeys) return 4;
  if (budget <= 0) return 0;
  const int npairs = t >= kD ? 0 : (mode == SD_PLAN_FIXED ? 1 : 4);  // keys of this thread
  if (t >= kD) t = 0;  // (loads in bounds; its keys are not counted)
  uint32_t key[4] = {0u, 0u, 0u, 0u};
  if (mode == SD_PLAN_FIXED) {
    key[0] = key_of_f32(sigma2[(int64_t)h * kD + t]);
  } else {
    float acc = 0.0f;  // gains in fp32, group sum in ascending g, no fused multiply-add
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float x = bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + t]);
      acc = __fadd_rn(acc, __fmul_rn(x, x));
    }
    const float w = __fmul_rn(acc, sigma2[(int64_t)h * kD + t]);
    const float scale4[4] = {1.0f, 0.25f, 0.0625f, 0.015625f};
#pragma unroll
    for (int p = 0; p < 4; ++p) key[p] = key_of_f32(__fmul_rn(w, scale4[p]));
  }
  // group-wide count of keys satisfying pred, through two alternating tables
  int parity = 0;
  auto count = [&](auto pred) {
    int c = 0;
#pragma unroll
    for (int p = 0; p < 4; ++p) c += p < npairs && pred(key[p]);
    c = __reduce_add_sync(0xFFFFFFFFu, c);
    int* tab = sums + parity * NW;
    parity ^= 1;
    if (lane == 0 && warp < NW) tab[warp] = c;
    bar();
    int tot = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) tot += tab[w];
    return tot;
  };
  // T: the largest key value with at least `budget` keys >= it
  uint32_t T = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t cand = T | (1u << bit);
    if (count([&](uint32_t k) { return k >= cand; }) >= budget) T = cand;
  }
  const int above = count([&](uint32_t k) { return k > T; });
  // rank of each key equal to T among the equal keys, in pair order 4j + p
  int eq = 0;
#pragma unroll
  for (int p = 0; p < 4; ++p) eq += p < npairs && key[p] == T;
  int incl = eq;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  int* tab = sums + parity * NW;
  if (lane == 31 && warp < NW) tab[warp] = incl;
  bar();
  int before = incl - eq;
  for (int w = 0; w < warp && w < NW; ++w) before += tab[w];
  int taken = 0;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    if (p >= npairs) break;
    const bool e = key[p] == T;
    if (key[p] > T || (e && before < budget - above)) ++taken;
    before += e;
  }
  return mode == SD_PLAN_FIXED ? (taken ? 4 : 0) : taken;
}

// Builds R for row bh = b * Hkv + h.  Every thread of the calling group runs it
// and `bar()` synchronises exactly that group; threads t < kD (t = the thread's
// index within the group) do the per-channel work, warp t / 32 == 0 the scan.
// With pl.sigma2 set, the row's plan is computed here (ps_plan_row) instead of
// read from `plan`, and written to pl.out when pl.write.
struct PsPlanIn {
  const float* sigma2;
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
  if (pl.sigma2) {  // every thread of the group takes part in the plan's counts
    tb = ps_plan_row<G>(t, q, pl.sigma2, b, h, Hq, pl.mode, pl.budget,
                        reinterpret_cast<int*>(R.slot_of), bar);
    bar();  // slot_of served as the plan's scratch
    if (write_plan && t < kD && pl.out) pl.out[bh * kD + t] = (uint8_t)tb;
  }
  if (t < kD) {
    const int j = t;
    float a = 0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g)
      a = __fadd_rn(a, bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + j]));
    R.qt[j] = a;
    R.tb[j] = pl.sigma2 ? tb : min((int)plan[bh * kD + j], 4);  // 0..4 bits per channel
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

}  // namespace sd
