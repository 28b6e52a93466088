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

// Builds R for row bh = b * Hkv + h.  Every thread of the calling group runs it
// and `bar()` synchronises exactly that group; threads t < kD (t = the thread's
// index within the group) do the per-channel work, warp t / 32 == 0 the scan.
template <int G, class Bar>
__device__ __noinline__ void ps_build_row(PsRow& R, int t, const uint16_t* __restrict__ q,
                                          const uint8_t* __restrict__ plan, int b, int h, int Hq,
                                          int64_t bh, Bar bar) {
  const int lane = t & 31;
  if (t < kD) {
    const int j = t;
    float a = 0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g)
      a = __fadd_rn(a, bf16_to_f32(q[((int64_t)b * Hq + h * G + g) * kD + j]));
    R.qt[j] = a;
    R.tb[j] = min((int)plan[bh * kD + j], 4);  // a plan holds 0..4 bits per channel
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
