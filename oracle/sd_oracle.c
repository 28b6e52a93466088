/*
 * CPU ORACLE for the sparse-decode hot path (SCORE -> TOPK -> GATHER-ATT).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the CUDA library computes.  Only the tests, the smoke check
 * and the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or helper with the CUDA library; each side was written from the pages.
 *
 * Arithmetic: double unless the method fixes fp32 (signature chains, water-filling
 * gains, quantiser division), built with -ffp-contract=off so that no FMA is
 * formed behind our back.  OpenMP runs independent (sequence, KV head) units in
 * parallel; no result depends on the thread count.
 *
 * Sources (page title, section/equation):
 *   [HA]  HashAttention: Semantic Sparsity for Faster Inference
 *         (2.1 inputs/outputs and the three stages; 2.2 eq. phi(x), SCORE, H;
 *          2.2 worked example; 2.5 page size 1; 3.1 fixed 128+128 positions)
 *   [FA]  Fathom: Per-Query Read Depth for Sparse Decoding over Offloaded KV Caches
 *         (paragraph "store as bit planes per channel"; paragraph "per-query
 *          reverse water-filling"; paragraph "host planes are channel-contiguous")
 *   [OK]  OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead Sparse
 *         Prefetching (prerequisites: "sparse attention (Quest-style block
 *         summaries)"; core method; method details: 129 blocks incl. 1 local)
 *
 * Readings of points the pages leave open are marked READING below.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------ */
/* number formats                                                                  */
/* ------------------------------------------------------------------------------ */

/* bf16 -> float: the bf16 pattern is the top half of the float pattern. */
static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static uint32_t f32_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

/* IEEE binary32 -> binary16, round to nearest, ties to even (hand-written). */
uint16_t orc_f32_to_f16(float f) {
  uint32_t x = f32_bits(f);
  uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  uint32_t ax = x & 0x7FFFFFFFu;
  if (ax >= 0x7F800000u) return sign | (ax > 0x7F800000u ? 0x7E00u : 0x7C00u);
  int e = (int)(ax >> 23) - 127;         /* unbiased exponent */
  uint32_t mant = ax & 0x7FFFFFu;
  if (e >= -14) {                         /* normal binary16 range (or overflow) */
    if (e > 15) return sign | 0x7C00u;
    uint32_t v = ((uint32_t)(e + 15) << 10) | (mant >> 13);
    uint32_t rem = mant & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (v & 1u))) v += 1; /* may carry to inf */
    return sign | (uint16_t)v;
  }
  /* subnormal binary16: value = m * 2^(e-23) with m the 24-bit significand,
     counted in units of 2^-24 it is m * 2^(e+1); shift right by -(e+1). */
  if (ax == 0) return sign;
  uint32_t m = mant | 0x800000u;
  int shift = -(e + 1);
  if (shift > 25) return sign;
  uint32_t q = m >> shift;
  uint32_t rem = m & ((1u << shift) - 1u);
  uint32_t half = 1u << (shift - 1);
  if (rem > half || (rem == half && (q & 1u))) q += 1;
  return sign | (uint16_t)q;
}

/* binary16 -> binary32 (exact). */
float orc_f16_to_f32(uint16_t h) {
  uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  uint32_t e = (h >> 10) & 0x1Fu, m = h & 0x3FFu;
  uint32_t u;
  if (e == 0x1F) u = sign | 0x7F800000u | (m << 13);
  else if (e != 0) u = sign | ((e + 112u) << 23) | (m << 13);
  else if (m == 0) u = sign;
  else { /* subnormal: m * 2^-24 */
    float f = (float)m * (1.0f / 16777216.0f);
    u = sign | f32_bits(f);
  }
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* threads the oracle's parallel loops use (for reporting a CPU baseline) */
int orc_threads(void) { return omp_get_max_threads(); }
/* sets them (the CPU baseline's single-thread leg); returns the previous count */
int orc_set_threads(int t) {
  int prev = omp_get_max_threads();
  if (t >= 1) omp_set_num_threads(t);
  return prev;
}

static int popcount32(uint32_t x) {
  int c = 0;
  while (x) { x &= x - 1u; ++c; }
  return c;
}

/* ------------------------------------------------------------------------------ */
/* S1  signatures  [HA 2.2, eq. phi(x) = ReLU(sign(F(x)))]                         */
/* ------------------------------------------------------------------------------ */
/*
 * One 32-bit code per input row.  F is either one fp32 projection W1[32][d]
 * (+ b1) or a two-layer MLP: hidden u = max(0, W1[u].x + b1[u]) (hidden units),
 * output o = W2[o].hidden + b2[o].  Bit o of the packed word is 1 iff F_o > 0
 * (ReLU(sign(0)) = 0, so +-0 give 0).
 * Each dot product is the canonical fp32 chain acc = fmaf(w_j, x_j, acc) for
 * j = 0..len-1 from acc = +0, then acc = acc + bias (fmaf is correctly rounded,
 * so any correct implementation of this chain gives the same bits).
 * READING: the pages give no MLP activation or bias; ReLU hidden units and zero
 * biases in the synthetic encoders.
 */
static float fp32_chain(const float* w, const float* x, int len, float bias) {
  float acc = 0.0f;
  for (int j = 0; j < len; ++j) acc = fmaf(w[j], x[j], acc);
  return acc + bias;
}

int orc_sig_encode(const uint16_t* x_bf16, int64_t rows, int d, const float* W1,
                   const float* b1, int hidden, const float* W2, const float* b2,
                   uint32_t* out) {
  if (d < 1 || d > 512 || hidden < 0 || hidden > 1024) return -1;
#pragma omp parallel for schedule(dynamic, 256)
  for (int64_t r = 0; r < rows; ++r) {
    float x[512], hbuf[1024];
    for (int j = 0; j < d; ++j) x[j] = bf16_to_f32(x_bf16[r * d + j]);
    uint32_t word = 0;
    if (hidden == 0) {
      for (int o = 0; o < 32; ++o)
        if (fp32_chain(W1 + (int64_t)o * d, x, d, b1 ? b1[o] : 0.0f) > 0.0f) word |= 1u << o;
    } else {
      for (int u = 0; u < hidden; ++u) {
        float a = fp32_chain(W1 + (int64_t)u * d, x, d, b1 ? b1[u] : 0.0f);
        hbuf[u] = a > 0.0f ? a : 0.0f;
      }
      for (int o = 0; o < 32; ++o)
        if (fp32_chain(W2 + (int64_t)o * hidden, hbuf, hidden, b2 ? b2[o] : 0.0f) > 0.0f)
          word |= 1u << o;
    }
    out[r] = word;
  }
  return 0;
}

/* ------------------------------------------------------------------------------ */
/* S5a  Hamming score  [HA 2.2, SCORE = -H(phi_kv(k), phi_q(q)), H = popcount(XOR)] */
/* ------------------------------------------------------------------------------ */
/*
 * score[b][h][i] = - sum over the query heads g of KV head h of
 *                  popcount(sig[b][h][i] XOR qsig[b][g]).
 * READING: one selection per KV head; the group's per-head scores are summed.
 */
void orc_hamming_score(const uint32_t* sig, int64_t B, int Hq, int Hkv, int64_t n,
                       const uint32_t* qsig, int32_t* score) {
  int G = Hq / Hkv;
#pragma omp parallel for collapse(3) schedule(static)
  for (int64_t b = 0; b < B; ++b)
    for (int h = 0; h < Hkv; ++h)
      for (int64_t i = 0; i < n; ++i) {
        const uint32_t* s = sig + (b * Hkv + h) * n;
        int acc = 0;
        for (int g = 0; g < G; ++g) acc += popcount32(s[i] ^ qsig[b * Hq + h * G + g]);
        score[(b * Hkv + h) * n + i] = -acc;
      }
}

/* ------------------------------------------------------------------------------ */
/* S2  bit-plane index  [FA "store as bit planes per channel"]                     */
/* ------------------------------------------------------------------------------ */
/*
 * Per (sequence, KV head, channel j, 64-token block c):
 *   s = f16_rn(absmax / 7) in fp32 arithmetic, replaced by 1 when it is 0;
 *   code_i = clamp(rint(k_ij / s) + 8, 0, 15)  (fp32 IEEE divide, ties-to-even);
 *   plane p (0 = MSB) holds bit (3 - p) of the code.
 * Layout: planes uint32 [B][Hkv][d][4][nw] (token i is bit i%32 of word i/32),
 *         scales f16   [B][Hkv][d][nb], nb = ceil(n/64) blocks, nw = 2 nb words.
 * READING: the pages fix a 4-bit uniform code with an fp16 scale per channel per
 * 64-token block; absmax/7 with offset 8 is the symmetric [-8, 7] reading.
 * READING (partial block): the pages write keys into the index as they arrive
 * ["compressed-key update" on the KV-write path], so a last block may hold fewer
 * than 64 tokens: its scale is taken over the tokens it holds and the bits of the
 * positions past n are 0 (storage padding, not keys).  A full rebuild of that block
 * on each arrival is what keeps the index equal to this definition.
 */
int orc_plane_build(const uint16_t* K, int64_t B, int Hkv, int64_t n, int d,
                    uint32_t* planes, uint16_t* scales) {
  if (n < 1) return -1;
  int64_t nb = (n + 63) / 64, nw = 2 * nb;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t b = 0; b < B; ++b)
    for (int h = 0; h < Hkv; ++h) {
      const uint16_t* Kh = K + (b * Hkv + h) * n * d;
      for (int j = 0; j < d; ++j) {
        uint32_t* pl = planes + (((b * Hkv + h) * d + j) * 4) * nw;
        memset(pl, 0, sizeof(uint32_t) * 4 * nw);
        for (int64_t c = 0; c < nb; ++c) {
          const int64_t t1 = (c + 1) * 64 < n ? (c + 1) * 64 : n; /* tokens held */
          float amax = 0.0f;
          for (int64_t i = c * 64; i < t1; ++i) {
            float v = fabsf(bf16_to_f32(Kh[i * d + j]));
            if (v > amax) amax = v;
          }
          uint16_t s16 = orc_f32_to_f16(amax / 7.0f);
          if ((s16 & 0x7FFFu) == 0) s16 = 0x3C00u; /* scale 0 -> 1 */
          scales[((b * Hkv + h) * d + j) * nb + c] = s16;
          float s = orc_f16_to_f32(s16);
          for (int64_t i = c * 64; i < t1; ++i) {
            float r = rintf(bf16_to_f32(Kh[i * d + j]) / s);
            int code = r <= -8.0f ? 0 : (r >= 7.0f ? 15 : (int)r + 8);
            for (int p = 0; p < 4; ++p)
              if ((code >> (3 - p)) & 1) pl[p * nw + i / 32] |= 1u << (i % 32);
          }
        }
      }
    }
  return 0;
}

/* t-bit reconstruction from the first t planes (prefix = code >> (4-t) << (4-t)).
 * READING: bin midpoint of [-8s, 8s) split into 2^t bins, i.e.
 *   khat_t = s * (prefix + 2^(3-t) - 8) for t < 4 (0 when t = 0),
 *   khat_4 = s * (code - 8). */
double orc_reconstruct(int prefix, int t, double s) {
  double h = t < 4 ? (double)(1 << (3 - t)) : 0.0;
  return s * ((double)prefix + h - 8.0);
}

/* ------------------------------------------------------------------------------ */
/* S4  read plan  [FA "per-query reverse water-filling"]                           */
/* ------------------------------------------------------------------------------ */
/*
 * mode 0 WATERFILL(budget): gain w_j = fl32(fl32(sum_g q_gj^2) * sigma2_j) (sum
 *   over the GQA group in ascending g).  Starting from b = 0, repeat budget times:
 *   give one more bit to the channel with the largest w_j * 4^-b_j among b_j < 4
 *   (lowest j on ties).  Every b_j = 4 once budget >= 4d.
 * mode 1 FIXED(r): the r channels with the largest sigma2_j (lowest j on ties)
 *   get 4 bits, the others 0.
 * mode 2 FULL: every channel gets 4 bits.
 * One plan per (sequence, KV head): the query heads of a group share it.
 * READING: "average budget B" is sum_j b_j = B bits per token per KV head.
 */
/*
 * mode 4 SPLIT(budget): the budget split across the KV heads of a sequence.  The
 *   sequence's total Hkv * budget bits go, one at a time, to the (head h, channel j)
 *   with the largest w_hj * 4^-b_hj among b_hj < 4, w_hj = fl32(fl32(sum over head
 *   h's group of q_gj^2) * sigma2_hj); ties to the lower h, then the lower j.  With
 *   one KV head it is WATERFILL.
 *   READING: the Fathom page keeps one budget per query and layer by default and
 *   calibrates per-layer budgets; the natural extension of its marginal-gain rule to
 *   the heads of a layer is one greedy over all of them under their summed budget.
 */
static void plan_split(const uint16_t* q, const float* sigma2, int64_t b, int Hq, int Hkv, int d,
                       int budget, uint8_t* plan) {
  int G = Hq / Hkv;
  float* w = (float*)malloc(sizeof(float) * (size_t)Hkv * d);
  for (int h = 0; h < Hkv; ++h)
    for (int j = 0; j < d; ++j) {
      float acc = 0.0f;
      for (int g = 0; g < G; ++g) {
        float x = bf16_to_f32(q[(b * Hq + h * G + g) * d + j]);
        float sq = x * x;
        acc = acc + sq;
      }
      w[h * d + j] = acc * sigma2[(int64_t)h * d + j];
    }
  uint8_t* pb = plan + b * Hkv * d;
  memset(pb, 0, (size_t)Hkv * d);
  int64_t total = (int64_t)Hkv * budget, cap = (int64_t)Hkv * 4 * d;
  if (total > cap) total = cap;
  for (int64_t st = 0; st < total; ++st) {
    int best = -1;
    float bestg = 0.0f;
    for (int hj = 0; hj < Hkv * d; ++hj) {  /* h ascending, then j ascending */
      if (pb[hj] >= 4) continue;
      float gj = ldexpf(w[hj], -2 * pb[hj]);
      if (best < 0 || gj > bestg) { best = hj; bestg = gj; }
    }
    pb[best] += 1;
  }
  free(w);
}

int orc_plan(const uint16_t* q, const float* sigma2, int64_t B, int Hq, int Hkv, int d,
             int mode, int budget, uint8_t* plan) {
  int G = Hq / Hkv;
  if (budget < 0 || mode < 0 || mode > 4 || d < 1 || d > 512) return -1;
  if ((mode == 1 || mode == 3) && budget > d) return -1;
  if (mode == 4) {
    if (budget > 4 * d) return -1;
    for (int64_t b = 0; b < B; ++b) plan_split(q, sigma2, b, Hq, Hkv, d, budget, plan);
    return 0;
  }
  for (int64_t b = 0; b < B; ++b)
    for (int h = 0; h < Hkv; ++h) {
      uint8_t* pb = plan + (b * Hkv + h) * d;
      const float* s2 = sigma2 + (int64_t)h * d;
      if (mode == 2) { memset(pb, 4, d); continue; }
      memset(pb, 0, d);
      if (mode == 3) {
        /* SparQ-style [FA "comparison points": top-r |q| channels at full depth]:
         * the r channels of largest group query mass u_j = sum_g q_gj^2 (fp32, g
         * ascending, no contraction), 4 bits each, ties to the lower channel.
         * READING: a group of G query heads ranks channels by the summed squares,
         * the same query mass the water-filling gain uses, without sigma2. */
        float u[512];
        for (int j = 0; j < d; ++j) {
          float acc = 0.0f;
          for (int g = 0; g < G; ++g) {
            float x = bf16_to_f32(q[(b * Hq + h * G + g) * d + j]);
            float sq = x * x;
            acc = acc + sq;
          }
          u[j] = acc;
        }
        for (int r = 0; r < budget; ++r) {
          int best = -1;
          for (int j = 0; j < d; ++j)
            if (pb[j] == 0 && (best < 0 || u[j] > u[best])) best = j;
          pb[best] = 4;
        }
        continue;
      }
      if (mode == 1) {
        for (int r = 0; r < budget; ++r) {
          int best = -1;
          for (int j = 0; j < d; ++j)
            if (pb[j] == 0 && (best < 0 || s2[j] > s2[best])) best = j;
          pb[best] = 4;
        }
        continue;
      }
      float w[512];
      for (int j = 0; j < d; ++j) {
        float acc = 0.0f;
        for (int g = 0; g < G; ++g) {
          float x = bf16_to_f32(q[(b * Hq + h * G + g) * d + j]);
          float sq = x * x;
          acc = acc + sq;
        }
        w[j] = acc * s2[j];
      }
      int steps = budget < 4 * d ? budget : 4 * d;
      for (int st = 0; st < steps; ++st) {
        int best = -1;
        float bestg = 0.0f;
        for (int j = 0; j < d; ++j) {
          if (pb[j] >= 4) continue;
          float gj = ldexpf(w[j], -2 * pb[j]);
          if (best < 0 || gj > bestg) { best = j; bestg = gj; }
        }
        pb[best] += 1;
      }
    }
  return 0;
}

/* ------------------------------------------------------------------------------ */
/* S5b  bit-plane prefix score  [FA "store as bit planes", "water-filling"]        */
/* ------------------------------------------------------------------------------ */
/*
 * score[b][h][i] = sum_g sum_j q_gj * khat_ij(t = plan_j), khat from the first
 * plan_j planes of channel j and the block's scale (orc_reconstruct), in double,
 * for the n tokens i < n.  The planes hold nb = ceil(n / 64) blocks (2 nb words per
 * plane), as orc_plane_build writes them: a partial last block is scored with its
 * own scale (READING: keys enter the index as they are written).
 */
void orc_plane_score(const uint32_t* planes, const uint16_t* scales, const uint8_t* plan,
                     const uint16_t* q, int64_t B, int Hq, int Hkv, int64_t n, int d,
                     double* score) {
  int G = Hq / Hkv;
  int64_t nb = (n + 63) / 64, nw = 2 * nb;
#pragma omp parallel for collapse(3) schedule(static)
  for (int64_t b = 0; b < B; ++b)
    for (int h = 0; h < Hkv; ++h)
      for (int64_t i = 0; i < n; ++i) {
        const uint8_t* pb = plan + (b * Hkv + h) * d;
        double acc = 0.0;
        for (int g = 0; g < G; ++g) {
          const uint16_t* qg = q + (b * Hq + h * G + g) * d;
          for (int j = 0; j < d; ++j) {
            int t = pb[j];
            const uint32_t* pl = planes + (((b * Hkv + h) * d + j) * 4) * nw;
            int prefix = 0;
            for (int p = 0; p < t; ++p)
              if ((pl[p * nw + i / 32] >> (i % 32)) & 1u) prefix |= 1 << (3 - p);
            double s = (double)orc_f16_to_f32(scales[((b * Hkv + h) * d + j) * nb + i / 64]);
            acc += (double)bf16_to_f32(qg[j]) * orc_reconstruct(prefix, t, s);
          }
        }
        score[(b * Hkv + h) * n + i] = acc;
      }
}

/* Sum of |terms| of each plane score, the scale of its rounding tolerance. */
void orc_plane_score_l1(const uint32_t* planes, const uint16_t* scales, const uint8_t* plan,
                        const uint16_t* q, int64_t B, int Hq, int Hkv, int64_t n, int d,
                        double* l1) {
  int G = Hq / Hkv;
  int64_t nb = (n + 63) / 64, nw = 2 * nb;
#pragma omp parallel for collapse(3) schedule(static)
  for (int64_t b = 0; b < B; ++b)
    for (int h = 0; h < Hkv; ++h)
      for (int64_t i = 0; i < n; ++i) {
        const uint8_t* pb = plan + (b * Hkv + h) * d;
        double acc = 0.0;
        for (int g = 0; g < G; ++g)
          for (int j = 0; j < d; ++j) {
            int t = pb[j];
            const uint32_t* pl = planes + (((b * Hkv + h) * d + j) * 4) * nw;
            int prefix = 0;
            for (int p = 0; p < t; ++p)
              if ((pl[p * nw + i / 32] >> (i % 32)) & 1u) prefix |= 1 << (3 - p);
            double s = (double)orc_f16_to_f32(scales[((b * Hkv + h) * d + j) * nb + i / 64]);
            acc += fabs((double)bf16_to_f32(q[(b * Hq + h * G + g) * d + j]) *
                        orc_reconstruct(prefix, t, s));
          }
        l1[(b * Hkv + h) * n + i] = acc;
      }
}

/* ------------------------------------------------------------------------------ */
/* S3 / S5c  block min/max summaries and block bound  [OK "Quest-style summaries"] */
/* ------------------------------------------------------------------------------ */
/*
 * summ[b][h][c][0][j] = min, summ[b][h][c][1][j] = max of k_ij over the tokens of
 * 16-token block c (the last block may be short).  Values are the exact bf16
 * keys.  READING: -0.0 orders below +0.0 so that min/max are unique bit patterns.
 */
static int bf16_less(uint16_t a, uint16_t b) { /* total order, -0 < +0 */
  uint32_t ka = (a & 0x8000u) ? (uint32_t)(~a & 0xFFFFu) : (uint32_t)(a | 0x8000u);
  uint32_t kb = (b & 0x8000u) ? (uint32_t)(~b & 0xFFFFu) : (uint32_t)(b | 0x8000u);
  return ka < kb;
}

void orc_minmax_build(const uint16_t* K, int64_t B, int Hkv, int64_t n, int d,
                      uint16_t* summ) {
  int64_t nblk = (n + 15) / 16;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t b = 0; b < B; ++b)
    for (int h = 0; h < Hkv; ++h) {
      const uint16_t* Kh = K + (b * Hkv + h) * n * d;
      for (int64_t c = 0; c < nblk; ++c) {
        uint16_t* out = summ + ((b * Hkv + h) * nblk + c) * 2 * d;
        int64_t t1 = (c + 1) * 16 < n ? (c + 1) * 16 : n;
        for (int j = 0; j < d; ++j) {
          uint16_t mn = Kh[c * 16 * d + j], mx = mn;
          for (int64_t t = c * 16 + 1; t < t1; ++t) {
            uint16_t v = Kh[t * d + j];
            if (bf16_less(v, mn)) mn = v;
            if (bf16_less(mx, v)) mx = v;
          }
          out[j] = mn;
          out[d + j] = mx;
        }
      }
    }
}

/* U[b][h][c] = sum_g sum_j max(q_gj * min_cj, q_gj * max_cj), in double. */
void orc_quest_score(const uint16_t* summ, const uint16_t* q, int64_t B, int Hq, int Hkv,
                     int64_t nblk, int d, double* U, double* l1) {
  int G = Hq / Hkv;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t b = 0; b < B; ++b)
    for (int h = 0; h < Hkv; ++h)
      for (int64_t c = 0; c < nblk; ++c) {
        const uint16_t* s = summ + ((b * Hkv + h) * nblk + c) * 2 * d;
        double acc = 0.0, mass = 0.0;
        for (int g = 0; g < G; ++g)
          for (int j = 0; j < d; ++j) {
            double qq = bf16_to_f32(q[(b * Hq + h * G + g) * d + j]);
            double lo = qq * bf16_to_f32(s[j]), hi = qq * bf16_to_f32(s[d + j]);
            double m = lo > hi ? lo : hi;
            acc += m;
            mass += fabs(m);
          }
        U[(b * Hkv + h) * nblk + c] = acc;
        if (l1) l1[(b * Hkv + h) * nblk + c] = mass;
      }
}

/* ------------------------------------------------------------------------------ */
/* S6  exact top-k with forced windows  [HA 2.1 TOPK; HA 3.1; OK method details]  */
/* ------------------------------------------------------------------------------ */
/*
 * Per row of n_units scores (units are tokens when block == 1, blocks of `block`
 * tokens otherwise):
 *   forced units: [0, sink) and [n_units - local, n_units);
 *   candidates:   the units in between; if there are at most k of them all are
 *                 taken, else the first k in the order (score desc, unit asc);
 *   output:       the union in ascending order, each unit expanded to its tokens
 *                 [u*block, min((u+1)*block, n_tokens)).
 * count[row] = number of tokens written; -1 if the row holds a NaN score.
 * READING: the retrieval budget k is counted apart from the forced windows.
 */
typedef struct { double s; int64_t u; } cand_t;

static int cand_cmp(const void* a, const void* b) {
  const cand_t* x = (const cand_t*)a;
  const cand_t* y = (const cand_t*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->u > y->u) - (x->u < y->u);
}

static int i64_cmp(const void* a, const void* b) {
  int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
  return (x > y) - (x < y);
}

/* kind: 0 = int32 scores, 1 = float32 scores, 2 = double scores */
void orc_topk(const void* scores, int kind, int64_t rows, int64_t n_units, int k, int sink,
              int local, int block, int64_t n_tokens, int32_t* idx, int64_t idx_stride,
              int32_t* count) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < rows; ++r) {
    cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (size_t)(n_units > 0 ? n_units : 1));
    int64_t* sel = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_units > 0 ? n_units : 1));
    int bad = 0;
    int64_t lead = sink < n_units ? sink : n_units;
    int64_t tail = n_units - local > lead ? n_units - local : lead;
    int64_t nc = 0, ns = 0;
    for (int64_t u = lead; u < tail; ++u) {
      double s;
      if (kind == 0) s = ((const int32_t*)scores)[r * n_units + u];
      else if (kind == 1) s = ((const float*)scores)[r * n_units + u];
      else s = ((const double*)scores)[r * n_units + u];
      if (s != s) bad = 1;
      c[nc].s = s;
      c[nc].u = u;
      ++nc;
    }
    if (bad) {
      count[r] = -1;
      free(c);
      free(sel);
      continue;
    }
    for (int64_t u = 0; u < lead; ++u) sel[ns++] = u;
    if (nc <= k) {
      for (int64_t i = 0; i < nc; ++i) sel[ns++] = c[i].u;
    } else {
      qsort(c, (size_t)nc, sizeof(cand_t), cand_cmp);
      for (int i = 0; i < k; ++i) sel[ns++] = c[i].u;
    }
    for (int64_t u = tail; u < n_units; ++u) sel[ns++] = u;
    qsort(sel, (size_t)ns, sizeof(int64_t), i64_cmp);
    int64_t w = 0;
    for (int64_t i = 0; i < ns; ++i) {
      int64_t t0 = sel[i] * block, t1 = (sel[i] + 1) * block;
      if (t1 > n_tokens) t1 = n_tokens;
      for (int64_t t = t0; t < t1; ++t) idx[r * idx_stride + w++] = (int32_t)t;
    }
    count[r] = (int32_t)w;
    free(c);
    free(sel);
  }
}

/* ------------------------------------------------------------------------------ */
/* S7  gather-attend  [HA 2.1: o_hat over the selected set, corrected denominator; */
/*                     HA 2.5: rows read in place, page size 1]                   */
/* ------------------------------------------------------------------------------ */
/*
 * For query head g of sequence b (KV head h = g / G), over I = idx[b][h][0..count):
 *   z_i = scale * <q_g, k_i>,  o = sum_i e^{z_i - m} v_i / sum_i e^{z_i - m},
 *   lse = m + log(sum_i e^{z_i - m}),  m = max_i z_i;
 * an empty set gives o = 0 and lse = -inf.  Double throughout.
 */
void orc_gather_attend(const uint16_t* q, const uint16_t* K, const uint16_t* V, int64_t B,
                       int Hq, int Hkv, int64_t n, int d, const int32_t* idx,
                       int64_t idx_stride, const int32_t* count, double scale, double* out,
                       double* lse) {
  int G = Hq / Hkv;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int64_t b = 0; b < B; ++b)
    for (int g = 0; g < Hq; ++g) {
      int h = g / G;
      const int32_t* I = idx + (b * Hkv + h) * idx_stride;
      int64_t c = count[b * Hkv + h];
      const uint16_t* qg = q + (b * Hq + g) * d;
      double* o = out + (b * Hq + g) * d;
      for (int j = 0; j < d; ++j) o[j] = 0.0;
      if (c <= 0) { lse[b * Hq + g] = -INFINITY; continue; }
      double* z = (double*)malloc(sizeof(double) * (size_t)c);
      double m = -INFINITY;
      for (int64_t i = 0; i < c; ++i) {
        const uint16_t* kr = K + ((b * Hkv + h) * n + I[i]) * d;
        double acc = 0.0;
        for (int j = 0; j < d; ++j) acc += (double)bf16_to_f32(qg[j]) * bf16_to_f32(kr[j]);
        z[i] = scale * acc;
        if (z[i] > m) m = z[i];
      }
      double l = 0.0;
      for (int64_t i = 0; i < c; ++i) {
        double a = exp(z[i] - m);
        l += a;
        const uint16_t* vr = V + ((b * Hkv + h) * n + I[i]) * d;
        for (int j = 0; j < d; ++j) o[j] += a * bf16_to_f32(vr[j]);
      }
      for (int j = 0; j < d; ++j) o[j] /= l;
      lse[b * Hq + g] = m + log(l);
      free(z);
    }
}

/* ------------------------------------------------------------------------------ */
/* S8  planned-prefix copy  [FA "host planes are channel-contiguous; one gather    */
/*                           copies the active channels' prefixes"]                */
/* ------------------------------------------------------------------------------ */
/*
 * For every (sequence, KV head, channel j) with plan_j > 0: the first plan_j
 * planes of channel j (plan_j * n/32 words) and channel j's scales are copied
 * from src to dst; everything else in dst is left as it was.
 */
void orc_prefix_copy(const uint32_t* src_planes, const uint16_t* src_scales,
                     const uint8_t* plan, int64_t B, int Hkv, int64_t n, int d,
                     uint32_t* dst_planes, uint16_t* dst_scales) {
  int64_t nw = n / 32, nb = n / 64;
  for (int64_t b = 0; b < B; ++b)
    for (int h = 0; h < Hkv; ++h)
      for (int j = 0; j < d; ++j) {
        int t = plan[(b * Hkv + h) * d + j];
        if (t == 0) continue;
        int64_t base = ((b * Hkv + h) * d + j);
        memcpy(dst_planes + base * 4 * nw, src_planes + base * 4 * nw,
               sizeof(uint32_t) * (size_t)(t * nw));
        memcpy(dst_scales + base * nb, src_scales + base * nb, sizeof(uint16_t) * (size_t)nb);
      }
}

/* ------------------------------------------------------------------------------ */
/* F3  delta selection against a resident set  [OA "method details": intersect the  */
/*     predicted top-K with the resident set, admit at most C non-resident blocks   */
/*     per head, each paired with the least-recently-selected resident block]       */
/* ------------------------------------------------------------------------------ */
/*
 * One decode step of the selection worker, per row r = (sequence, KV head).
 * State (kept by the caller between steps; all -1 initially):
 *   slot_unit [rows][R]   unit held by each of the R resident slots, -1 empty;
 *   slot_last [rows][R]   step at which that unit was last selected, -1 empty;
 *   unit_slot [rows][nu]  slot holding each unit, -1 if it is not resident.
 * Input: the top-k output (idx, count) in units of `block` tokens (tokens of each
 * selected unit expanded, ascending, as the top-k writes them): the predicted set P
 * is every unit u with token u*block listed.  A row with count < 0 (a NaN score)
 * is left alone: plan_count = pool_count = -1.
 * 1. Hits: units of P already resident; their slot_last becomes `step`.
 * 2. Misses, in admission order: forced units first (sink [0, sink), local
 *    [nu - local, nu)), unit ascending; then the others by score descending, unit
 *    ascending (-0.0 equal to +0.0).
 * 3. Eviction targets: the slots not holding a unit of P, by slot_last ascending
 *    (empty slots, -1, first), slot ascending.
 * 4. a = min(C, misses, targets): miss i goes to target i; the target's old unit
 *    (if any) stops being resident; slot_last of the slot becomes `step`.  The plan
 *    lists (slot, unit, evicted unit or -1) for i < a; plan_count = a.
 * 5. pool_idx: for the units of P resident after the step, in unit order, the pool
 *    rows slot*block + t for the unit's tokens t < min(block, n_tokens - u*block);
 *    pool_count = their number.
 * READING: the pages fix the intersection, the cap C, the pairing with a
 * least-recently-selected target and that hits move nothing; which misses go first
 * when more than C are missing, and the order of equally old targets, are not
 * stated: forced units (the local block being written) first, then by score, and
 * the lower slot first are the readings taken.
 */
int orc_delta_select(int64_t rows, int64_t nu, int64_t n_tokens, int block, int sink,
                     int local, const float* scores, const int32_t* idx, int64_t idx_stride,
                     const int32_t* count, int C, int64_t step, int R, int32_t* slot_unit,
                     int64_t* slot_last, int32_t* unit_slot, int32_t* plan_slot,
                     int32_t* plan_unit, int32_t* plan_evict, int32_t* plan_count,
                     int32_t* pool_idx, int64_t pool_stride, int32_t* pool_count) {
  if (block < 1 || R < 1 || C < 0 || step < 0) return -1;
  int32_t* P = malloc(sizeof(int32_t) * (size_t)(nu > 0 ? nu : 1));
  char* inP = malloc((size_t)(R > 0 ? R : 1));
  char* taken = malloc((size_t)(nu > 0 ? nu : 1));
  for (int64_t r = 0; r < rows; ++r) {
    int32_t* su = slot_unit + r * R;
    int64_t* sl = slot_last + r * R;
    int32_t* us = unit_slot + r * nu;
    const float* sc = scores + r * nu;
    const int64_t c = count[r];
    if (c < 0) {
      plan_count[r] = -1;
      pool_count[r] = -1;
      continue;
    }
    /* the predicted units, ascending */
    int64_t np = 0;
    for (int64_t i = 0; i < c; ++i) {
      int32_t t = idx[r * idx_stride + i];
      if (t >= 0 && t < n_tokens && t % block == 0 && t / block < nu) P[np++] = t / block;
    }
    /* 1. hits */
    memset(inP, 0, (size_t)R);
    for (int64_t i = 0; i < np; ++i) {
      int32_t s = us[P[i]];
      if (s >= 0) {
        inP[s] = 1;
        sl[s] = step;
      }
    }
    /* 2-4. admit misses one at a time: the best remaining miss to the oldest target */
    int a = 0;
    for (int64_t i = 0; i < np; ++i) taken[P[i]] = 0;
    while (a < C) {
      int64_t best = -1; /* index into P */
      for (int64_t i = 0; i < np; ++i) {
        int32_t u = P[i];
        if (us[u] >= 0 || taken[u]) continue;
        if (best < 0) { best = i; continue; }
        int32_t v = P[best];
        int fu = u < sink || u >= nu - local, fv = v < sink || v >= nu - local;
        float xu = sc[u], xv = sc[v];
        int better;
        if (fu != fv) better = fu;
        else if (fu) better = u < v;
        else if (xu != xv) better = xu > xv;
        else better = u < v;
        if (better) best = i;
      }
      if (best < 0) break; /* no miss left */
      int s_t = -1;
      for (int s = 0; s < R; ++s) {
        if (inP[s]) continue;
        if (s_t < 0 || sl[s] < sl[s_t]) s_t = s; /* strict: the lower slot on ties */
      }
      if (s_t < 0) break; /* no target left */
      int32_t u = P[best], old = su[s_t];
      if (old >= 0) us[old] = -1;
      su[s_t] = u;
      sl[s_t] = step;
      us[u] = s_t;
      inP[s_t] = 1;
      taken[u] = 1;
      plan_slot[r * (int64_t)C + a] = s_t;
      plan_unit[r * (int64_t)C + a] = u;
      plan_evict[r * (int64_t)C + a] = old;
      ++a;
    }
    plan_count[r] = a;
    /* 5. pool rows of the resident predicted units */
    int64_t pc = 0;
    for (int64_t i = 0; i < np; ++i) {
      int32_t u = P[i], s = us[u];
      if (s < 0) continue;
      int64_t len = n_tokens - (int64_t)u * block;
      if (len > block) len = block;
      for (int64_t t = 0; t < len; ++t) pool_idx[r * pool_stride + pc++] = (int32_t)(s * block + t);
    }
    pool_count[r] = (int32_t)pc;
  }
  free(P);
  free(inP);
  free(taken);
  return 0;
}

/* ------------------------------------------------------------------------------ */
/* F2  block landmarks  [FA results: the "8-token block landmark" scan, a          */
/*     comparison point the 56-bit read is timed against]                          */
/* ------------------------------------------------------------------------------ */
/*
 * READING: the page names the scan and its 8-token blocks only.  The landmark of a
 * block is taken as the mean of its keys: per channel the fp32 sum of the block's
 * held tokens in token order, divided (fp32, IEEE) by their count and rounded to
 * bf16 (nearest, ties to even); a short last block averages the tokens it holds.
 * The block's score is the summed group query's dot product with its landmark,
 * sum_g sum_j q_gj L_j (here in double), like every other scorer's group sum.
 */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

void orc_landmark_build(const uint16_t* K, int64_t B, int Hkv, int64_t n, int d, int blk,
                        uint16_t* L) {
  int64_t nblk = (n + blk - 1) / blk;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t b = 0; b < B; ++b)
    for (int h = 0; h < Hkv; ++h) {
      const uint16_t* Kh = K + (b * Hkv + h) * n * d;
      for (int64_t c = 0; c < nblk; ++c) {
        int64_t t1 = (c + 1) * blk < n ? (c + 1) * blk : n;
        float cnt = (float)(t1 - c * blk);
        for (int j = 0; j < d; ++j) {
          float s = 0.0f;
          for (int64_t t = c * blk; t < t1; ++t) s += bf16_to_f32(Kh[t * d + j]);
          L[((b * Hkv + h) * nblk + c) * d + j] = f32_to_bf16_rne(s / cnt);
        }
      }
    }
}

void orc_landmark_score(const uint16_t* L, const uint16_t* q, int64_t B, int Hq, int Hkv,
                        int64_t nblk, int d, double* U, double* l1) {
  int G = Hq / Hkv;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t b = 0; b < B; ++b)
    for (int h = 0; h < Hkv; ++h)
      for (int64_t c = 0; c < nblk; ++c) {
        const uint16_t* lm = L + ((b * Hkv + h) * nblk + c) * d;
        double acc = 0.0, mass = 0.0;
        for (int g = 0; g < G; ++g)
          for (int j = 0; j < d; ++j) {
            double v = (double)bf16_to_f32(q[(b * Hq + h * G + g) * d + j]) * bf16_to_f32(lm[j]);
            acc += v;
            mass += fabs(v);
          }
        U[(b * Hkv + h) * nblk + c] = acc;
        if (l1) l1[(b * Hkv + h) * nblk + c] = mass;
      }
}
