/*
 * Seeded synthetic input generator for the sparse-decode workloads.
 *
 * This file only produces random inputs (keys, values, queries, encoder weights,
 * calibration variances).  It holds none of the sparse-decode arithmetic: no
 * signature, quantiser, score, selection or attention step.  Both the CUDA
 * library's tests and the CPU oracle consume what it writes.
 *
 * Random numbers are counter-based, so every element depends only on
 * (seed, tensor id, element index) and never on the thread count:
 *   u64(seed, tid, i) = mix64(key(seed, tid) + (i + 1) * GAMMA)
 *   key(seed, tid)    = mix64(seed ^ mix64(tid + KEY_SALT))
 * with mix64 the SplitMix64 output finaliser (Steele, Lea, Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014).  A uniform double is
 * the top 53 bits times 2^-53.  A standard normal is Box-Muller on the two
 * uniforms with counters 2i and 2i+1 (cosine branch only).
 *
 * Floating point values are rounded double -> float (RN) -> bfloat16 (RN-even).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL
#define KEY_SALT 0x632BE59BD9B4E019ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tid) {
  return mix64(seed ^ mix64(tid + KEY_SALT));
}

static inline double uniform_at(uint64_t key, uint64_t i) {
  uint64_t u = mix64(key + (i + 1) * GAMMA);
  return (double)(u >> 11) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t key, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  double u1 = uniform_at(key, 2 * i);
  double u2 = uniform_at(key, 2 * i + 1);
  double r = sqrt(-2.0 * log(1.0 - u1)); /* 1-u1 is in (0, 1] */
  return r * cos(two_pi * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0u; /* NaN */
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* out[i] = U[0,1)(seed, tid, start + i) */
void synth_uniform(uint64_t seed, uint64_t tid, int64_t start, int64_t count, double* out) {
  uint64_t key = stream_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) out[i] = uniform_at(key, (uint64_t)(start + i));
}

/* out[i] = N(0,1)(seed, tid, start + i) */
void synth_normal_f64(uint64_t seed, uint64_t tid, int64_t start, int64_t count, double* out) {
  uint64_t key = stream_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) out[i] = normal_at(key, (uint64_t)(start + i));
}

/* out[i] = (float)(std * N(0,1)(seed, tid, i)) */
void synth_normal_f32(uint64_t seed, uint64_t tid, int64_t count, double std, float* out) {
  uint64_t key = stream_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) out[i] = (float)(std * normal_at(key, (uint64_t)i));
}

/*
 * Row-major bf16 fill of nrows x ncols normals.  Row r uses the per-column
 * standard deviations sigma[((r / rows_per_sigma) % nsig) * ncols + c]; sigma may
 * be NULL for unit variance.  Element (r, c) draws counter r * ncols + c.
 */
void synth_fill_normal_bf16(uint64_t seed, uint64_t tid, int64_t nrows, int64_t ncols,
                            const double* sigma, int64_t rows_per_sigma, int64_t nsig,
                            uint16_t* out) {
  uint64_t key = stream_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; ++r) {
    const double* srow = sigma ? sigma + ((r / rows_per_sigma) % nsig) * ncols : 0;
    for (int64_t c = 0; c < ncols; ++c) {
      double x = normal_at(key, (uint64_t)(r * ncols + c));
      if (srow) x *= srow[c];
      out[r * ncols + c] = f32_to_bf16_rne((float)x);
    }
  }
}

/* bf16 rounding of doubles: double -> float (RN) -> bf16 (RN-even). */
void synth_f64_to_bf16(const double* in, int64_t count, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) out[i] = f32_to_bf16_rne((float)in[i]);
}
