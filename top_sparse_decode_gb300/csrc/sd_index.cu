// Key-side index builds (KV-write path) and the per-step query map.
//
//  * signatures  -- HashAttention: Semantic Sparsity for Faster Inference, 2.2
//                   (phi(x) = ReLU(sign(F(x))), 32-bit codes cached at KV write)
//  * bit planes  -- Fathom: Per-Query Read Depth ..., "store as bit planes per
//                   channel" (4-bit code, fp16 scale per channel per 64 tokens)
//  * min/max     -- OasisKV: Scaling In-Decode KV Cache Beyond HBM ...,
//                   prerequisites, Quest-style per-block per-channel summaries
#include <cuda_fp16.h>

#include <cuda_bf16.h>

#include "sd_internal.cuh"

namespace sd {

// =====================================================================================
// Signatures.  Every dot product is the canonical fp32 chain
//   acc = +0; for j ascending: acc = fma(w_j, x_j, acc); acc = acc + bias
// so that the code bits do not depend on the machine.  No tensor cores here:
// their accumulation order is unspecified.
// =====================================================================================

// Keys: one thread per key row.  Weights staged in shared memory, transposed so
// that the 32 weights a thread needs for one input element are contiguous and
// read as warp-wide broadcasts.
template <int HID>
__global__ void __launch_bounds__(128)
sig_build_kernel(const uint16_t* __restrict__ K, int64_t n, int64_t ncap, int64_t t0,
                 int64_t rows, const float* __restrict__ W1, const float* __restrict__ b1,
                 const float* __restrict__ W2, const float* __restrict__ b2,
                 uint32_t* __restrict__ sig) {
  constexpr int H1 = HID ? HID : 32;  // width of the first layer
  extern __shared__ __align__(16) float smem[];
  float* W1T = smem;                   // [kD][H1]
  float* B1 = W1T + kD * H1;           // [H1]
  float* W2T = B1 + H1;                // [HID][32]
  float* B2 = W2T + HID * 32;          // [32]
  for (int e = threadIdx.x; e < kD * H1; e += blockDim.x) {
    int u = e / kD, j = e % kD;
    W1T[j * H1 + u] = W1[e];
  }
  for (int e = threadIdx.x; e < H1; e += blockDim.x) B1[e] = b1 ? b1[e] : 0.0f;
  if (HID) {
    for (int e = threadIdx.x; e < 32 * HID; e += blockDim.x) {
      int o = e / HID, u = e % HID;
      W2T[u * 32 + o] = W2[e];
    }
    for (int e = threadIdx.x; e < 32; e += blockDim.x) B2[e] = b2 ? b2[e] : 0.0f;
  }
  __syncthreads();
  int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= rows) return;
  const int64_t cnt = n - t0;  // tokens [t0, n) of every row
  const int64_t bh = r / cnt, i = t0 + (r - bh * cnt);
  const uint4* xrow = reinterpret_cast<const uint4*>(K + (bh * ncap + i) * kD);

  float out[32];
#pragma unroll
  for (int o = 0; o < 32; ++o) out[o] = 0.0f;

  constexpr int NCHUNK = HID ? HID / 32 : 1;
#pragma unroll 1
  for (int uc = 0; uc < NCHUNK; ++uc) {
    float acc[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) acc[u] = 0.0f;
#pragma unroll 1
    for (int jc = 0; jc < kD; jc += 8) {
      uint4 raw = __ldg(xrow + jc / 8);
      uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        float x = (jj & 1) ? bf16_hi(w4[jj / 2]) : bf16_lo(w4[jj / 2]);
        const float4* wrow = reinterpret_cast<const float4*>(W1T + (jc + jj) * H1 + uc * 32);
#pragma unroll
        for (int u4 = 0; u4 < 8; ++u4) {
          float4 w = wrow[u4];
          acc[4 * u4 + 0] = __fmaf_rn(w.x, x, acc[4 * u4 + 0]);
          acc[4 * u4 + 1] = __fmaf_rn(w.y, x, acc[4 * u4 + 1]);
          acc[4 * u4 + 2] = __fmaf_rn(w.z, x, acc[4 * u4 + 2]);
          acc[4 * u4 + 3] = __fmaf_rn(w.w, x, acc[4 * u4 + 3]);
        }
      }
    }
    if (HID == 0) {
#pragma unroll
      for (int o = 0; o < 32; ++o) out[o] = __fadd_rn(acc[o], B1[o]);
    } else {
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        float h = __fadd_rn(acc[u], B1[uc * 32 + u]);
        h = h > 0.0f ? h : 0.0f;
        const float4* w2 = reinterpret_cast<const float4*>(W2T + (uc * 32 + u) * 32);
#pragma unroll
        for (int o4 = 0; o4 < 8; ++o4) {
          float4 w = w2[o4];
          out[4 * o4 + 0] = __fmaf_rn(w.x, h, out[4 * o4 + 0]);
          out[4 * o4 + 1] = __fmaf_rn(w.y, h, out[4 * o4 + 1]);
          out[4 * o4 + 2] = __fmaf_rn(w.z, h, out[4 * o4 + 2]);
          out[4 * o4 + 3] = __fmaf_rn(w.w, h, out[4 * o4 + 3]);
        }
      }
    }
  }
  uint32_t word = 0;
#pragma unroll
  for (int o = 0; o < 32; ++o) {
    float v = HID ? __fadd_rn(out[o], B2[o]) : out[o];
    word |= (v > 0.0f ? 1u : 0u) << o;
  }
  sig[bh * ncap + i] = word;
}

// Queries: few rows, so parallelise over the units instead.  A CTA encodes up
// to kQRows rows; thread u runs unit u's chain for each of them (independent
// chains give the FMA pipe some parallelism).  Same chains, same bits.
constexpr int kQRows = 8;

template <int HID>
__global__ void __launch_bounds__(128)
encode_query_kernel(const uint16_t* __restrict__ q, int rows, const float* __restrict__ W1,
                    const float* __restrict__ b1, const float* __restrict__ W2,
                    const float* __restrict__ b2, uint32_t* __restrict__ qsig) {
  constexpr int H1 = HID ? HID : 32;
  constexpr int P1 = kD + 1;      // padded row pitch of W1: conflict-free column walks
  constexpr int P2 = HID + 1;
  extern __shared__ __align__(16) float smem[];
  float* Ws1 = smem;                       // [H1][P1]
  float* Ws2 = Ws1 + H1 * P1;              // [32][P2]
  float* xs = Ws2 + (HID ? 32 * P2 : 0);   // [kQRows][kD]
  float* hs = xs + kQRows * kD;            // [kQRows][HID]
  int r0 = blockIdx.x * kQRows;
  int nr = min(kQRows, rows - r0);
  for (int e = threadIdx.x; e < H1 * kD; e += blockDim.x) Ws1[(e / kD) * P1 + e % kD] = W1[e];
  if (HID)
    for (int e = threadIdx.x; e < 32 * HID; e += blockDim.x) Ws2[(e / HID) * P2 + e % HID] = W2[e];
  for (int e = threadIdx.x; e < kQRows * kD; e += blockDim.x) {
    int rr = e / kD;
    xs[e] = rr < nr ? bf16_to_f32(q[(int64_t)(r0 + rr) * kD + e % kD]) : 0.0f;
  }
  __syncthreads();
  float acc[kQRows];
  if (threadIdx.x < H1) {
    int u = threadIdx.x;
#pragma unroll
    for (int rr = 0; rr < kQRows; ++rr) acc[rr] = 0.0f;
#pragma unroll 4
    for (int j = 0; j < kD; ++j) {
      float w = Ws1[u * P1 + j];
#pragma unroll
      for (int rr = 0; rr < kQRows; ++rr) acc[rr] = __fmaf_rn(w, xs[rr * kD + j], acc[rr]);
    }
    float bias = b1 ? b1[u] : 0.0f;
#pragma unroll
    for (int rr = 0; rr < kQRows; ++rr) {
      float v = __fadd_rn(acc[rr], bias);
      if (HID) hs[rr * HID + u] = v > 0.0f ? v : 0.0f;
      else acc[rr] = v;
    }
  }
  if (HID) {
    __syncthreads();
    if (threadIdx.x < 32) {
      int o = threadIdx.x;
#pragma unroll
      for (int rr = 0; rr < kQRows; ++rr) acc[rr] = 0.0f;
#pragma unroll 4
      for (int u = 0; u < HID; ++u) {
        float w = Ws2[o * P2 + u];
#pragma unroll
        for (int rr = 0; rr < kQRows; ++rr) acc[rr] = __fmaf_rn(w, hs[rr * HID + u], acc[rr]);
      }
      float bias = b2 ? b2[o] : 0.0f;
#pragma unroll
      for (int rr = 0; rr < kQRows; ++rr) acc[rr] = __fadd_rn(acc[rr], bias);
    }
  }
  if (threadIdx.x < 32) {
#pragma unroll
    for (int rr = 0; rr < kQRows; ++rr) {
      uint32_t word = __ballot_sync(0xFFFFFFFFu, acc[rr] > 0.0f);
      if (threadIdx.x == 0 && rr < nr) qsig[r0 + rr] = word;
    }
  }
}

template <int HID>
static int sig_build_t(const Dims& s, const uint16_t* K, const sd_encoder& e, uint32_t* sig,
                       int64_t t0, cudaStream_t st) {
  constexpr int H1 = HID ? HID : 32;
  size_t smem = sizeof(float) * (kD * H1 + H1 + HID * 32 + 32);
  auto kern = sig_build_kernel<HID>;
  if (int rc_ = set_smem_limit((const void*)kern, smem, "sig_build: smem attribute")) return rc_;
  int64_t rows = (int64_t)s.B * s.Hkv * (s.n - t0);
  unsigned grid = (unsigned)((rows + 127) / 128);
  kern<<<grid, 128, smem, st>>>(K, s.n, s.ncap, t0, rows, e.W1, e.b1, e.W2, e.b2, sig);
  note_launches(1);
  return check_launch("sig_build");
}

template <int HID>
static int encode_query_t(const Dims& s, const uint16_t* q, const sd_encoder& e, uint32_t* qsig,
                          cudaStream_t st) {
  constexpr int H1 = HID ? HID : 32;
  size_t smem = sizeof(float) * (H1 * (kD + 1) + (HID ? 32 * (HID + 1) : 0) + kQRows * kD +
                                 kQRows * HID);
  auto kern = encode_query_kernel<HID>;
  if (int rc_ = set_smem_limit((const void*)kern, smem, "encode_query: smem attribute")) return rc_;
  int rows = s.B * s.Hq;
  kern<<<(rows + kQRows - 1) / kQRows, 128, smem, st>>>(q, rows, e.W1, e.b1, e.W2, e.b2, qsig);
  note_launches(1);
  return check_launch("encode_query");
}

int launch_sig_build(const Dims& s, const uint16_t* K, const sd_encoder& e, uint32_t* sig,
                     cudaStream_t st, int64_t t0) {
  switch (e.hidden) {
    case 0: return sig_build_t<0>(s, K, e, sig, t0, st);
    case 32: return sig_build_t<32>(s, K, e, sig, t0, st);
    case 64: return sig_build_t<64>(s, K, e, sig, t0, st);
    default: return sig_build_t<128>(s, K, e, sig, t0, st);
  }
}

int launch_encode_query(const Dims& s, const uint16_t* q, const sd_encoder& e, uint32_t* qsig,
                        cudaStream_t st) {
  switch (e.hidden) {
    case 0: return encode_query_t<0>(s, q, e, qsig, st);
    case 32: return encode_query_t<32>(s, q, e, qsig, st);
    case 64: return encode_query_t<64>(s, q, e, qsig, st);
    default: return encode_query_t<128>(s, q, e, qsig, st);
  }
}

// =====================================================================================
// Bit planes.  Per (channel, 64-token block): s = f16_rn(absmax / 7) (1 if 0),
// code = clamp(rint(k / s) + 8, 0, 15) with an IEEE fp32 divide; plane p holds bit
// (3 - p).  A CTA covers 1024 tokens (16 blocks) of one (sequence, KV head) so
// that each (channel, plane) row it writes is 128 contiguous bytes.  A last block
// holding fewer than 64 tokens takes its scale over them (rows past n are staged
// as zeros, which leave absmax unchanged) and gets zero bits past n.  The blocks
// from tok_begin (a multiple of 64) on are written, so an append rebuilds only
// the block it extends and the ones after it.
// =====================================================================================
constexpr int kPbTile = 1024;
constexpr int kPbPitch = kD + 8;  // bf16 row pitch of the staged block

__global__ void __launch_bounds__(256)
plane_build_kernel(const uint16_t* __restrict__ K, int64_t n, int64_t ncap, int64_t tok_begin,
                   uint32_t* __restrict__ planes, uint16_t* __restrict__ scales) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw);                   // [64][kPbPitch]
  uint32_t* ws = reinterpret_cast<uint32_t*>(xs + 64 * kPbPitch);         // [kD][4][32]
  uint16_t* ss = reinterpret_cast<uint16_t*>(ws + kD * 4 * 32);           // [kD][16]
  const int64_t bh = blockIdx.y;
  const int64_t tok0 = tok_begin + (int64_t)blockIdx.x * kPbTile;
  const int nblk = (int)imin64(kPbTile / 64, (n - tok0 + 63) / 64);
  const uint16_t* Kb = K + (bh * ncap + tok0) * kD;
  const int j = threadIdx.x & (kD - 1), half = threadIdx.x >> 7;

  for (int blk = 0; blk < nblk; ++blk) {
    // stage 64 rows x 256 B
    for (int e = threadIdx.x; e < 64 * 16; e += 256) {
      int row = e >> 4, seg = e & 15;
      const int64_t t = (int64_t)blk * 64 + row;  // token tok0 + t
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (tok0 + t < n) v = __ldg(reinterpret_cast<const uint4*>(Kb + t * kD) + seg);
      *reinterpret_cast<uint4*>(xs + row * kPbPitch + seg * 8) = v;
    }
    __syncthreads();
    float amax = 0.0f;
#pragma unroll 8
    for (int r = 0; r < 64; ++r) amax = fmaxf(amax, fabsf(bf16_to_f32(xs[r * kPbPitch + j])));
    __half sh = __float2half_rn(__fdiv_rn(amax, 7.0f));
    uint16_t s16 = __half_as_ushort(sh);
    if ((s16 & 0x7FFFu) == 0) s16 = 0x3C00u;
    float s = __half2float(__ushort_as_half(s16));
    uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
#pragma unroll 4
    for (int r = 0; r < 32; ++r) {
      float k = bf16_to_f32(xs[(half * 32 + r) * kPbPitch + j]);
      float rq = rintf(__fdiv_rn(k, s));
      int code = rq <= -8.0f ? 0 : (rq >= 7.0f ? 15 : (int)rq + 8);
      w0 |= (uint32_t)((code >> 3) & 1) << r;
      w1 |= (uint32_t)((code >> 2) & 1) << r;
      w2 |= (uint32_t)((code >> 1) & 1) << r;
      w3 |= (uint32_t)(code & 1) << r;
    }
    // positions past n hold no key: their bits are 0
    const int64_t held = n - (tok0 + (int64_t)blk * 64 + half * 32);
    const uint32_t keep = held >= 32 ? 0xFFFFFFFFu : (held <= 0 ? 0u : (1u << held) - 1u);
    w0 &= keep;
    w1 &= keep;
    w2 &= keep;
    w3 &= keep;
    uint32_t* wj = ws + j * 128 + blk * 2 + half;
    wj[0] = w0;
    wj[32] = w1;
    wj[64] = w2;
    wj[96] = w3;
    if (half == 0) ss[j * 16 + blk] = s16;
    __syncthreads();
  }
  // write each (channel, plane) row: 2 * nblk words
  const int nw = nblk * 2;
  const int64_t wstride = ncap / 32;
  for (int e = threadIdx.x; e < kD * 4 * 32; e += 256) {
    int row = e >> 5, w = e & 31;
    if (w < nw) planes[(bh * kD * 4 + row) * wstride + tok0 / 32 + w] = ws[row * 32 + w];
  }
  const int64_t sstride = ncap / 64;
  for (int e = threadIdx.x; e < kD * 16; e += 256) {
    int jj = e >> 4, b = e & 15;
    if (b < nblk) scales[(bh * kD + jj) * sstride + tok0 / 64 + b] = ss[jj * 16 + b];
  }
}

int launch_plane_build(const Dims& s, const uint16_t* K, uint32_t* planes, uint16_t* scales,
                       cudaStream_t st, int64_t t0) {
  size_t smem = 64 * kPbPitch * 2 + kD * 4 * 32 * 4 + kD * 16 * 2;
  if (int rc_ = set_smem_limit((const void*)plane_build_kernel, smem, "plane_build: smem attribute")) return rc_;
  const int64_t tb = t0 / 64 * 64;  // the block holding token t0 starts the rebuild
  dim3 grid((unsigned)((s.n - tb + kPbTile - 1) / kPbTile), (unsigned)(s.B * s.Hkv));
  plane_build_kernel<<<grid, 256, smem, st>>>(K, s.n, s.ncap, tb, planes, scales);
  note_launches(1);
  return check_launch("plane_build");
}

// =====================================================================================
// Min/max summaries.  One warp per 16-token block, lane l owns channels 4l..4l+3.
// -0.0 orders below +0.0 (total order on bf16 patterns) so min/max are unique.
// =====================================================================================
__device__ __forceinline__ uint32_t ord16(uint32_t x) {
  return (x & 0x8000u) ? (~x & 0xFFFFu) : (x | 0x8000u);
}
__device__ __forceinline__ uint32_t unord16(uint32_t k) {
  return (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
}

__global__ void __launch_bounds__(256)
minmax_build_kernel(const uint16_t* __restrict__ K, int64_t n, int64_t ncap, int64_t c0,
                    uint16_t* __restrict__ summ) {
  const int64_t bh = blockIdx.y;
  const int64_t c = c0 + (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t nblk_valid = (n + 15) / 16, nblk_cap = (ncap + 15) / 16;
  if (c >= nblk_valid) return;
  const int64_t t0 = c * 16, t1 = imin64(t0 + 16, n);
  const uint16_t* Kb = K + bh * ncap * kD + lane * 4;
  uint32_t mn[4], mx[4];
  {
    uint2 v = __ldg(reinterpret_cast<const uint2*>(Kb + t0 * kD));
    uint32_t e[4] = {v.x & 0xFFFFu, v.x >> 16, v.y & 0xFFFFu, v.y >> 16};
#pragma unroll
    for (int k = 0; k < 4; ++k) mn[k] = mx[k] = ord16(e[k]);
  }
  for (int64_t t = t0 + 1; t < t1; ++t) {
    uint2 v = __ldg(reinterpret_cast<const uint2*>(Kb + t * kD));
    uint32_t e[4] = {v.x & 0xFFFFu, v.x >> 16, v.y & 0xFFFFu, v.y >> 16};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t o = ord16(e[k]);
      mn[k] = min(mn[k], o);
      mx[k] = max(mx[k], o);
    }
  }
  uint16_t* out = summ + (bh * nblk_cap + c) * 2 * kD + lane * 4;
  uint2 lo, hi;
  lo.x = unord16(mn[0]) | (unord16(mn[1]) << 16);
  lo.y = unord16(mn[2]) | (unord16(mn[3]) << 16);
  hi.x = unord16(mx[0]) | (unord16(mx[1]) << 16);
  hi.y = unord16(mx[2]) | (unord16(mx[3]) << 16);
  *reinterpret_cast<uint2*>(out) = lo;
  *reinterpret_cast<uint2*>(out + kD) = hi;
}

int launch_minmax_build(const Dims& s, const uint16_t* K, uint16_t* summ, cudaStream_t st,
                        int64_t t0) {
  const int64_t nblk = (s.n + 15) / 16, c0 = t0 / 16;  // blocks [c0, nblk) are rebuilt
  dim3 grid((unsigned)((nblk - c0 + 7) / 8), (unsigned)(s.B * s.Hkv));
  minmax_build_kernel<<<grid, 256, 0, st>>>(K, s.n, s.ncap, c0, summ);
  note_launches(1);
  return check_launch("minmax_build");
}

// =====================================================================================
// Block landmarks (the Fathom page's 8-token block landmark scan): per block of 8
// tokens the bf16 rounding (nearest even) of the fp32 mean of its held keys, summed
// in token order.  One warp per block, lane l owns channels 4l..4l+3.
// =====================================================================================
__global__ void __launch_bounds__(256)
landmark_build_kernel(const uint16_t* __restrict__ K, int64_t n, int64_t ncap, int64_t c0,
                      uint16_t* __restrict__ L) {
  const int64_t bh = blockIdx.y;
  const int64_t c = c0 + (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t nblk_valid = (n + kLmBlock - 1) / kLmBlock;
  const int64_t nblk_cap = (ncap + kLmBlock - 1) / kLmBlock;
  if (c >= nblk_valid) return;
  const int64_t t0 = c * kLmBlock, t1 = imin64(t0 + kLmBlock, n);
  const uint16_t* Kb = K + bh * ncap * kD + lane * 4;
  float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int64_t t = t0; t < t1; ++t) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(Kb + t * kD));
    s[0] = __fadd_rn(s[0], bf16_lo(v.x));
    s[1] = __fadd_rn(s[1], bf16_hi(v.x));
    s[2] = __fadd_rn(s[2], bf16_lo(v.y));
    s[3] = __fadd_rn(s[3], bf16_hi(v.y));
  }
  const float cnt = (float)(t1 - t0);
  uint32_t h[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    h[k] = __bfloat16_as_ushort(__float2bfloat16_rn(__fdiv_rn(s[k], cnt)));
  uint2 out;
  out.x = h[0] | (h[1] << 16);
  out.y = h[2] | (h[3] << 16);
  *reinterpret_cast<uint2*>(L + (bh * nblk_cap + c) * kD + lane * 4) = out;
}

int launch_landmark_build(const Dims& s, const uint16_t* K, uint16_t* L, cudaStream_t st,
                          int64_t t0) {
  const int64_t nblk = (s.n + kLmBlock - 1) / kLmBlock, c0 = t0 / kLmBlock;
  dim3 grid((unsigned)((nblk - c0 + 7) / 8), (unsigned)(s.B * s.Hkv));
  landmark_build_kernel<<<grid, 256, 0, st>>>(K, s.n, s.ncap, c0, L);
  note_launches(1);
  return check_launch("landmark_build");
}

}  // namespace sd
