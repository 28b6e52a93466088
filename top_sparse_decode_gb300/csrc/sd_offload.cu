// Planned-prefix gather from pinned host memory (Fathom: Per-Query Read Depth ...,
// "host planes are channel-contiguous": one gather copies the active channels'
// prefixes into HBM before the scan; OasisKV: ..., method details: a UVA gather
// kernel reads pinned CPU memory directly, on its own stream).
//
// In the channel-major layout the first t planes of channel j are one
// contiguous run of t * n_cap / 8 bytes, so each active (sequence, KV head,
// channel) is a single linear copy.  Device loads of the mapped host buffer go
// over the host link (PCIe or NVLink-C2C); many 16-byte loads are kept in
// flight per thread to cover the link latency.
#include "sd_internal.cuh"

namespace sd {

constexpr int kOgThreads = 256;
constexpr int kOgUnroll = 8;
constexpr int64_t kOgBytesPerCta = (int64_t)kOgThreads * 16 * kOgUnroll;  // 32 KB

__global__ void __launch_bounds__(kOgThreads)
offload_gather_kernel(const uint32_t* __restrict__ hp, const uint16_t* __restrict__ hs,
                      const uint8_t* __restrict__ plan, int64_t ncap,
                      uint32_t* __restrict__ dp, uint16_t* __restrict__ ds) {
  const int64_t r = blockIdx.x;  // (sequence * hkv + head) * d + channel
  const int t = min((int)plan[r], 4);  // a plan holds 0..4 bits per channel
  if (t == 0) return;
  const int64_t plane_bytes = ncap / 8;
  const int64_t bytes = t * plane_bytes;
  const int64_t off0 = (int64_t)blockIdx.y * kOgBytesPerCta;
  const uint8_t* src = reinterpret_cast<const uint8_t*>(hp) + r * 4 * plane_bytes;
  uint8_t* dst = reinterpret_cast<uint8_t*>(dp) + r * 4 * plane_bytes;
  if (off0 < bytes) {
    const int64_t end = imin64(off0 + kOgBytesPerCta, bytes);
    const int64_t nvec = (end - off0) / 16;  // whole 16-byte vectors
    uint4 buf[kOgUnroll];
#pragma unroll
    for (int u = 0; u < kOgUnroll; ++u) {
      int64_t v = threadIdx.x + (int64_t)u * kOgThreads;
      if (v < nvec) buf[u] = *reinterpret_cast<const uint4*>(src + off0 + v * 16);
    }
#pragma unroll
    for (int u = 0; u < kOgUnroll; ++u) {
      int64_t v = threadIdx.x + (int64_t)u * kOgThreads;
      if (v < nvec) *reinterpret_cast<uint4*>(dst + off0 + v * 16) = buf[u];
    }
    // an 8-byte remainder (t * n_cap / 8 is a multiple of 8)
    const int64_t rem = (end - off0) - nvec * 16;
    if (rem && threadIdx.x == 0) {
      const int64_t o = off0 + nvec * 16;
      *reinterpret_cast<uint2*>(dst + o) = *reinterpret_cast<const uint2*>(src + o);
    }
  }
  if (blockIdx.y == 0) {  // the channel's scales: n_cap / 64 fp16 values
    const int64_t ns = ncap / 64;
    for (int64_t i = threadIdx.x; i < ns; i += kOgThreads) ds[r * ns + i] = hs[r * ns + i];
  }
}

int launch_offload_gather(const Dims& s, const uint32_t* host_planes, const uint16_t* host_scales,
                          const uint8_t* plan, uint32_t* dev_planes, uint16_t* dev_scales,
                          cudaStream_t st) {
  const int64_t max_bytes = 4 * (s.ncap / 8);
  dim3 grid((unsigned)((int64_t)s.B * s.Hkv * kD),
            (unsigned)((max_bytes + kOgBytesPerCta - 1) / kOgBytesPerCta));
  offload_gather_kernel<<<grid, kOgThreads, 0, st>>>(host_planes, host_scales, plan, s.ncap,
                                                     dev_planes, dev_scales);
  note_launches(1);
  return check_launch("offload_gather");
}

}  // namespace sd
