// sd_gather_attend_noalloc: gather-attend for callers that cannot allocate device
// memory or hand the library a workspace: attention back-ends whose host framework
// owns every device allocation (a pool or custom allocator the library must not
// bypass), real-time loops that must not take allocator locks or let cudaMalloc
// synchronise the device, and code that runs where cudaMalloc may not be called.
// This entry point runs the same kernels as sd_gather_attend; when the split-n
// kernel (GPUs where the 16-CTA cluster kernel cannot be co-resident) or the
// many-row streaming kernel runs, its ticket and partial (m, l, o) results are
// kept in one file-scope device array instead of a caller workspace.  The cluster
// kernel needs no scratch and leaves the array alone.
//
// The array is a module global: every GPU that loads libsd holds its
// kNoallocScratchBytes until the process exits, and every call on a GPU shares
// that GPU's copy.  The size limit applies to every call, whichever kernel runs,
// so that a call accepted on one GPU is accepted on all.  The array keeps the
// previous call's contents: a call that runs either of those kernels first clears
// the per-row counters that must start at zero (with a memset on the caller's
// stream), and the kernel writes every partial before it reads it.  Such calls
// whose work overlaps on the GPU (different streams without ordering, or host
// threads) race on the array.  The array's device address is looked up once per
// device and kept for the process: after a device reset (cudaDeviceReset) it is
// stale, so the entry point must not be used on a device that has been reset.
#include <mutex>

#include "sd_internal.cuh"

namespace sd {

// Partials of at most 4 MiB: e.g. 8 KV heads x 1,152 selected tokens x 4 query
// heads (the 32k Hamming step) needs 0.3 MiB, 32 KV heads x 512 tokens x 4
// query heads (the 128k bit-plane step) 0.5 MiB.
constexpr size_t kNoallocScratchBytes = (size_t)4 << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
static void* g_scratch_ptr[kMaxDevices];
static std::mutex g_scratch_mu;

// Device address of this GPU's array.  In host code g_noalloc_scratch is a
// host-side stand-in, not a device address, so it is looked up once per device
// with that device current.
static int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SD_ERR_CUDA, "sd_gather_attend_noalloc: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(SD_ERR_UNSUPPORTED, "sd_gather_attend_noalloc: device %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return fail(SD_ERR_CUDA, "sd_gather_attend_noalloc: cudaGetSymbolAddress: %s",
                  cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SD_OK;
}

}  // namespace sd

using namespace sd;

extern "C" {

int sd_gather_attend_noalloc(const sd_shape* shape, const void* q, const void* K, const void* V,
                             const int32_t* idx, int64_t idx_stride, const int32_t* count,
                             int64_t max_count, float scale, float* out, float* lse,
                             void* stream) {
  // the same argument checks as sd_gather_attend, minus the workspace
  if (!shape) return fail(SD_ERR_INVALID_ARG, "sd_gather_attend_noalloc: shape is NULL");
  size_t need = sd_gather_attend_workspace_size(shape, max_count);
  if (need == 0 && max_count != 0)
    return sd_gather_attend(shape, q, K, V, idx, idx_stride, count, max_count, scale, out, lse,
                            nullptr, 0, stream);  // reports the shape error
  if (need > kNoallocScratchBytes)
    return fail(SD_ERR_UNSUPPORTED,
                "sd_gather_attend_noalloc: this problem needs %zu bytes of scratch, more than "
                "the %zu bytes the no-allocation entry point holds; use sd_gather_attend with "
                "a workspace", need, kNoallocScratchBytes);
  void* scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  return sd_gather_attend(shape, q, K, V, idx, idx_stride, count, max_count, scale, out, lse,
                          scratch, kNoallocScratchBytes, stream);
}

}  // extern "C"
