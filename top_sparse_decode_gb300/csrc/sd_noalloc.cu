// sd_gather_attend_noalloc: gather-attend for callers that cannot allocate device
// memory.  Some callers cannot call cudaMalloc or hand over a workspace: code that
// runs while a stream is being captured into a CUDA graph (cudaMalloc is not a
// stream operation and may synchronise the device), attention back-ends whose
// host framework owns every device allocation, and real-time loops that must not
// take allocator locks.  This entry point runs the same split-n kernels as
// sd_gather_attend, with their partial (m, l, o) results kept in one file-scope
// device array instead of a caller workspace.
//
// The array is a module global: every GPU that loads libsd holds its
// kNoallocScratchBytes until the process exits, and every call on a GPU shares
// that GPU's copy.  The array keeps the previous call's contents; every call
// first clears the per-row counters that must start at zero (with a memset on the
// caller's stream), and the kernels write every partial before they read it.  Calls whose work overlaps on the GPU (different streams without
// ordering, or host threads) race on the array.
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
