// vr_verify_select_noalloc: the candidate-pool select with its scratch
// compiled into the library instead of taken from a caller's workspace.
//
// Who needs it: callers that cannot hand the library device memory of its
// own.  Examples are a plugin whose host application owns every device
// allocation through its own pool and offers no hook to borrow from it, or a
// process that must not grow its device footprint after start-up.  Such a
// caller still owns the inputs and outputs; only the select's intermediate
// candidates need a home, and here they live in one fixed array that every
// GPU loading this library reserves until the process exits.
//
// Rules of use (also stated in include/verifyrow.h):
//   * rows <= VR_NOALLOC_SELECT_MAX_ROWS; any vocab (the select never splits a
//     row into more than 64 segments of candidates);
//   * the array is shared by every call on a device and keeps the last
//     call's contents; calls that overlap on the GPU (two streams, or two
//     host threads) race on it and must be serialised by the caller;
//   * the row counters that pick each row's merging CTA must start at zero;
//     every call clears them (an asynchronous memset on the caller's stream)
//     before its kernel; the candidate slots are written before they are
//     read;
//   * the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress with that device current) and remembers it, so
//     make that first call before any stream capture on that device.
#include <mutex>

#include "vr_common.cuh"
#include "vr_kernels.h"

namespace vr {
namespace {

constexpr int kNoallocMaxSegments = 64;
constexpr size_t kNoallocSlots =
    static_cast<size_t>(VR_NOALLOC_SELECT_MAX_ROWS) * kNoallocMaxSegments * kPool;
constexpr size_t kCounterSlots = 32;   // 256 bytes holding the 32 uint32 row counters

// the row counters, then 32 rows x 64 segments x 64 candidates x 8 bytes:
// 1 MiB + 256 B
static __device__ __align__(256) uint64_t g_select_scratch[kCounterSlots + kNoallocSlots];

std::mutex g_mutex;
uint64_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device); nullptr on failure.
uint64_t* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_ptr[dev] = static_cast<uint64_t*>(p);
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace vr

extern "C" int vr_verify_select_noalloc(const float* logits, int rows, int vocab,
                                        int32_t* pool_ids, float* pool_vals, void* stream) {
  if (!logits || !pool_ids || !pool_vals || rows < 1 || vocab < 1) return VR_ERR_ARG;
  if (rows > VR_NOALLOC_SELECT_MAX_ROWS) return VR_ERR_UNSUPPORTED;
  if (static_cast<size_t>(rows) * vr::select_segments(vocab) * vr::kPool > vr::kNoallocSlots)
    return VR_ERR_UNSUPPORTED;
  uint64_t* scratch = vr::scratch_for_current_device();
  if (!scratch) return VR_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* counters = reinterpret_cast<uint32_t*>(scratch);
  if (cudaMemsetAsync(counters, 0, VR_NOALLOC_SELECT_MAX_ROWS * sizeof(uint32_t), s) != cudaSuccess)
    return VR_ERR_CUDA;
  return vr::launch_sample(logits, rows, vocab, scratch + vr::kCounterSlots, counters, nullptr,
                           nullptr, pool_ids, pool_vals, nullptr, nullptr, nullptr, s);
}
