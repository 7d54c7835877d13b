// noalloc.cu -- grouped_mlp_fwd_noalloc: the grouped MLP forward for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point where they run
// the forward: code inside an allocator hook or an out-of-memory handler, a host runtime whose
// memory pool is owned elsewhere, or a plug-in whose host forbids allocations after start-up.
// For them this entry point takes its scratch memory (schedule, quantized activations and the
// quantized intermediate) from one file-scope device array of fixed size instead of a
// caller-provided workspace.  The caller still passes every input and output buffer.
//
// Facts a caller must know:
//   - The array is kNoAllocScratchBytes (64 MiB).  It lives in a module of its own, which CUDA
//     loads (lazy module loading, the default) on the first call made on a device; from then on
//     that device holds it until the process exits.  Problems whose workspace
//     (grouped_mlp_workspace_size) exceeds it are rejected with MXFP8_ERR_WORKSPACE before
//     anything is enqueued.
//   - The first call on a device is the set-up call: with that device current it looks up the
//     array's device address (cudaGetSymbolAddress), which makes CUDA load the array, and it sets
//     the kernels' launch attributes, which loads the library's kernels.  Both take device memory
//     inside the driver, so make that first call on each device while allocation is still
//     allowed, and before any stream capture.  Calls after it allocate nothing.
//   - Every call on a device shares the one array and leaves the last call's contents in it.
//     Nothing in it needs to start at zero: each call rewrites the schedule, the error word and
//     every scratch row it reads.  Calls that overlap on the GPU (different streams, or
//     different host threads without ordering) race on the array and corrupt each other.
//   - Device-side conditions (split_sizes that do not sum to R, a timed-out wait) are recorded
//     in the array's error word, which this entry point does not expose; callers that need to
//     read them use grouped_mlp_fwd with their own workspace.
//   - No call here calls cudaMalloc, cudaFree or an allocating library routine; after the
//     set-up call on a device, nothing on that device is allocated at all.
#include <cuda_runtime.h>

#include <mutex>

#include "mx_internal.h"
#include "mxfp8moe.h"

namespace mx {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device (looked up once per device).
void* scratch_address() {
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mx

using namespace mx;

extern "C" int grouped_mlp_fwd_noalloc(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E,
                                       const int32_t* split_sizes, const float* gates, const uint8_t* w1_q,
                                       const uint8_t* w1_sf, const uint8_t* w2_q, const uint8_t* w2_sf, void* y,
                                       void* stream) {
  if (R < 0 || E < 1 || E > 1024 || H <= 0 || F <= 0) return MXFP8_ERR_INVALID_ARG;
  if (H % 128 != 0 || F % 128 != 0) return MXFP8_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(E) * 2 * F > INT32_MAX || static_cast<int64_t>(E) * H > INT32_MAX)
    return MXFP8_ERR_UNSUPPORTED;
  const void* ptrs[] = {x_sorted, split_sizes, w1_q, w1_sf, w2_q, w2_sf, y};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return MXFP8_ERR_INVALID_ARG;
  if (gates != nullptr && !aligned16(gates)) return MXFP8_ERR_INVALID_ARG;
  WsLayout L;
  if (!ws_layout(R, H, F, E, &L)) return MXFP8_ERR_UNSUPPORTED;
  if (L.total > kNoAllocScratchBytes) return MXFP8_ERR_WORKSPACE;
  void* scratch = scratch_address();
  if (scratch == nullptr) return MXFP8_ERR_CUDA;
  return launch_grouped_mlp(x_sorted, R, H, F, E, split_sizes, gates, w1_q, w1_sf, w2_q, w2_sf, y, scratch, L,
                            static_cast<cudaStream_t>(stream), nullptr);
}
