// awq_gemv_noalloc: the decode GEMV for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: a plugin loaded into an
// inference runtime that owns all device memory and hands the plugin no allocator,
// or a latency-critical serving loop that forbids allocation after start-up
// (cudaMalloc may synchronize the device and stall every other stream).  They can
// still pass their inputs and outputs, but not the split-K workspace that awq_gemv
// takes.  This entry point keeps that scratch in a fixed array that lives inside the
// library image on every GPU that loads it (kNoAllocScratchBytes, held until the
// process exits) and otherwise runs exactly the awq_gemv kernel.
//
// Host code must not pass the array's name to a kernel: in host code the name is a
// host-side stand-in, not a device address.  The device address is resolved once
// per device with cudaGetSymbolAddress (with that device current) and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/awq.h"
#include "awq_internal.h"

namespace awq {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;  // 8 MiB per device
constexpr int kMaxDevicesNoAlloc = 64;

static __device__ __align__(256) unsigned char g_gemv_scratch[kNoAllocScratchBytes];

// Device address of g_gemv_scratch on the current device (resolved on first use per device).
void* scratch_address() {
  static void* ptrs[kMaxDevicesNoAlloc] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesNoAlloc) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_gemv_scratch) != cudaSuccess || p == nullptr) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace awq

using namespace awq;

extern "C" awq_status awq_gemv_noalloc(const uint16_t* x, const int32_t* qweight, const int32_t* qzeros,
                                       const uint16_t* scales, uint16_t* y, int64_t M, int64_t K, int64_t N,
                                       int32_t group_size, int32_t split_k, awq_stream_t stream) {
  if (M < 0 || M > kGemvMaxM || K <= 0 || K % kGroup != 0 || K > ((int64_t)1 << 30) || N <= 0 || N % 32 != 0 ||
      N > ((int64_t)1 << 30) || group_size != kGroup || split_k < 0)
    return AWQ_EINVAL;
  if (M == 0) return AWQ_OK;
  if (!x || !qweight || !scales || !y) return AWQ_ENULL;
  if (!aligned16(x) || !aligned16(qweight) || !aligned16(scales) || !aligned16(y) || (qzeros && !aligned16(qzeros)))
    return AWQ_EALIGN;

  // Choose the K split; the automatic choice shrinks until its scratch fits the fixed array,
  // an explicit split_k that needs more scratch than the array holds is rejected.
  GemvPlan plan = gemv_plan(M, K, N, split_k);
  if (gemv_workspace_bytes(plan, M, N) > kNoAllocScratchBytes) {
    if (split_k > 0) return AWQ_EWORKSPACE;
    // split 1 (one CTA per tile) needs no scratch, so the search always ends
    int s = plan.split;
    while (gemv_workspace_bytes(plan, M, N) > kNoAllocScratchBytes) plan = gemv_plan(M, K, N, s > 1 ? --s : 1);
  }

  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return AWQ_ECUDA;
  if (major != 10 || minor != 3) return AWQ_EARCH;

  // The split-K tickets occupy the first kCounterBytes of the array, one per tile; the partials follow.
  if (plan.maxc > 1 && plan.tiles > kMaxCounters) return AWQ_EINVAL;
  // The device error word is another file-scope __device__ variable of the library, so reporting a
  // timed-out wait (awq_last_device_error) allocates nothing either.
  int* err = device_error_ptr();
  if (!err) return AWQ_ECUDA;

  void* scratch = nullptr;
  if (gemv_workspace_bytes(plan, M, N) > 0) {
    scratch = scratch_address();
    if (!scratch) return AWQ_ECUDA;
    // The split-K tickets at the start of the array must read zero when the kernel starts; the
    // array keeps whatever the previous call left, so clear them on this call's stream.
    if (cudaMemsetAsync(scratch, 0, (size_t)plan.tiles * sizeof(int), (cudaStream_t)stream) != cudaSuccess)
      return AWQ_ECUDA;
  }
  const cudaError_t e = launch_gemv(x, reinterpret_cast<const uint32_t*>(qweight),
                                    reinterpret_cast<const uint32_t*>(qzeros), scales, y, M, K, N, plan, scratch,
                                    err, (cudaStream_t)stream);
  return e == cudaSuccess ? AWQ_OK : AWQ_ECUDA;
}
