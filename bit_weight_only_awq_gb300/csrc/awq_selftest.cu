// awq_selftest_wait_timeout: proves, on the GPU in use, that an expired device-side wait is
// reported as a status and leaves the CUDA context usable.
//
// Every wait of the library's kernels on an mbarrier phase is bounded (wait_bounded): when the
// phase does not complete in time, the waiting thread records the wait's id in the per-device
// error word, raises its CTA's abort flag and returns, and the host reads the word with
// awq_last_device_error.  This entry point runs that same wait on a barrier that nothing ever
// arrives on, with a short caller-chosen limit, so the path can be exercised without a fault,
// a trap or a hang.
#include <cuda_runtime.h>

#include "../../include/awq.h"
#include "awq_internal.h"
#include "awq_ptx.cuh"

namespace awq {
namespace {

constexpr int kSelftestWaitId = 901;

__global__ void selftest_wait_kernel(int* err, long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // expects one arrival that never comes
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_try(smem_u32(&bar), 0))
      wait_bounded_slow(smem_u32(&bar), 0, &abort_flag, err, kSelftestWaitId, limit_ns);
  }
  __syncthreads();
}

}  // namespace
}  // namespace awq

using namespace awq;

extern "C" awq_status awq_selftest_wait_timeout(int64_t limit_ns, awq_stream_t stream) {
  if (limit_ns <= 0 || limit_ns > kWaitLimitNs) return AWQ_EINVAL;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return AWQ_ECUDA;
  if (major != 10 || minor != 3) return AWQ_EARCH;
  int* err = device_error_ptr();
  if (!err) return AWQ_ECUDA;
  selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err, (long long)limit_ns);
  return cudaGetLastError() == cudaSuccess ? AWQ_OK : AWQ_ECUDA;
}
