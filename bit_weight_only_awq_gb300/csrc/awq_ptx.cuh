// Inline-PTX helpers shared by the TMA / mbarrier kernels (GEMV and tensor-core GEMM).
#pragma once

#include <cuda.h>
#include <cstdint>

namespace awq {
namespace {  // every translation unit gets its own copy

constexpr long long kWaitLimitNs = 2000000000LL;  // bound of every device-side wait: 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ long long now_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase.  Gives up when `abort` is raised by another
// thread or after kWaitLimitNs; a timeout records `id` in the device error word
// and raises `abort`.  Returns true when the phase completed.
__device__ __noinline__ bool wait_bounded_slow(uint32_t bar, uint32_t parity, volatile int* abort, int* err, int id) {
  const long long t0 = now_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try(bar, parity)) return true;
    if ((spin & 255u) == 0) {
      if (*abort) return false;
      if (now_ns() - t0 > kWaitLimitNs) {
        if (err) atomicExch(err, id);
        *abort = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort, int* err, int id) {
  if (mbar_try(bar, parity)) return true;  // fast path stays inline
  return wait_bounded_slow(bar, parity, abort, err, id);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}


}  // namespace
}  // namespace awq
