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
// The first 1024-byte-aligned byte at or after `p` in shared memory.  Written as pointer arithmetic
// on the shared array itself, not through an integer, so that the compiler still knows the result
// points to shared memory and accesses through it stay shared-memory loads and stores.
__device__ __forceinline__ uint8_t* align_smem_1024(uint8_t* p) {
  return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
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
__device__ __noinline__ bool wait_bounded_slow(uint32_t bar, uint32_t parity, volatile int* abort, int* err, int id,
                                               long long limit_ns = kWaitLimitNs) {
  const long long t0 = now_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try(bar, parity)) return true;
    if ((spin & 255u) == 0) {
      if (*abort) return false;
      if (now_ns() - t0 > limit_ns) {
        if (err) atomicExch(err, id);
        *abort = 1;
        return false;
      }
    }
  }
}
// Bounded wait that sleeps `sleep_ns` between polls: for a thread that shares its scheduler with
// warps that have work and does not need to react within nanoseconds (a copy producer refilling a
// ring several microseconds deep), so that its polling does not take their issue slots.
__device__ __noinline__ bool wait_backoff_slow(uint32_t bar, uint32_t parity, volatile int* abort, int* err, int id,
                                               uint32_t sleep_ns) {
  const long long t0 = now_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try(bar, parity)) return true;
    __nanosleep(sleep_ns);
    if ((spin & 15u) == 0) {
      if (*abort) return false;
      if (now_ns() - t0 > kWaitLimitNs) {
        if (err) atomicExch(err, id);
        *abort = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool wait_backoff(uint32_t bar, uint32_t parity, volatile int* abort, int* err, int id,
                                             uint32_t sleep_ns) {
  if (mbar_try(bar, parity)) return true;
  return wait_backoff_slow(bar, parity, abort, err, id, sleep_ns);
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

// One tiled TMA store of a shared-memory box (128-byte aligned, dense rows) to global memory; rows and
// columns outside the tensor are not written.  The caller commits the bulk group and waits until the
// shared memory has been read before reusing it or exiting.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// One contiguous copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from global to
// shared memory, completing on `bar` with its byte count.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// ---- tcgen05 (5th-generation tensor cores, tensor memory)

// Shared-memory matrix descriptor, 128-byte swizzle: start, leading / stride byte offsets.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}
// Arrives on `bar` once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 8 consecutive 32-bit columns of this thread's TMEM lane (32x32b shape), waited for.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(taddr)
               : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (32x32b shape); the caller waits
// (tcgen05.wait::ld) before using them.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 16 consecutive 32-bit columns into this thread's TMEM lane; the caller waits (tcgen05.wait::st)
// before another thread may read them.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace
}  // namespace awq
