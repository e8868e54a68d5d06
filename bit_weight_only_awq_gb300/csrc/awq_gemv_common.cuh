// Inline-PTX helpers shared by the two decode GEMV kernels (AWQ layout and prepared layout).
#pragma once

#include <cstdint>

namespace awq {
namespace {  // every translation unit gets its own copy

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (a & mask) | 0x64006400 in one LOP3: the nibbles under the mask become the exact fp16 halves
// 1024 + q (mask 0x000F000F) or 1024 + 16 q (mask 0x00F000F0)
template <uint32_t MASK>
__device__ __forceinline__ uint32_t magic(uint32_t a) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "n"(0x64006400u));
  return d;
}

// D += A B, m16n8k16, fp16 operands, fp32 accumulators (the legacy tensor path, fed from registers)
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Activation pair (k, k+1), k even (0..62), of token g in a 128-byte-swizzled box of 64 fp16 per token.
__device__ __forceinline__ uint32_t x_offset(int g, int k) {
  return (uint32_t)(g * 128 + ((((k >> 3) ^ g)) << 4) + (k & 7) * 2);
}

}  // namespace
}  // namespace awq
