// Pack / unpack / dequantize: memory-bound elementwise kernels (one packed word per thread).
//
// Packing follows the older AWQ format ("Speed up AWQ 2.5x with updated kernel",
// casper-hansen's format differences): nibble slot i of word c holds logical
// column 8c + map[i], map = [0, 2, 4, 6, 1, 3, 5, 7].
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kThreads = 256;

inline int grid_for(int64_t work) {
  int64_t blocks = (work + kThreads - 1) / kThreads;
  // grid-stride loops cap the grid at a few waves of 152 SMs
  const int64_t cap = 152 * 16;
  return (int)(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
}

// slot of logical column `col` in a packed word: the older format's map, or (NEW) the new format's [0..7]
template <bool NEW>
__device__ __forceinline__ int slot_for(int col) { return NEW ? col : slot_of_col(col); }

template <bool NEW>
__global__ void pack_kernel(const uint8_t* __restrict__ q, int64_t words, uint32_t* __restrict__ out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < words;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint2 b = __ldg(reinterpret_cast<const uint2*>(q) + i);  // 8 codes, columns 0..7
    uint32_t w = 0;
#pragma unroll
    for (int col = 0; col < 8; ++col) {
      uint32_t code = ((col < 4 ? b.x : b.y) >> (8 * (col & 3))) & 0xFFu;
      code = code > 15u ? 15u : code;  // clamp (packer fix on the W4A8 page)
      w |= code << (4 * slot_for<NEW>(col));
    }
    out[i] = w;
  }
}

template <bool NEW>
__global__ void unpack_kernel(const uint32_t* __restrict__ packed, int64_t words, uint8_t* __restrict__ q) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < words;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t w = __ldg(packed + i);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int col = 0; col < 8; ++col) {
      const uint32_t code = (w >> (4 * slot_for<NEW>(col))) & 0xFu;
      if (col < 4) lo |= code << (8 * col);
      else hi |= code << (8 * (col - 4));
    }
    reinterpret_cast<uint2*>(q)[i] = make_uint2(lo, hi);
  }
}

// One thread per packed word (k, c): eight outputs W[k, 8c..8c+7], fp16 or (BF16) bf16 like the scales.
// (q - z) is an exact small integer and (q - z) * s is exact in fp32 (at most 5 + 11 significant bits), so
// the conversion to the output format (round to nearest even) performs the single rounding.
template <bool BF16>
__global__ void dequant_kernel(const uint32_t* __restrict__ qw, const uint32_t* __restrict__ qz,
                               const uint16_t* __restrict__ scales, int64_t K, int64_t nw, int group,
                               uint16_t* __restrict__ w) {
  const int64_t words = K * nw;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < words;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t k = i / nw;
    const int64_t c = i - k * nw;
    const int64_t grp = k / group;
    const uint32_t word = __ldg(qw + i);
    const uint32_t zword = qz ? __ldg(qz + grp * nw + c) : 0x88888888u;  // symmetric: z = 8
    const uint4 sv = __ldg(reinterpret_cast<const uint4*>(scales + grp * nw * 8 + c * 8));
    const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
    uint32_t outw[4];
#pragma unroll
    for (int pair = 0; pair < 4; ++pair) {
      uint32_t halves = 0;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int col = 2 * pair + e;
        const int sh = 4 * slot_of_col(col);
        const int d = (int)((word >> sh) & 0xFu) - (int)((zword >> sh) & 0xFu);
        const unsigned short sbits = (unsigned short)(sw[pair] >> (16 * e));
        unsigned short r;
        if constexpr (BF16) {
          r = __bfloat16_as_ushort(__float2bfloat16_rn((float)d * __bfloat162float(__ushort_as_bfloat16(sbits))));
        } else {
          r = __half_as_ushort(__float2half_rn((float)d * __half2float(__ushort_as_half(sbits))));
        }
        halves |= (uint32_t)r << (16 * e);
      }
      outw[pair] = halves;
    }
    reinterpret_cast<uint4*>(w)[i] = make_uint4(outw[0], outw[1], outw[2], outw[3]);
  }
}

}  // namespace

cudaError_t launch_pack(const uint8_t* q, int64_t rows, int64_t n, uint32_t* packed, cudaStream_t s, bool new_order) {
  const int64_t words = rows * (n / 8);
  if (words == 0) return cudaSuccess;
  if (new_order) pack_kernel<true><<<grid_for(words), kThreads, 0, s>>>(q, words, packed);
  else pack_kernel<false><<<grid_for(words), kThreads, 0, s>>>(q, words, packed);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t* packed, int64_t rows, int64_t n, uint8_t* q, cudaStream_t s,
                          bool new_order) {
  const int64_t words = rows * (n / 8);
  if (words == 0) return cudaSuccess;
  if (new_order) unpack_kernel<true><<<grid_for(words), kThreads, 0, s>>>(packed, words, q);
  else unpack_kernel<false><<<grid_for(words), kThreads, 0, s>>>(packed, words, q);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const uint32_t* qw, const uint32_t* qz, const uint16_t* scales, int64_t K,
                           int64_t N, int group, uint16_t* w, cudaStream_t s, bool bf16) {
  const int64_t words = K * (N / 8);
  if (words == 0) return cudaSuccess;
  if (bf16) dequant_kernel<true><<<grid_for(words), kThreads, 0, s>>>(qw, qz, scales, K, N / 8, group, w);
  else dequant_kernel<false><<<grid_for(words), kThreads, 0, s>>>(qw, qz, scales, K, N / 8, group, w);
  return cudaGetLastError();
}

}  // namespace awq
