// W4A8 activation kernels: per-token dynamic int8 quantization and the exact int8 -> fp16
// widening that feeds the fp16 tensor path.
//
// Source: "Support W4A8 quantization for vllm" (vLLM pull request #5218): the dynamic_quant
// function of brisker's consistency script (scale = absmax of the fp16 row / 127 computed in
// fp16, widened to float; codes = round(x / scale) clamped to [-128, 127]) and HandH1998's
// note that this per-token scale is computed online.
#include <cuda_fp16.h>

#include "awq_host.h"
#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kQThreads = 256;
constexpr int kQ1MaxK = 32768;  // rows up to this length are held in shared memory (64 KB)

// code = rint(x / s) for s > 0, clamped to [-128, 127], with the IEEE fp32 quotient of the pages'
// script, as a float (an integer).  x * (1 / s) differs from the correctly rounded quotient by at most
// a few ulp, which can change the rounded integer only next to a half-integer: where the product lies
// within 1e-4 of one (|r - rint(r)| within 1e-4 of 0.5; the difference is exact in fp32) the quotient
// is taken exactly.
__device__ __forceinline__ float code_value(float xv, float s, float inv) {
  const float r = xv * inv;
  float q = rintf(r);
  if (fabsf(fabsf(r - q) - 0.5f) < 1.0e-4f) q = rintf(__fdiv_rn(xv, s));
  return fminf(fmaxf(q, -128.f), 127.f);
}

// The eight codes of one 16-byte activation vector: as int8 into xq (when given) and widened to fp16
// (exact) into x16 (when given), the operand of the fp16 tensor path.
__device__ __forceinline__ void store_codes(const uint32_t (&out)[2], int8_t* xq, __half* x16, int64_t r, int K, int i) {
  if (xq) reinterpret_cast<uint2*>(xq + r * (int64_t)K)[i] = make_uint2(out[0], out[1]);
  if (x16) {
    uint32_t h[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const uint32_t w = out[p >> 1] >> (16 * (p & 1));
      const int a = (int)(int8_t)(w & 0xFFu), b = (int)(int8_t)((w >> 8) & 0xFFu);
      h[p] = (uint32_t)__half_as_ushort(__int2half_rn(a)) | ((uint32_t)__half_as_ushort(__int2half_rn(b)) << 16);
    }
    reinterpret_cast<uint4*>(x16 + r * (int64_t)K)[i] = make_uint4(h[0], h[1], h[2], h[3]);
  }
}

// One CTA per token row, the row read from DRAM once: it is kept in shared memory between the absmax
// pass and the coding pass.  T threads: 1024 when the rows are too few to fill the GPU (more of a
// row's loads in flight per CTA), 256 otherwise (more rows per SM).
template <int T>
__global__ void __launch_bounds__(T)
quant_act_smem_kernel(const __half* __restrict__ x, int8_t* __restrict__ xq, float* __restrict__ s_tok,
                      __half* __restrict__ x16, int K) {
  // the GEMM that reads these codes is launched as a programmatic dependent: it may start its setup
  // and weight stream now and waits for this grid to complete before it reads them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint4 row[];
  __shared__ uint32_t warp_max[T / 32];
  __shared__ float s_shared;
  const int64_t r = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + r * (int64_t)K);
  const int nvec = K / 8;
  // |x| as fp16 bits, two per word (integer order equals magnitude order for finite values)
  uint32_t mx2 = 0;
#pragma unroll 4
  for (int i = threadIdx.x; i < nvec; i += T) {
    const uint4 v = __ldcs(xr + i);
    row[i] = v;
    mx2 = __vmaxu2(mx2, v.x & 0x7FFF7FFFu);
    mx2 = __vmaxu2(mx2, v.y & 0x7FFF7FFFu);
    mx2 = __vmaxu2(mx2, v.z & 0x7FFF7FFFu);
    mx2 = __vmaxu2(mx2, v.w & 0x7FFF7FFFu);
  }
  uint32_t mx = max(mx2 & 0xFFFFu, mx2 >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = 0;
    for (int w = 0; w < T / 32; ++w) m = max(m, warp_max[w]);
    const float absmax = __half2float(__ushort_as_half((unsigned short)m));
    const float s = __half2float(__float2half_rn(__fdiv_rn(absmax, 127.0f)));
    s_shared = s;
    s_tok[r] = s;
  }
  __syncthreads();
  const float s = s_shared;
  const float inv = s > 0.f ? __frcp_rn(s) : 0.f;
#pragma unroll 2
  for (int i = threadIdx.x; i < nvec; i += T) {
    const uint4 v = row[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float q[8];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[p]));
      q[2 * p] = s > 0.f ? code_value(f.x, s, inv) : 0.f;
      q[2 * p + 1] = s > 0.f ? code_value(f.y, s, inv) : 0.f;
    }
    if (x16) {  // integers of at most 8 bits: exact in fp16
      uint32_t h[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const __half2 hv = __floats2half2_rn(q[2 * p], q[2 * p + 1]);
        h[p] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      reinterpret_cast<uint4*>(x16 + r * (int64_t)K)[i] = make_uint4(h[0], h[1], h[2], h[3]);
    }
    if (xq) {
      uint32_t out[2] = {0, 0};
#pragma unroll
      for (int j = 0; j < 8; ++j) out[j >> 2] |= ((uint32_t)(int)q[j] & 0xFFu) << (8 * (j & 3));
      reinterpret_cast<uint2*>(xq + r * (int64_t)K)[i] = make_uint2(out[0], out[1]);
    }
  }
}

// One CTA per token row: pass 1 finds absmax, pass 2 writes the codes (second read hits L2).
__global__ void __launch_bounds__(kQThreads)
quant_act_kernel(const __half* __restrict__ x, int8_t* __restrict__ xq, float* __restrict__ s_tok,
                 __half* __restrict__ x16, int K) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ uint32_t warp_max[kQThreads / 32];
  __shared__ float s_shared;
  const int64_t row = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * (int64_t)K);
  const int nvec = K / 8;

  uint32_t mx = 0;  // |x| as fp16 bits: integer order equals magnitude order for finite values
  for (int i = threadIdx.x; i < nvec; i += kQThreads) {
    const uint4 v = __ldg(xr + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      mx = max(mx, w[j] & 0x7FFFu);
      mx = max(mx, (w[j] >> 16) & 0x7FFFu);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = 0;
    for (int w = 0; w < kQThreads / 32; ++w) m = max(m, warp_max[w]);
    const float absmax = __half2float(__ushort_as_half((unsigned short)m));
    // fp16 division of the page's script: fp32 quotient rounded once to fp16, then widened
    const float s = __half2float(__float2half_rn(__fdiv_rn(absmax, 127.0f)));
    s_shared = s;
    s_tok[row] = s;
  }
  __syncthreads();
  const float s = s_shared;
  for (int i = threadIdx.x; i < nvec; i += kQThreads) {
    const uint4 v = __ldg(xr + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2] = {0, 0};
    if (s > 0.f) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float xv = __half2float(__ushort_as_half((unsigned short)(w[j >> 1] >> (16 * (j & 1)))));
        float qv = rintf(__fdiv_rn(xv, s));
        qv = fminf(fmaxf(qv, -128.f), 127.f);
        out[j >> 2] |= ((uint32_t)(int)qv & 0xFFu) << (8 * (j & 3));
      }
    }
    store_codes(out, xq, x16, row, K, i);
  }
}

__global__ void i8_to_f16_kernel(const int8_t* __restrict__ xq, __half* __restrict__ out, int64_t nvec) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nvec; i += (int64_t)gridDim.x * blockDim.x) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(xq) + i);
    uint32_t o[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const uint32_t w = p < 2 ? v.x : v.y;
      const int a = (int)(int8_t)((w >> (16 * (p & 1))) & 0xFF);
      const int b = (int)(int8_t)((w >> (16 * (p & 1) + 8)) & 0xFF);
      o[p] = (uint32_t)__half_as_ushort(__int2half_rn(a)) | ((uint32_t)__half_as_ushort(__int2half_rn(b)) << 16);
    }
    reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

cudaError_t launch_quant_act(const uint16_t* x, int8_t* xq, float* s_tok, int64_t M, int64_t K, cudaStream_t s,
                             uint16_t* x16) {
  if (M == 0) return cudaSuccess;
  if (K <= kQ1MaxK) {
    const int smem = (int)K * 2;
    const bool wide = M <= 2 * (int64_t)device_sm_count();  // two 1024-thread CTAs fit one SM
    const void* fn = wide ? reinterpret_cast<const void*>(quant_act_smem_kernel<1024>)
                          : reinterpret_cast<const void*>(quant_act_smem_kernel<kQThreads>);
    if (smem > 48 * 1024) {
      const cudaError_t e = set_smem_once(fn, kQ1MaxK * 2);
      if (e != cudaSuccess) return e;
    }
    if (wide)
      quant_act_smem_kernel<1024><<<(unsigned)M, 1024, smem, s>>>(reinterpret_cast<const __half*>(x), xq, s_tok,
                                                                   reinterpret_cast<__half*>(x16), (int)K);
    else
      quant_act_smem_kernel<kQThreads><<<(unsigned)M, kQThreads, smem, s>>>(
          reinterpret_cast<const __half*>(x), xq, s_tok, reinterpret_cast<__half*>(x16), (int)K);
  } else {
    quant_act_kernel<<<(unsigned)M, kQThreads, 0, s>>>(reinterpret_cast<const __half*>(x), xq, s_tok,
                                                       reinterpret_cast<__half*>(x16), (int)K);
  }
  return cudaGetLastError();
}

cudaError_t launch_i8_to_f16(const int8_t* xq, uint16_t* x16, int64_t count, cudaStream_t s) {
  const int64_t nvec = count / 8;
  if (nvec == 0) return cudaSuccess;
  int64_t blocks = (nvec + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  i8_to_f16_kernel<<<(unsigned)blocks, 256, 0, s>>>(xq, reinterpret_cast<__half*>(x16), nvec);
  return cudaGetLastError();
}

}  // namespace awq
