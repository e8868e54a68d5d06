// Decode GEMV (M <= 8 tokens): y[m, n] = sum_k x[m, k] * W[k, n], W dequantized in registers.
//
// Source of the operation: the M <= 8 branch of the AWQ dispatch snippet,
// gemv_forward_cuda(inputs, qweight, scales, qzeros, group_size) ("Speed up AWQ
// 2.5x with updated kernel").  The kernel design is this library's own:
//
//  * The weight stream dominates (0.52 B per weight); every packed word is read
//    exactly once with 64-bit non-allocating loads, many loads in flight per warp.
//  * The tensor pipe does the multiply: each warp issues mma.sync m16n8k16 with the
//    dequantized weights as the A operand (16 output columns x 16 k) and the
//    activations as B (16 k x 8 tokens), fp32 accumulation.  The mma wants k-pairs in
//    each 32-bit A register while a packed word holds 8 columns of one k, so a PRMT
//    takes the same byte of two consecutive rows, and a LOP3 with the fp16 magic
//    0x6400 turns its low / high nibbles into (1024 + q) / (1024 + 16 q) halves.
//  * HSUB2 of the zero (same magic) then HMUL2 by the scale (s, or s / 16 for the
//    high nibble) give fp16_RN((q - z) * s), the same value the dequant kernel writes.
//  * The 16 k-slots of one mma are assigned to 16 rows so that each lane's four
//    k-slots are four consecutive rows: the activations for two mmas are then one
//    128-bit load.  The assignment is the same for A and B, so the sum is unchanged.
//  * K is split over the 4 warps of a CTA (reduced through shared memory) and over
//    `split` CTAs (fp32 partials in the workspace; the last CTA of a column tile,
//    found with an atomic ticket, sums the partials in slice order and rounds once).
#include <cuda_fp16.h>

#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kWarps = 4;          // warps per CTA, each on its own 128-row groups
constexpr int kTileWords = 16;     // packed words per CTA tile = 128 output columns
constexpr int kTileCols = kTileWords * 8;

__device__ __forceinline__ uint2 ld_stream_u2(const uint32_t* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (a & mask) | 0x64006400 in one LOP3
template <uint32_t MASK>
__device__ __forceinline__ uint32_t magic(uint32_t a) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "n"(0x64006400u));
  return d;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// PRMT selector: byte b of operand a -> result bytes 0,1; byte b of operand b -> bytes 2,3.
__device__ __forceinline__ constexpr uint32_t byte_sel(int b) {
  return (uint32_t)(b | (b << 4) | ((b + 4) << 8) | ((b + 4) << 12));
}

// Broadcast fp16 number `idx` (0..7) of an 8-half vector into both halves.
__device__ __forceinline__ uint32_t bcast_half(const uint4& v, int idx) {
  const uint32_t w = idx < 2 ? v.x : idx < 4 ? v.y : idx < 6 ? v.z : v.w;
  return (idx & 1) ? prmt(w, w, 0x3232u) : prmt(w, w, 0x1010u);
}

__global__ void __launch_bounds__(kWarps * 32)
gemv_kernel(const __half* __restrict__ x, const uint32_t* __restrict__ qw, const uint32_t* __restrict__ qz,
            const __half* __restrict__ scales, __half* __restrict__ y, float* __restrict__ part,
            int* __restrict__ counters, int M, int K, int N, int groups_per_split) {
  __shared__ float red[kWarps][kGemvMaxM][kTileCols];
  __shared__ int s_last;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2;  // mma group: A rows g / g+8, B column (token) g
  const int t = lane & 3;   // mma thread-in-group: k-slots 2t, 2t+1, 2t+8, 2t+9
  const int nw = N >> 3;
  const int tile = blockIdx.x;
  const int cw0 = tile * kTileWords + 2 * g;  // this lane's two packed word columns
  const bool col_ok = cw0 < nw;               // nw is even, so cw0 + 1 < nw as well
  const bool tok_ok = g < M;
  const int n_groups = K / kGroup;
  const int g_begin = blockIdx.y * groups_per_split;
  const int g_end = min(n_groups, g_begin + groups_per_split);

  float acc[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][b][e] = 0.f;

  for (int grp = g_begin + warp; grp < g_end; grp += kWarps) {
    // per-group constants for this lane's 2 words x 4 bytes (lo / hi nibble columns)
    uint32_t zlo[2][4], zhi[2][4], slo[2][4], shi[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint32_t zword = 0x88888888u;  // symmetric variant: z = 8 in every nibble
      uint4 sv = make_uint4(0, 0, 0, 0);
      if (col_ok) {
        if (qz) zword = __ldg(qz + (size_t)grp * nw + cw0 + i);
        sv = __ldg(reinterpret_cast<const uint4*>(scales + (size_t)grp * N + 8 * (cw0 + i)));
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t zb = prmt(zword, zword, byte_sel(b));
        zlo[i][b] = magic<0x000F000Fu>(zb);  // 1024 + z(slot 2b)
        zhi[i][b] = magic<0x00F000F0u>(zb);  // 1024 + 16 z(slot 2b+1)
        slo[i][b] = bcast_half(sv, order_map(2 * b));
        shi[i][b] = hmul2(bcast_half(sv, order_map(2 * b + 1)), 0x2C002C00u);  // s / 16
      }
    }

#pragma unroll
    for (int q = 0; q < 4; ++q) {  // four 32-row chunks of the group
      const int row0 = grp * kGroup + 32 * q + 8 * t;
      uint2 wv[8];
#pragma unroll
      for (int r = 0; r < 8; ++r)
        wv[r] = col_ok ? ld_stream_u2(qw + (size_t)(row0 + r) * nw + cw0) : make_uint2(0, 0);
      uint4 xv = make_uint4(0, 0, 0, 0);
      if (tok_ok) xv = __ldg(reinterpret_cast<const uint4*>(x + (size_t)g * K + row0));
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // two mmas: rows 8t+4h .. 8t+4h+3 in each lane
        const uint32_t b0 = h ? xv.z : xv.x;
        const uint32_t b1 = h ? xv.w : xv.y;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint32_t r0 = i ? wv[4 * h + 0].y : wv[4 * h + 0].x;
          const uint32_t r1 = i ? wv[4 * h + 1].y : wv[4 * h + 1].x;
          const uint32_t r2 = i ? wv[4 * h + 2].y : wv[4 * h + 2].x;
          const uint32_t r3 = i ? wv[4 * h + 3].y : wv[4 * h + 3].x;
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const uint32_t p01 = prmt(r0, r1, byte_sel(b));
            const uint32_t p23 = prmt(r2, r3, byte_sel(b));
            const uint32_t a0 = hmul2(hsub2(magic<0x000F000Fu>(p01), zlo[i][b]), slo[i][b]);
            const uint32_t a1 = hmul2(hsub2(magic<0x00F000F0u>(p01), zhi[i][b]), shi[i][b]);
            const uint32_t a2 = hmul2(hsub2(magic<0x000F000Fu>(p23), zlo[i][b]), slo[i][b]);
            const uint32_t a3 = hmul2(hsub2(magic<0x00F000F0u>(p23), zhi[i][b]), shi[i][b]);
            mma16816(acc[i][b], a0, a1, a2, a3, b0, b1);
          }
        }
      }
    }
  }

  // D fragment: d0/d1 = (column lo, tokens 2t, 2t+1), d2/d3 = (column hi, tokens 2t, 2t+1)
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int nlo = (2 * g + i) * 8 + order_map(2 * b);
      const int nhi = (2 * g + i) * 8 + order_map(2 * b + 1);
      red[warp][2 * t][nlo] = acc[i][b][0];
      red[warp][2 * t + 1][nlo] = acc[i][b][1];
      red[warp][2 * t][nhi] = acc[i][b][2];
      red[warp][2 * t + 1][nhi] = acc[i][b][3];
    }
  __syncthreads();

  const int nl = threadIdx.x;  // one output column per thread (128 threads)
  const int n = tile * kTileCols + nl;
  const bool n_ok = n < N;
  float sum[kGemvMaxM];
#pragma unroll
  for (int m = 0; m < kGemvMaxM; ++m) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += red[w][m][nl];
    sum[m] = s;
  }

  const int split = gridDim.y;
  if (split == 1) {
    if (n_ok)
      for (int m = 0; m < M; ++m) y[(size_t)m * N + n] = __float2half_rn(sum[m]);
    return;
  }

  if (n_ok)
    for (int m = 0; m < M; ++m) part[((size_t)blockIdx.y * M + m) * N + n] = sum[m];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(counters + tile, 1) == split - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (n_ok) {
    for (int m = 0; m < M; ++m) {
      float s = 0.f;
      for (int sp = 0; sp < split; ++sp) s += __ldcg(part + ((size_t)sp * M + m) * N + n);
      y[(size_t)m * N + n] = __float2half_rn(s);
    }
  }
  if (threadIdx.x == 0) atomicExch(counters + tile, 0);  // leave the ticket at zero for the next call
}

}  // namespace

GemvPlan gemv_plan(int64_t M, int64_t K, int64_t N, int split_k) {
  (void)M;
  GemvPlan p;
  p.tiles = (int)((N / 8 + kTileWords - 1) / kTileWords);
  const int n_groups = (int)(K / kGroup);
  int split = split_k;
  if (split <= 0) {
    // one 128-row group per warp when that keeps the grid within ~4 waves of 4-warp CTAs,
    // else two or more groups per warp
    const int target_ctas = 152 * 4 * 4;
    int gpw = 1;
    while (p.tiles * ((n_groups + kWarps * gpw - 1) / (kWarps * gpw)) > target_ctas && gpw < n_groups) ++gpw;
    split = (n_groups + kWarps * gpw - 1) / (kWarps * gpw);
  }
  if (split > n_groups) split = n_groups;
  if (p.tiles > kMaxCounters) split = 1;  // the ticket counters would not fit the workspace block
  if (split < 1) split = 1;
  p.groups_per_split = (n_groups + split - 1) / split;
  p.split = (n_groups + p.groups_per_split - 1) / p.groups_per_split;  // no empty slices
  return p;
}

size_t gemv_workspace_bytes(const GemvPlan& p, int64_t M, int64_t N) {
  if (p.split <= 1) return 0;
  return kCounterBytes + align256((size_t)p.split * (size_t)M * (size_t)N * sizeof(float));
}

cudaError_t launch_gemv(const uint16_t* x, const uint32_t* qw, const uint32_t* qz, const uint16_t* sc,
                        uint16_t* y, int64_t M, int64_t K, int64_t N, const GemvPlan& p, void* ws,
                        int* err, cudaStream_t s) {
  (void)err;
  float* part = nullptr;
  int* counters = nullptr;
  if (p.split > 1) {
    counters = static_cast<int*>(ws);
    part = reinterpret_cast<float*>(static_cast<char*>(ws) + kCounterBytes);
  }
  dim3 grid(p.tiles, p.split);
  gemv_kernel<<<grid, kWarps * 32, 0, s>>>(reinterpret_cast<const __half*>(x), qw, qz,
                                           reinterpret_cast<const __half*>(sc), reinterpret_cast<__half*>(y),
                                           part, counters, (int)M, (int)K, (int)N, p.groups_per_split);
  return cudaGetLastError();
}

}  // namespace awq
