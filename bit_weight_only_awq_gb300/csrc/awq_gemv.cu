// Decode GEMV (M <= 16 tokens): y[m, n] = sum_k x[m, k] * W[k, n], W dequantized in registers.
//
// Source of the operation: the M <= 8 branch of the AWQ dispatch snippet,
// gemv_forward_cuda(inputs, qweight, scales, qzeros, group_size) ("Speed up AWQ
// 2.5x with updated kernel").  The kernel design is this library's own:
//
//  * HBM-bound: every packed word is read exactly once.  Measured on GB300 with this
//    kernel's access pattern (512-column tiles walked down K, 256-byte runs per row), a
//    TMA stream reaches ~6.1 TB/s with 32 KB stages but only ~5.4 TB/s with 16 KB ones,
//    whatever the ring depth; and a decode GEMV of a 7B-model layer moves only 8-47 MB,
//    so per-call latency (first bytes, the cross-CTA reduction, the launch) matters as
//    much as the streaming rate.  One persistent CTA per SM: a producer warp streams
//    36 KB stages (one whole quantization group: 128 rows x 512 columns of packed words
//    as four 128-byte-swizzled TMA boxes, the group's zero-point / scale rows and the
//    128 activations of every token) through a 3-deep ring, and 8 consumer warps (one
//    64-column slice each) copy their share of a stage into registers 64 rows at a time
//    and release the slot after the last copy.  The registers are sized for one CTA per
//    SM (the SM sub-partition holding the producer warp runs three warps); programmatic
//    dependent launch starts the next call's CTA on an SM as soon as this call's CTA
//    there exits, and it streams its first stages before waiting for this call.
//  * Persistent, evenly balanced grid: the (512-column tile, 64-row block) units are cut
//    into equal contiguous ranges, one per SM; a CTA's units are grouped into stages of
//    one quantization group (or a lone 64-row block at a range edge).  A tile finished by
//    one CTA is written directly.  A tile shared by several CTAs is completed by the one
//    holding its first row block (for which it is the last tile of the range): after its
//    range it waits, bounded, until the other contributors have published their fp32
//    partials (stores, a fence, a count on the tile), adds them to its own sums in
//    contributor order and rounds once to fp16, so results are bit-reproducible.  The
//    other contributors publish after their range and exit at once, which frees their SMs
//    for the next call.  No CTA waits before publishing its own partial, and a grid with
//    shared tiles has at most one CTA per SM, so all of them are resident and every wait
//    ends.
//  * Programmatic dependent launch: the GEMV starts streaming its weights before waiting
//    for the previous kernel, and touches activations, outputs and the workspace only
//    after that wait.
//  * The multiply runs on the tensor pipe: mma.sync m16n8k16 with the packed weights as
//    the A operand (16 output columns x 16 k) and the activations as B (16 k x 8 tokens),
//    fp32 accumulation.  The mma wants k-pairs in each 32-bit A register while a packed
//    word holds 8 columns of one k, so a PRMT takes the same byte of two consecutive rows,
//    and a LOP3 with the fp16 magic 0x6400 turns its low / high nibbles into the exact
//    halves 1024 + q / 1024 + 16 q.  Those enter the mma as they are: the group's zero
//    point and scale are applied once per group and column to the fp32 sums, by linearity
//        sum_k (q - z) s x = s (sum_k (1024 + q) x - (1024 + z) sum_k x)
//    (high nibble: s / 16 and 1024 + 16 z), with sum_k x from one more mma against an
//    all-ones A.  This drops the two fp16 operations per weight pair that dominated the
//    issue slots; the price is that the products use s (q - z) in fp32 instead of its
//    fp16 rounding, a relative difference of at most 2^-11 per weight, far inside the
//    output tolerance, and a cancellation of the 1024 offsets in fp32 that costs about
//    eight of its 24 bits.
//  * 9..16 tokens (gemv_kernel<16>): the same stages, with 16-token activation boxes; every
//    dequantized A fragment feeds two mmas, one per 8-token half.  A per-group fold would need a
//    second set of group sums and overflow the registers, so this variant makes W exactly as the
//    dequant kernel does (HSUB2 of the zero, HMUL2 by the scale) and multiplies it straight into
//    the accumulators; streaming the weights once for 16 tokens beats the tensor-core GEMM's
//    16-token tiles by 1.3-2.9x.
//  * W4A8 from 9 to 16 tokens (gemv_kernel<16, true>): the same instance with the symmetric zero
//    point and unit scales, on activations that are int8 codes widened to fp16.  Each weight is the
//    exact half u - 8 and each product an integer of magnitude at most 1024; with at most 16384 rows
//    of a tile per CTA every fp32 sum is exact, partials are added across CTAs as int32, and the
//    output is the W4A8 epilogue fp16((acc * s_tok) * s_ch) ("Support W4A8 quantization for vllm").
//    Up to 8 tokens (gemv_kernel<8, true>) the folded loop runs instead, with the fold taken per
//    64-row block, where sum (1024 + u) x and sum x are exact integers below 2^24, and the offset
//    subtracted by one fused multiply-add, exactly.
//  * Lane (g, t) of the mma reads rows 2t, 2t+1 (+8) of each 16-row step; with the
//    128-byte swizzle those 32-bit shared-memory loads, and the activation loads, are
//    free of bank conflicts, and every address is a lane constant plus an immediate.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "awq_internal.h"
#include "awq_host.h"
#include "awq_ptx.cuh"
#include "awq_gemv_common.cuh"

namespace awq {
namespace {

constexpr int kConsumers = 8;                  // consumer warps, one 64-column slice of the tile each
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kStages = 3;
// Stages streamed before the wait on the previous kernel: more of them compete with that kernel's
// last CTAs for DRAM and measured slower (3: -2 to -3 % on 12-25 MB calls).
constexpr int kPrefetch = 2;
static_assert(kPrefetch >= 1 && kPrefetch <= kStages, "prefetch within the ring");
// Polling pauses: the producer's empty-slot waits and the consumers' full-slot waits share their
// schedulers with consumer warps that have arithmetic to issue.
constexpr uint32_t kProducerSleepNs = 1000;
constexpr uint32_t kConsumerSleepNs = 0;
constexpr int kRows = 64;                      // rows per unit (a TMA box, half a quantization group)
constexpr int kTileWords = 64;                 // packed words per tile row = 512 output columns
constexpr int kTileCols = kTileWords * 8;
constexpr int kBoxWords = 32;                  // one 128-byte-swizzled TMA box is 32 words wide
constexpr int kBoxBytes = kRows * kBoxWords * 4;   // 8 KB
constexpr int kUnitsPerStage = 2;              // 64-row units per stage: 2 = one quantization group
constexpr int kUnitQBytes = kRows * kTileWords * 4;  // 16 KB of packed words per unit
constexpr int kColStride = kUnitsPerStage * kBoxBytes;  // box (column half c, unit h) at c * kColStride + h * 8 KB
constexpr int kQBytes = kUnitsPerStage * kUnitQBytes;
constexpr int kZBytes = kTileWords * 4;            // 256 B
constexpr int kSBytes = kTileCols * 2;             // 1 KB
// Stage layout for calls of up to T tokens: T = 8 (the folded kernel) or 16 (two 8-token halves)
template <int T>
struct Geo {
  static constexpr int kXBoxBytes = T * kRows * 2;  // one 128B-swizzled box, T tokens x 64 (1 or 2 KB)
  static constexpr int kXBytes = kUnitsPerStage * kXBoxBytes;
  static constexpr int kXOff = kQBytes;
  static constexpr int kZOff = kXOff + kXBytes;
  static constexpr int kSOff = kZOff + kZBytes;
  static constexpr int kStageBytes = ((kSOff + kSBytes) + 1023) / 1024 * 1024;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 512;  // alignment slack | ring | barriers, flags
  static_assert(T * kTileCols * 4 <= kStageBytes, "a completer's own sums fit one ring slot");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget of one CTA");
};
static_assert(kTileWords == kConsumers * 8, "one 8-word slice per consumer warp");

// PRMT selector: byte b of operand a -> result bytes 0,1; byte b of operand b -> bytes 2,3.
__device__ __forceinline__ constexpr uint32_t byte_sel(int b) {
  return (uint32_t)(b | (b << 4) | ((b + 4) << 8) | ((b + 4) << 12));
}

__device__ __forceinline__ void consumers_sync() {  // the consumer warps only (named barrier 1)
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
}
// consumers_sync that also returns whether `v` holds in any consumer thread
__device__ __forceinline__ bool consumers_any(bool v) {
  uint32_t r;
  asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}"
               : "=r"(r) : "r"((uint32_t)v), "r"(kConsumers * 32) : "memory");
  return r != 0;
}

// 32-bit word `word` (0..63) of packed row `row` (0..127) in the stage tile: 128-byte-swizzled
// boxes of 32 words x 64 rows, column half c = word / 32 at c * 16 KB, rows 64..127 8 KB further.
__device__ __forceinline__ uint32_t q_offset(int row, int word) {
  return (uint32_t)((word >> 5) * kColStride + row * 128 + (((((word & 31) >> 2) ^ (row & 7))) << 4) +
                    (word & 3) * 4);
}

// Lane-constant parts of the shared-memory addresses a consumer lane reads; every load of a
// stage is then one of these plus a compile-time row offset.
struct LaneOffsets {
  uint32_t q[2];  // packed word of row 2t + c, c = 0, 1 (rows +8 are +1024 bytes)
  uint32_t x[4];  // activation pair k = 16i + 2t of token g for the four 16-row steps i
};

template <int T>
__device__ __forceinline__ LaneOffsets lane_offsets(int word, int g, int t) {
  LaneOffsets o;
#pragma unroll
  for (int c = 0; c < 2; ++c) o.q[c] = q_offset(2 * t + c, word);
#pragma unroll
  for (int i = 0; i < 4; ++i) o.x[i] = Geo<T>::kXOff + x_offset(g, 16 * i + 2 * t);
  return o;
}

// A consumer lane's share of one stage, copied out of shared memory so the slot can be
// released before the arithmetic starts.
template <int T>
struct StageRegs {
  uint32_t r[4][4];         // [16-row step][rows 2t, 2t+1, 2t+8, 2t+9]
  uint32_t b[T / 8][4][2];  // [8-token half][16-row step][activation pairs k = 2t, 2t+8]
};

// 64-row unit `hh` (0, 1) of the stage at `sb`
template <int T>
__device__ __forceinline__ void load_stage(const uint8_t* sb, int hh, const LaneOffsets& lo, StageRegs<T>& sr) {
  const uint8_t* q0 = sb + hh * kBoxBytes + lo.q[0];
  const uint8_t* q1 = sb + hh * kBoxBytes + lo.q[1];
  const uint8_t* xb = sb + hh * Geo<T>::kXBoxBytes;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int base = 16 * it;  // (base + 2t + c) & 7 == (2t + c) & 7
    sr.r[it][0] = *reinterpret_cast<const uint32_t*>(q0 + base * 128);
    sr.r[it][1] = *reinterpret_cast<const uint32_t*>(q1 + base * 128);
    sr.r[it][2] = *reinterpret_cast<const uint32_t*>(q0 + (base + 8) * 128);
    sr.r[it][3] = *reinterpret_cast<const uint32_t*>(q1 + (base + 8) * 128);
    // k + 8 is the neighbouring 16-byte chunk: physical chunk ^ 1, address ^ 16; token g + 8 of the
    // second half has the same swizzle, 8 rows (1 KB) further
#pragma unroll
    for (int h = 0; h < T / 8; ++h) {
      sr.b[h][it][0] = *reinterpret_cast<const uint32_t*>(xb + h * 1024 + lo.x[it]);
      sr.b[h][it][1] = *reinterpret_cast<const uint32_t*>(xb + h * 1024 + (lo.x[it] ^ 16u));
    }
  }
}

// Zero-point / scale constants of this lane's packed word for one quantization group, as the fp32
// factors of the fold: sf[b] = s and s / 16 of slots 2b / 2b + 1 (low / high nibble of byte b), and
// szc[b] = sf times the magic-offset zero point, 1024 + z and 1024 + 16 z.
struct GroupConsts {
  float sf[4][2], szc[4][2];
};

__device__ __forceinline__ void group_consts(uint32_t zword, const uint4& sv, GroupConsts& c) {
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    // 1024 + z and 1024 + 16 z as fp32 bit patterns: byte b's nibbles land in the mantissa of 1024.0f
    // (whose last place is 2^-13) at bits 13..16 and 17..20, both from one shift of the zero word
    const uint32_t zs = 8 * b <= 13 ? zword << (13 - 8 * b) : zword >> (8 * b - 13);
    const float zl = __uint_as_float(0x44800000u | (zs & 0x0001E000u));
    const float zh = __uint_as_float(0x44800000u | (zs & 0x001E0000u));
    const __half* sh = reinterpret_cast<const __half*>(&sv);
    c.sf[b][0] = __half2float(sh[order_map(2 * b)]);
    c.sf[b][1] = __half2float(sh[order_map(2 * b + 1)]) * 0.0625f;  // s / 16, exact
    c.szc[b][0] = c.sf[b][0] * zl;
    c.szc[b][1] = c.sf[b][1] * zh;
  }
}

// Over the 64 rows held in `sr` (this lane's packed word column, 8 tokens): acc += (1024 + q)^T x
// (1024 + 16 q for the high nibbles) and sx += sum_k x, the latter as an mma against an all-ones A
// so that it lands in the accumulator layout.  Each 16-row step is written as phases over its four
// independent byte positions (PRMT, LOP3, mma) so that no instruction waits on the one issued just
// before it.
__device__ __forceinline__ void compute_stage(const StageRegs<8>& sr, float (&acc)[4][4], float (&sx)[4]) {
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    uint32_t p01[4], p23[4], a[4][4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      p01[b] = prmt(sr.r[it][0], sr.r[it][1], byte_sel(b));
      p23[b] = prmt(sr.r[it][2], sr.r[it][3], byte_sel(b));
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      a[b][0] = magic<0x000F000Fu>(p01[b]);
      a[b][1] = magic<0x00F000F0u>(p01[b]);
      a[b][2] = magic<0x000F000Fu>(p23[b]);
      a[b][3] = magic<0x00F000F0u>(p23[b]);
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) mma16816(acc[b], a[b][0], a[b][1], a[b][2], a[b][3], sr.b[0][it][0], sr.b[0][it][1]);
    mma16816(sx, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, sr.b[0][it][0], sr.b[0][it][1]);
  }
}

// Two-half (9..16 token) variant: each dequantized weight feeds two mmas, one per 8-token half, so the
// weights are made exactly as the dequant kernel makes them, W = fp16_RN((q - z) s), and multiplied
// straight into the fp32 accumulators (no per-group fold, which would need a second set of group
// sums per half).  zlo / zhi = 1024 + z and 1024 + 16 z of slots 2b / 2b + 1 (both halves of the
// register), slo / shi = s and s / 16.
struct GroupConstsH {
  uint32_t zlo[4], zhi[4], slo[4], shi[4];
};

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
// fp16 number `idx` (0..7) of an 8-half vector, in both halves of a register
__device__ __forceinline__ uint32_t bcast_half(const uint4& v, int idx) {
  const uint32_t w = idx < 2 ? v.x : idx < 4 ? v.y : idx < 6 ? v.z : v.w;
  return (idx & 1) ? prmt(w, w, 0x3232u) : prmt(w, w, 0x1010u);
}

__device__ __forceinline__ void group_consts_h(uint32_t zword, const uint4& sv, GroupConstsH& c) {
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t zb = prmt(zword, zword, byte_sel(b));
    c.zlo[b] = magic<0x000F000Fu>(zb);  // 1024 + z(slot 2b)
    c.zhi[b] = magic<0x00F000F0u>(zb);  // 1024 + 16 z(slot 2b+1)
    c.slo[b] = bcast_half(sv, order_map(2 * b));
    c.shi[b] = hmul2(bcast_half(sv, order_map(2 * b + 1)), 0x2C002C00u);  // s / 16, exact
  }
}

// bf16 variant: 128 + q is exact in bf16 but 128 + 16 q does not fit its 8 significant bits' magic form
// (the high nibble would reach the exponent), so high nibbles are shifted down first; both nibbles then
// give 128 + code, zero points 128 + z, and the scale is s for both.
__device__ __forceinline__ uint32_t magic_bf16(uint32_t a) {  // (a & 0x000F000F) | 0x43004300
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(0x000F000Fu), "n"(0x43004300u));
  return d;
}
__device__ __forceinline__ uint32_t bsub2(uint32_t a, uint32_t b) {  // exact here: (128 + q) - (128 + z)
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {  // one rounding to nearest even
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ void mma16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void group_consts_bf16(uint32_t zword, const uint4& sv, GroupConstsH& c) {
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t zb = prmt(zword, zword, byte_sel(b));
    c.zlo[b] = magic_bf16(zb);       // 128 + z(slot 2b)
    c.zhi[b] = magic_bf16(zb >> 4);  // 128 + z(slot 2b+1)
    c.slo[b] = bcast_half(sv, order_map(2 * b));
    c.shi[b] = bcast_half(sv, order_map(2 * b + 1));
  }
}

// acc[h] += W^T x_h over the 64 rows held in `sr`, for the two 8-token halves h.  HSUB2 of the zero
// (exact) then HMUL2 by the scale (s / 16 for the 16 q of the high nibble) give W = fp16_RN((q - z) s);
// BF16: the bf16 forms, W = bf16_RN((q - z) s).
template <int T, bool BF16 = false>
__device__ __forceinline__ void compute_stage_exact(const StageRegs<T>& sr, const GroupConstsH& c,
                                                    float (&acc)[T / 8][4][4]) {
  if constexpr (BF16) {
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      uint32_t p01[4], p23[4], a[4][4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        p01[b] = prmt(sr.r[it][0], sr.r[it][1], byte_sel(b));
        p23[b] = prmt(sr.r[it][2], sr.r[it][3], byte_sel(b));
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        a[b][0] = bmul2(bsub2(magic_bf16(p01[b]), c.zlo[b]), c.slo[b]);
        a[b][1] = bmul2(bsub2(magic_bf16(p01[b] >> 4), c.zhi[b]), c.shi[b]);
        a[b][2] = bmul2(bsub2(magic_bf16(p23[b]), c.zlo[b]), c.slo[b]);
        a[b][3] = bmul2(bsub2(magic_bf16(p23[b] >> 4), c.zhi[b]), c.shi[b]);
      }
#pragma unroll
      for (int h = 0; h < T / 8; ++h)
#pragma unroll
        for (int b = 0; b < 4; ++b)
          mma16816_bf16(acc[h][b], a[b][0], a[b][1], a[b][2], a[b][3], sr.b[h][it][0], sr.b[h][it][1]);
    }
  } else {
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      uint32_t p01[4], p23[4], a[4][4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        p01[b] = prmt(sr.r[it][0], sr.r[it][1], byte_sel(b));
        p23[b] = prmt(sr.r[it][2], sr.r[it][3], byte_sel(b));
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        a[b][0] = hmul2(hsub2(magic<0x000F000Fu>(p01[b]), c.zlo[b]), c.slo[b]);
        a[b][1] = hmul2(hsub2(magic<0x00F000F0u>(p01[b]), c.zhi[b]), c.shi[b]);
        a[b][2] = hmul2(hsub2(magic<0x000F000Fu>(p23[b]), c.zlo[b]), c.slo[b]);
        a[b][3] = hmul2(hsub2(magic<0x00F000F0u>(p23[b]), c.zhi[b]), c.shi[b]);
      }
#pragma unroll
      for (int h = 0; h < T / 8; ++h)
#pragma unroll
        for (int b = 0; b < 4; ++b)
          mma16816(acc[h][b], a[b][0], a[b][1], a[b][2], a[b][3], sr.b[h][it][0], sr.b[h][it][1]);
    }
  }
}

// two fp32 outputs rounded (to nearest even) to the layer's output format, fp16 or bf16, as one word
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

__device__ __forceinline__ int4 f4_to_i4(const float4& v) {
  return make_int4(__float2int_rn(v.x), __float2int_rn(v.y), __float2int_rn(v.z), __float2int_rn(v.w));
}
// W4A8 outputs of `n` consecutive columns of one token: y = fp16((acc * s_tok) * s_ch) (fp32 products in
// that order, one rounding), and the exact accumulators when `acc_out` is given.
__device__ __forceinline__ void store_w4a8(const int (&v)[8], float st, const __half* sch, __half* yp, int32_t* ap) {
  const uint4 sc = *reinterpret_cast<const uint4*>(sch);
  const __half* sh = reinterpret_cast<const __half*>(&sc);
  uint32_t h[4];
#pragma unroll
  for (int c = 0; c < 8; c += 2) {
    const __half lo = __float2half_rn(__fmul_rn(__fmul_rn((float)v[c], st), __half2float(sh[c])));
    const __half hi = __float2half_rn(__fmul_rn(__fmul_rn((float)v[c + 1], st), __half2float(sh[c + 1])));
    h[c / 2] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
  }
  *reinterpret_cast<uint4*>(yp) = make_uint4(h[0], h[1], h[2], h[3]);
  if (ap) {
    reinterpret_cast<int4*>(ap)[0] = make_int4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<int4*>(ap)[1] = make_int4(v[4], v[5], v[6], v[7]);
  }
}
__device__ __forceinline__ void store_w4a8_4(const int (&v)[4], float st, const __half* sch, __half* yp, int32_t* ap) {
  const uint2 sc = *reinterpret_cast<const uint2*>(sch);
  const __half* sh = reinterpret_cast<const __half*>(&sc);
  uint32_t h[2];
#pragma unroll
  for (int c = 0; c < 4; c += 2) {
    const __half lo = __float2half_rn(__fmul_rn(__fmul_rn((float)v[c], st), __half2float(sh[c])));
    const __half hi = __float2half_rn(__fmul_rn(__fmul_rn((float)v[c + 1], st), __half2float(sh[c + 1])));
    h[c / 2] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
  }
  *reinterpret_cast<uint2*>(yp) = make_uint2(h[0], h[1]);
  if (ap) *reinterpret_cast<int4*>(ap) = make_int4(v[0], v[1], v[2], v[3]);
}

// Stages of a CTA's unit range: a stage is a whole quantization group (two 64-row units) when the
// range holds both halves of it, else a lone unit.  Every role walks the same sequence.
// Tile and row block are tracked incrementally (no division per stage).
struct StageWalk {
  int u, u1, RB, tile, rb;
  __device__ __forceinline__ StageWalk(int u0_, int u1_, int RB_) : u(u0_), u1(u1_), RB(RB_) {
    tile = u0_ / RB_;
    rb = u0_ - tile * RB_;
  }
  // units of the stage starting at u: 2 if u is group-aligned and u + 1 is in the range and tile
  __device__ __forceinline__ int units_here() const {
    return (kUnitsPerStage == 2 && (rb & 1) == 0 && u + 1 < u1 && rb + 1 < RB) ? 2 : 1;
  }
  __device__ __forceinline__ void advance(int nh) {
    u += nh;
    rb += nh;
    if (rb == RB) {
      rb = 0;
      ++tile;
    }
  }
};

// Register cap for one CTA per SM: the 288 threads are 9 warps, so one SM sub-partition (a quarter of
// the 64 K registers) holds three of them.
constexpr int kMaxRegs = (65536 / 4) / (((kThreads / 32 + 3) / 4) * 32) / 8 * 8;
static_assert(kMaxRegs == 168, "9 warps: three on one sub-partition");

// EXACT (8- or 16-token instance): the W4A8 product.  x holds int8 codes widened to fp16, the weights are
// u - 8 with u the packed nibble (the symmetric zero point, unit scales), so every product and every
// fp32 partial sum is an exact integer (the host keeps a CTA's rows of a tile at or below 16384, so
// |sum| <= 1024 * 16384 = 2^24); partials are added as int32 and the output is
// fp16((acc * s_tok[m]) * s_ch[n]), with acc also stored to acc_out when given.
// BF16 (8- or 16-token instance): bf16 activations, scales and output, W = bf16_RN((q - z) s) made
// exactly.
template <int T, bool EXACT, bool BF16 = false>
__global__ void __maxnreg__(kMaxRegs)
gemv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_x,
            const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_s, int has_z,
            __half* __restrict__ y, float* __restrict__ part, int* __restrict__ counters, int* __restrict__ err,
            int M, int N, int RB, int tiles, int maxc, const float* __restrict__ s_tok,
            const __half* __restrict__ s_ch, int32_t* __restrict__ acc_out) {
  static_assert(!EXACT || T == 8 || T == 16, "the exact product has an 8- and a 16-token instance");
  static_assert(!BF16 || !EXACT, "the bf16 variant is a W4A16 instance");
  // fp16 with up to 8 tokens folds zero point and scale into the fp32 sums; the others make every
  // weight exactly (bf16 keeps exact weights at 8 tokens too: its 8-bit weights would not fit the fold).
  // The 8-token W4A8 product folds as well, per 64-row stage, where every sum is an exact integer.
  constexpr bool kFold = T == 8 && !BF16;
  // RB = K / 64 row blocks per tile; unit u = (tile u / RB, row block u % RB); units < 2^31 (host check)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  using G = Geo<T>;
  constexpr int kStageBytes = G::kStageBytes;
  constexpr int kXBoxBytes = G::kXBoxBytes;
  constexpr int kXOff = G::kXOff;
  constexpr int kZOff = G::kZOff;
  constexpr int kSOff = G::kSOff;
  constexpr int kHalves = T / 8;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kStages);
  volatile int* ready_flag = abort_flag + 1;  // the designated tile's partials have all arrived

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int units = tiles * RB;
  const int P = gridDim.x;
  const int p = blockIdx.x;
  const int u0 = (int)unit_begin(p, units, P);
  const int u1 = (int)unit_begin(p + 1, units, P);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + kStages + s); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kConsumers);
    }
    *abort_flag = 0;
    *ready_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    // the next kernel in the stream may launch now; it waits for this grid before touching shared data
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      // the activations' tensor map is read by the first copy after the wait: fetch it now
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
      auto tx_bytes = [&](int nh) {
        return (uint32_t)(nh * (kUnitQBytes + kXBoxBytes) + (has_z ? kZBytes : 0) + (EXACT ? 0 : kSBytes));
      };
      auto issue_weights = [&](int st, int tile, int rb, int nh) {
        const int grp = rb / (kGroup / kRows);
        uint8_t* sb = smem + st * kStageBytes;
        for (int hh = 0; hh < nh; ++hh)
#pragma unroll
          for (int bx = 0; bx < kTileWords / kBoxWords; ++bx)
            tma_load_2d(smem_u32(sb + bx * kColStride + hh * kBoxBytes), &tm_q, tile * kTileWords + bx * kBoxWords,
                        (rb + hh) * kRows, full_bar(st));
        if (has_z) tma_load_2d(smem_u32(sb + kZOff), &tm_z, tile * kTileWords, grp, full_bar(st));
        // scales viewed as int32 pairs: 512 columns = one 256-pair box
        if (!EXACT) tma_load_2d(smem_u32(sb + kSOff), &tm_s, tile * (kTileCols / 2), grp, full_bar(st));
      };
      auto issue_x = [&](int st, int rb, int nh) {
        for (int hh = 0; hh < nh; ++hh)
          tma_load_2d(smem_u32(smem + st * kStageBytes + kXOff + hh * kXBoxBytes), &tm_x, (rb + hh) * kRows, 0,
                      full_bar(st));
      };
      // the first stages' weights stream before the wait on the previous kernel
      StageWalk w(u0, u1, RB);
      int pre = 0;
      int pre_rb[kStages], pre_nh[kStages];
      while (pre < kPrefetch && w.u < u1) {
        const int nh = w.units_here();
        mbar_arrive_tx(full_bar(pre), tx_bytes(nh));
        issue_weights(pre, w.tile, w.rb, nh);
        pre_rb[pre] = w.rb;
        pre_nh[pre] = nh;
        ++pre;
        w.advance(nh);
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      for (int i = 0; i < pre; ++i) issue_x(i, pre_rb[i], pre_nh[i]);
      int issued = pre;
      for (; w.u < u1; ++issued) {
        const int st = issued % kStages;
        const uint32_t ph = (uint32_t)(issued / kStages) & 1u;
        if (!wait_backoff(empty_bar(st), ph ^ 1u, abort_flag, err, 501, kProducerSleepNs)) break;
        const int nh = w.units_here();
        mbar_arrive_tx(full_bar(st), tx_bytes(nh));
        issue_weights(st, w.tile, w.rb, nh);
        issue_x(st, w.rb, nh);
        w.advance(nh);
      }
      // never leave the CTA with copies in flight: the last stages issued must have landed
      volatile int no_abort = 0;
      for (int j = issued - kStages < 0 ? 0 : issued - kStages; j < issued; ++j)
        wait_bounded(full_bar(j % kStages), (uint32_t)(j / kStages) & 1u, &no_abort, err, 502);
    }
  } else {
    // ------------------------------------------------ consumer warps
    const int g = lane >> 2;          // mma group: A rows g / g+8, B column (token) g
    const int t = lane & 3;           // mma thread-in-group
    const int word = warp * 8 + g;    // this lane's packed word column in the tile
    const LaneOffsets lo = lane_offsets<T>(word, g, t);
    bool waited = false;
    int part_tile = -1;               // a shared tile whose partial this CTA wrote (at most one)
    int own_tile = -1;                // the shared tile this CTA completes (it holds its first unit)
    float hold[kHalves][4][4];        // own_tile's sums, kept in registers for its reduction
    bool failed = false;              // a wait ran out: error recorded, the rest of the call skipped
    // zero / scale constants of the current group (cached_grp)
    typename std::conditional<kFold, GroupConsts, GroupConstsH>::type gc;
    int cached_grp = -1;
    int i = 0;                        // stage counter, identical to the producer's
    int cst = 0;                      // its ring slot (i % kStages) and phase ((i / kStages) & 1)
    uint32_t cph = 0;
    StageWalk w(u0, u1, RB);
    while (w.u < u1) {
      const int tile = w.tile;
      float acc[kHalves][4][4];
#pragma unroll
      for (int h = 0; h < kHalves; ++h)
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[h][b][e] = 0.f;
      cached_grp = -1;  // a new tile: other columns
      for (; w.u < u1 && w.tile == tile; ++i) {
        const int nh = w.units_here();
        const int grp = w.rb / (kGroup / kRows);
        w.advance(nh);
        const int st = cst;
        const uint32_t ph = cph;
        if (++cst == kStages) {
          cst = 0;
          cph ^= 1u;
        }
        const uint8_t* sb = smem + st * kStageBytes;
        const bool ok = kConsumerSleepNs ? wait_backoff(full_bar(st), ph, abort_flag, err, 503, kConsumerSleepNs)
                                         : wait_bounded(full_bar(st), ph, abort_flag, err, 503);
        if (!ok) {  // error recorded; this CTA's outputs and tickets are abandoned
          failed = true;
          break;
        }
        if (grp != cached_grp) {  // a stage never spans two groups
          const uint32_t zword = has_z ? reinterpret_cast<const uint32_t*>(sb + kZOff)[word] : 0x88888888u;
          const uint4 sv = EXACT ? make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u)  // 1.0
                                 : reinterpret_cast<const uint4*>(sb + kSOff)[word];
          if constexpr (kFold) group_consts(zword, sv, gc);
          else if constexpr (BF16) group_consts_bf16(zword, sv, gc);
          else group_consts_h(zword, sv, gc);
          cached_grp = grp;
        }
        if constexpr (kFold) {
          float gacc[4][4], sx[4];  // (1024 + q)^T x and sum_k x of this stage (W4A8: of one 64-row block)
          auto clear = [&]() {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              sx[b] = 0.f;
#pragma unroll
              for (int e = 0; e < 4; ++e) gacc[b][e] = 0.f;
            }
          };
          // W4A8 (z = 8, s = 1), per 64-row block: |gacc| <= 64 * 1264 * 128 < 2^24 and |sx| <= 8192 are
          // exact integers (over a whole 128-row group gacc could pass 2^24 with an odd value), so
          // gacc - (1024 + 8 or 1024 + 128) sx = sum (16) (u - 8) x comes out of one fused multiply-add
          // exactly, and the power-of-two scale keeps it exact in acc
          auto fold_exact = [&]() {
#pragma unroll
            for (int b = 0; b < 4; ++b)
#pragma unroll
              for (int e = 0; e < 4; ++e)
                acc[0][b][e] = fmaf((e >> 1) ? 0.0625f : 1.f, fmaf((e >> 1) ? -1152.f : -1032.f, sx[e & 1], gacc[b][e]),
                                    acc[0][b][e]);
          };
          clear();
          StageRegs<8> sr;
          load_stage<8>(sb, 0, lo, sr);
          if (nh == 2) {
            compute_stage(sr, gacc, sx);
            if constexpr (EXACT) {
              fold_exact();
              clear();
            }
            load_stage<8>(sb, 1, lo, sr);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(empty_bar(st));  // slot free before the last unit's arithmetic
          compute_stage(sr, gacc, sx);
          if constexpr (EXACT) {
            fold_exact();
          } else {
            // the group's zero point and scale: acc += s (gacc - (1024 + z) sx)  (high nibble: s / 16, 1024 + 16 z)
#pragma unroll
            for (int b = 0; b < 4; ++b)
#pragma unroll
              for (int e = 0; e < 4; ++e)
                acc[0][b][e] = fmaf(gacc[b][e], gc.sf[b][e >> 1], fmaf(-gc.szc[b][e >> 1], sx[e & 1], acc[0][b][e]));
          }
        } else {
          StageRegs<T> sr;
          load_stage<T>(sb, 0, lo, sr);
          if (nh == 2) {
            compute_stage_exact<T, BF16>(sr, gc, acc);
            load_stage<T>(sb, 1, lo, sr);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(empty_bar(st));  // slot free before the last unit's arithmetic
          compute_stage_exact<T, BF16>(sr, gc, acc);
        }
      }
      if (failed) break;

      // ---- flush: this warp owns its 64 columns; CTAs sharing the tile meet in the workspace
      if (!waited) {
        asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs and workspace of the previous kernel
        waited = true;
      }
      const int pf = (int)cta_of_unit(tile * RB, units, P);
      const int pl = (int)cta_of_unit((tile + 1) * RB - 1, units, P);
      // D fragment of half h: acc[h][b][0/1] = (slot 2b, tokens 8h + 2t / 8h + 2t+1), acc[h][b][2/3] =
      // slot 2b+1: the lane holds all 8 columns of its word for tokens 8h + 2t and 8h + 2t+1, stored as
      // one 16-byte (fp16) or two 16-byte (fp32) vectors per token
      const int n0 = tile * kTileCols + word * 8;
      if (pf == pl) {
#pragma unroll
        for (int hf = 0; hf < kHalves; ++hf)
#pragma unroll
        for (int par = 0; par < 2; ++par) {
          const int m = 8 * hf + 2 * t + par;
          if (EXACT && m < M && n0 < N) {
            int v[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const int sl = slot_of_col(c);
              v[c] = __float2int_rn(acc[hf][sl >> 1][(sl & 1) * 2 + par]);
            }
            store_w4a8(v, s_tok[m], s_ch + n0, y + (size_t)m * N + n0, acc_out ? acc_out + (size_t)m * N + n0 : nullptr);
          } else if (m < M && n0 < N) {  // N % 32 == 0: the word's 8 columns are all in range
            uint32_t h[4];
#pragma unroll
            for (int c = 0; c < 8; c += 2) {
              const int s0 = slot_of_col(c), s1 = slot_of_col(c + 1);
              h[c / 2] = pack2<BF16>(acc[hf][s0 >> 1][(s0 & 1) * 2 + par], acc[hf][s1 >> 1][(s1 & 1) * 2 + par]);
            }
            *reinterpret_cast<uint4*>(y + (size_t)m * N + n0) = make_uint4(h[0], h[1], h[2], h[3]);
          }
        }
      } else if (p == pf) {
        // this CTA holds the tile's first unit, so the tile is the last of its range: it completes
        // the tile after its range, from these registers and the other contributors' partials
#pragma unroll
        for (int hf = 0; hf < kHalves; ++hf)
#pragma unroll
          for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int e = 0; e < 4; ++e) hold[hf][b][e] = acc[hf][b][e];
        own_tile = tile;
      } else {
        float* slot = part + ((size_t)tile * maxc + (size_t)(p - pf)) * T * kTileCols;
#pragma unroll
        for (int hf = 0; hf < kHalves; ++hf)
#pragma unroll
        for (int par = 0; par < 2; ++par) {
          const int m = 8 * hf + 2 * t + par;
          if (m < M) {
            float v[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const int sl = slot_of_col(c);
              v[c] = acc[hf][sl >> 1][(sl & 1) * 2 + par];
            }
            float4* dst = reinterpret_cast<float4*>(slot + m * kTileCols + word * 8);
            dst[0] = make_float4(v[0], v[1], v[2], v[3]);
            dst[1] = make_float4(v[4], v[5], v[6], v[7]);
          }
        }
        part_tile = tile;
      }
    }

    // ---- split K, after the whole range.  A shared tile is completed by the contributor that holds
    // its first unit (pf); every other contributor publishes its partial (fence, then a count on the
    // tile) and is done.  pf waits for the count, adds the partials to its own sums in contributor
    // order and rounds once to fp16, so results are bit-reproducible.  No CTA waits before it has
    // published its own partial, and the grid is at most one CTA per SM, so every wait ends.
    // a timed-out wait in any warp abandons the rest of the call for the whole CTA (every consumer
    // thread takes the same branches below, so the named barriers in them always complete)
    failed = consumers_any(failed);
    if (!failed && part_tile >= 0) {
      consumers_sync();  // every partial store of this CTA issued
      if (threadIdx.x == 0)  // release: the CTA's partial stores (ordered by the barrier) before the count
        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(counters + part_tile) : "memory");
    }
    if (!failed && own_tile >= 0) {
      const int pf = p;
      const int nt = (int)cta_of_unit((own_tile + 1) * RB - 1, units, P) - pf + 1;
      if (threadIdx.x == 0) {
        int* cnt = counters + own_tile;
        const long long t0 = now_ns();
        bool ok = true;
        for (;;) {
          int c;
          asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(c) : "l"(cnt) : "memory");
          if (c == nt - 1) break;
          if (now_ns() - t0 > kWaitLimitNs) {
            if (err) atomicExch(err, 504);
            ok = false;
            break;
          }
        }
        if (ok) *reinterpret_cast<volatile int*>(cnt) = 0;  // every other contributor has counted
        *ready_flag = ok ? 1 : 0;
      }
      // the ring is idle now (every stage consumed): its first slot takes this CTA's own sums in the
      // partials' layout, [token][512 columns] fp32
      float* own = reinterpret_cast<float*>(smem);
      consumers_sync();
#pragma unroll
      for (int hf = 0; hf < kHalves; ++hf)
#pragma unroll
      for (int par = 0; par < 2; ++par) {
        const int m = 8 * hf + 2 * t + par;
        if (m < M) {
          float v[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int sl = slot_of_col(c);
            v[c] = hold[hf][sl >> 1][(sl & 1) * 2 + par];
          }
          float4* dst = reinterpret_cast<float4*>(own + m * kTileCols + word * 8);
          dst[0] = make_float4(v[0], v[1], v[2], v[3]);
          dst[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
      }
      consumers_sync();
      if (*ready_flag) {
        // items (token, 4 columns): up to four per thread at a time, each with eight contributors' loads in
        // flight
        constexpr int kQuads = kTileCols / 4;
        constexpr int kThreadsC = kConsumers * 32;
        const int items = M * kQuads;
        const float4* base = reinterpret_cast<const float4*>(part + (size_t)own_tile * maxc * T * kTileCols);
        constexpr size_t kSlotQuads = (size_t)T * kQuads;
        for (int i0 = threadIdx.x; EXACT && i0 < items; i0 += 4 * kThreadsC) {
          int4 s4[4];  // exact: every partial is an integer below 2^24 in magnitude, their sum need not be
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int it = i0 + k * kThreadsC;
            s4[k] = it < items ? f4_to_i4(reinterpret_cast<const float4*>(own)[it]) : make_int4(0, 0, 0, 0);
          }
          for (int j0 = 1; j0 < nt; j0 += 8) {
            float4 a[4][8];
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const int it = i0 + k * kThreadsC;
                a[k][jj] = (it < items && j0 + jj < nt) ? __ldcg(base + (size_t)(j0 + jj) * kSlotQuads + it)
                                                        : make_float4(0.f, 0.f, 0.f, 0.f);
              }
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const int4 b = f4_to_i4(a[k][jj]);
                s4[k].x += b.x; s4[k].y += b.y; s4[k].z += b.z; s4[k].w += b.w;
              }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int it = i0 + k * kThreadsC;
            if (it >= items) continue;
            const int m = it / kQuads;
            const int n = own_tile * kTileCols + (it - m * kQuads) * 4;
            if (n < N) {
              const int v[4] = {s4[k].x, s4[k].y, s4[k].z, s4[k].w};
              store_w4a8_4(v, s_tok[m], s_ch + n, y + (size_t)m * N + n, acc_out ? acc_out + (size_t)m * N + n : nullptr);
            }
          }
        }
        for (int i0 = threadIdx.x; !EXACT && i0 < items; i0 += 4 * kThreadsC) {
          float4 s4[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int it = i0 + k * kThreadsC;
            s4[k] = it < items ? reinterpret_cast<const float4*>(own)[it] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          for (int j0 = 1; j0 < nt; j0 += 8) {
            float4 a[4][8];
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const int it = i0 + k * kThreadsC;
                a[k][jj] = (it < items && j0 + jj < nt) ? __ldcg(base + (size_t)(j0 + jj) * kSlotQuads + it)
                                                        : make_float4(0.f, 0.f, 0.f, 0.f);
              }
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                s4[k].x += a[k][jj].x; s4[k].y += a[k][jj].y; s4[k].z += a[k][jj].z; s4[k].w += a[k][jj].w;
              }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int it = i0 + k * kThreadsC;
            if (it >= items) continue;
            const int m = it / kQuads;
            const int n = own_tile * kTileCols + (it - m * kQuads) * 4;
            if (n < N) {  // N % 32 == 0: all four outputs are in range
              uint32_t* dst = reinterpret_cast<uint32_t*>(y + (size_t)m * N + n);
              dst[0] = pack2<BF16>(s4[k].x, s4[k].y);
              dst[1] = pack2<BF16>(s4[k].z, s4[k].w);
            }
          }
        }
      }
    }
  }
  __syncthreads();
}


}  // namespace

// SMs of the current device (the grid is at most one CTA per SM, so that every CTA of a call is
// resident together and a tile's completer may wait for its other contributors); GB300's count
// when no device can be queried.
int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return kNumSMs;
  }
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = kNumSMs;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

GemvPlan gemv_plan(int64_t M, int64_t K, int64_t N, int split_k) {
  (void)M;
  GemvPlan p;
  p.tiles = (int)((N / 8 + kTileWords - 1) / kTileWords);
  p.groups = (int)(K / kRows);  // row blocks of 64 (two per quantization group)
  const int64_t units = (int64_t)p.tiles * p.groups;
  const int64_t sms = device_sm_count();
  int64_t ctas;
  if (split_k == 1) {
    ctas = p.tiles;  // one CTA per tile: no tile is shared, so no CTA waits for another
  } else {
    ctas = split_k > 1 ? (int64_t)p.tiles * split_k : sms;
    if (ctas > sms) ctas = sms;  // shared tiles: at most one CTA per SM, all resident together
  }
  if (ctas > units) ctas = units;
  if (ctas < 1) ctas = 1;
  if (p.tiles > kMaxCounters) ctas = p.tiles;  // the tickets would not fit the workspace block
  p.ctas = (int)ctas;
  p.maxc = 1;
  for (int64_t t = 0; t < p.tiles; ++t) {
    const int64_t nt =
        cta_of_unit((t + 1) * p.groups - 1, units, ctas) - cta_of_unit(t * p.groups, units, ctas) + 1;
    if (nt > p.maxc) p.maxc = (int)nt;
  }
  p.split = (int)((ctas + p.tiles - 1) / p.tiles);
  return p;
}

size_t gemv_workspace_bytes(const GemvPlan& p, int64_t M, int64_t N) {
  (void)N;
  if (p.maxc <= 1) return 0;
  const size_t tokens = M <= 8 ? 8 : 16;  // token rows of a partial: the kernel's T
  return kCounterBytes + align256((size_t)p.tiles * p.maxc * tokens * kTileCols * sizeof(float));
}

namespace {

template <int T, bool EXACT, bool BF16 = false>
cudaError_t launch_gemv_t(const uint16_t* x, const uint32_t* qw, const uint32_t* qz, const uint16_t* sc,
                          uint16_t* y, int64_t M, int64_t K, int64_t N, const GemvPlan& p, void* ws, int* err,
                          cudaStream_t s, const float* s_tok = nullptr, const uint16_t* s_ch = nullptr,
                          int32_t* acc_out = nullptr, size_t part_offset = 0) {
  float* part = nullptr;
  int* counters = nullptr;
  if (p.maxc > 1) {
    counters = static_cast<int*>(ws);
    part = reinterpret_cast<float*>(static_cast<char*>(ws) + kCounterBytes + part_offset);
  }
  const uint64_t nw = (uint64_t)N / 8;
  const uint64_t ng = (uint64_t)K / kGroup;
  CUtensorMap tq, tx, tz, ts;
  const bool ok =
      make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, qw, nw, (uint64_t)K, kBoxWords, kRows,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
      make_map_2d(&tx, BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x, (uint64_t)K,
                  (uint64_t)M, kRows, T, CU_TENSOR_MAP_SWIZZLE_128B) &&
      make_map_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, qz ? (const void*)qz : (const void*)qw, nw,
                  qz ? ng : (uint64_t)K, kTileWords, 1, CU_TENSOR_MAP_SWIZZLE_NONE) &&
      (EXACT || make_map_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, sc, (uint64_t)N / 2, ng, kTileCols / 2, 1,
                            CU_TENSOR_MAP_SWIZZLE_NONE));
  if (!ok) return cudaErrorInvalidValue;
  if (EXACT) ts = tq;  // no scale rows are copied
  constexpr int kSmemBytes = Geo<T>::kSmemBytes;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(gemv_kernel<T, EXACT, BF16>), kSmemBytes);
  if (e != cudaSuccess) return e;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)p.ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemv_kernel<T, EXACT, BF16>, tq, tx, tz, ts, qz ? 1 : 0, reinterpret_cast<__half*>(y), part,
                         counters, err, (int)M, (int)N, (int)(K / kRows), p.tiles, p.maxc, s_tok,
                         reinterpret_cast<const __half*>(s_ch), acc_out);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const uint16_t* x, const uint32_t* qw, const uint32_t* qz, const uint16_t* sc,
                        uint16_t* y, int64_t M, int64_t K, int64_t N, const GemvPlan& p, void* ws,
                        int* err, cudaStream_t s, bool bf16) {
  // the kernel counts (tile, 64-row block) units in 32 bits; any tensor that fits a GPU stays far below
  if ((int64_t)p.tiles * p.groups >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  if (bf16) {
    if (M <= 8) return launch_gemv_t<8, false, true>(x, qw, qz, sc, y, M, K, N, p, ws, err, s);
    return launch_gemv_t<16, false, true>(x, qw, qz, sc, y, M, K, N, p, ws, err, s);
  }
  if (M <= 8) return launch_gemv_t<8, false>(x, qw, qz, sc, y, M, K, N, p, ws, err, s);
  return launch_gemv_t<16, false>(x, qw, qz, sc, y, M, K, N, p, ws, err, s);
}

bool gemv_w4a8_ok(const GemvPlan& p, int64_t M) {
  // every CTA's rows of a tile stay within 16384 (256 units of 64 rows), so fp32 sums stay exact
  const int64_t units = (int64_t)p.tiles * p.groups;
  return M >= 1 && M <= kGemvMaxM && (units + p.ctas - 1) / p.ctas <= 256;
}

cudaError_t launch_gemv_w4a8(const uint16_t* x16, const uint32_t* wq, const float* s_tok, const uint16_t* s_ch,
                             uint16_t* y, int32_t* acc_out, int64_t M, int64_t K, int64_t N, const GemvPlan& p,
                             void* ws, int* err, cudaStream_t s) {
  if ((int64_t)p.tiles * p.groups >= ((int64_t)1 << 31) || !gemv_w4a8_ok(p, M)) return cudaErrorInvalidValue;
  // workspace: counters | x16 (the caller's) | partials (sized for 16 token rows; up to 8 tokens the
  // 8-token instance, with half the mma work per stage, uses half of each slot)
  const size_t off = align256((size_t)M * (size_t)K * 2);
  if (M <= 8) return launch_gemv_t<8, true>(x16, wq, nullptr, nullptr, y, M, K, N, p, ws, err, s, s_tok, s_ch, acc_out, off);
  return launch_gemv_t<16, true>(x16, wq, nullptr, nullptr, y, M, K, N, p, ws, err, s, s_tok, s_ch, acc_out, off);
}

}  // namespace awq
