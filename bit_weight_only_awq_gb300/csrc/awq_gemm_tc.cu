// Tensor-core GEMM for the AWQ linear layer (prefill, M > 8) and for W4A8.
//
// Source of the operation: the M > 8 branch of the AWQ dispatch snippet,
// gemmv2_forward_cuda(inputs, qweight, scales, qzeros, group_size, split_k_iters)
// ("Speed up AWQ 2.5x with updated kernel"), and the W4A8 GEMM of "Support W4A8
// quantization for vllm" (int4 weights widened without a scale, per-channel scale
// applied on the output, int32 reduction in a temporary buffer).  Kernel design:
//
//  * Operands are swapped so that the weights are the MMA's A operand: one CTA owns
//    128 output columns (the MMA M dimension) and BT tokens (the MMA N dimension),
//    D^T[n, m] accumulates in tensor memory (fp32, BT columns of 128 lanes).
//  * A packed AWQ word holds 8 consecutive output columns of one input row, which is
//    exactly one 16-byte chunk of an MN-major operand.  Dequant warps therefore turn
//    each word into 8 fp16 values with shifts, one LOP3 per pair (fp16 magic 0x6400),
//    HSUB2 of the zero and HMUL2 of the scale, and store them straight into the
//    128-byte-swizzled MN-major layout; no transposition is needed.
//  * Three shared-memory rings per 64-row k-step, each sized for its own lifetime:
//    packed weights with the group's zero-point / scale rows (TMA, 8 deep, 4.4 KB each:
//    consumed by the dequant warps, so it can run far ahead of DRAM latency), the
//    dequantized fp16 weight tile (3 deep, written by the dequant warps, read by the
//    MMA), and the activation tile (TMA, K-major 128-byte swizzle, as deep as shared
//    memory allows; its slot is held only from the copy to the MMA that reads it).
//    Measured on GB300: with one ring for everything, a slot stayed busy from the copy
//    through dequantization to the MMA (~1.7 us) and four slots capped the tensor
//    pipe at ~45 %.
//  * Warp roles: warp 0 copies activations, warp 2 copies packed weights (TMA), warp 1
//    owns tensor memory and issues tcgen05.mma (one thread), warps 3..18 dequantize in
//    two groups of eight that take alternate k-steps, and the first group then runs the
//    epilogue (tcgen05.ld -> fp16 staged in the idle rings -> one TMA tensor store per
//    M-block; int32 partials go out with plain stores).  Rings are chained by mbarriers;
//    every wait is bounded in time and records an error id instead of hanging.
//  * split > 1: each K slice writes fp32 (W4A16) or int32 (W4A8) partials; the last
//    CTA of an output tile (atomic ticket) sums them in slice order.
//  * W4A8: int8 activations (converted once to fp16, exact) times int4 weights
//    (u - 8, exact in fp16): each product is an integer of magnitude <= 1024 and each
//    slice spans at most 16384 rows, so every fp32 partial sum is an exact integer.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "awq_internal.h"
#include "awq_host.h"
#include "awq_ptx.cuh"

namespace awq {
namespace {

constexpr int kBK = 64;          // input rows per k-step
constexpr int kBN = 128;         // weight columns per MMA (M) = per M-block
constexpr int kDqGroupWarps = 8;              // one group dequantizes one stage (256 threads)
constexpr int kDqGroups = 2;                  // groups alternate stages to overlap their latency
constexpr int kDqWarps = kDqGroupWarps * kDqGroups;
// Dequant warp rank of warp w >= 3 when the warps that share the mma warp's sub-partition (w % 4 == 1)
// are left out of the dequantization.
__device__ __forceinline__ int dq_rank_solo(int w) { return (w - 3) - ((w + 2) / 4 - 1); }
constexpr int kWBlockBytes = kBK * kBN * 2;     // dequantized tile of one M-block, 16 KB

template <int MODE>
constexpr bool kIsW4A8 = MODE == kModeW4A8 || MODE == kModeW4A8One || MODE == kModeW4A8G;
// modes whose k-step stage carries a row of per-(group, column) scales: W4A16 and W4A8 with group factors
template <int MODE>
constexpr bool kHasScales = !kIsW4A8<MODE> || MODE == kModeW4A8G;
// modes with several exact-integer accumulators per K slice (one per chunk of chunk_steps k-steps)
template <int MODE>
constexpr bool kChunked = MODE == kModeW4A8 || MODE == kModeW4A8G;
template <int MODE>
constexpr bool kIsBF16 = MODE == kModeZeroPointBF16 || MODE == kModeSymmetricBF16;
template <int MODE>
constexpr bool kHasZeros = MODE == kModeZeroPoint || MODE == kModeZeroPointBF16;

// NB M-blocks of 128 weight columns share every activation tile: with NB = 2 a CTA owns 256 columns
// and the activation bytes per flop halve (the ring that feeds them was the measured limit at NB = 1).
template <int BT, int NB, int MODE>
struct Cfg {
  static constexpr int kQWords = NB * kBN / 8;          // packed words per row of a stage
  static constexpr int kQBytes = kBK * kQWords * 4;     // packed tile, 4 KB per M-block
  static constexpr int kZBytes = kQWords * 4;           // one zero-point row
  static constexpr int kSBytes = NB * kBN * 2;          // one scale row
  static constexpr int kQStage = kQBytes + 128 + kSBytes;  // packed tile | zero row (padded) | scale row
  static constexpr int kWBytes = NB * kWBlockBytes;
  static constexpr int kQStages = NB == 1 ? 8 : 4;
  static constexpr int kWStages = NB == 1 ? 3 : 2;
  // With 256-token tiles and two M-blocks the activation tile of a k-step arrives as two 32-k halves
  // (64-byte swizzle), each in its own ring slot and released as soon as the mmas that read it are
  // done: the ring is bound by (copy latency + hold time) per slot, and half-size slots hold for half
  // as long (measured +5 %).  With fewer mmas per slot (smaller tiles, one M-block) the per-copy cost
  // wins (measured -10 % for one M-block at 256 tokens).
  static constexpr int kXK = (BT >= 256 && NB == 2) ? 32 : 64;
  static constexpr int kXSub = kBK / kXK;
  static constexpr int kXSlotBytes = BT * kXK * 2;
  static constexpr int kFixed = kWStages * kWBytes + kQStages * kQStage + 2048;
  static constexpr int kFit = (227 * 1024 - 1024 - kFixed) / kXSlotBytes;
  static constexpr int kXStages = kFit > 16 ? 16 : kFit;   // slots
  static constexpr int kSmem = kXStages * kXSlotBytes + kFixed + 1024;
  // W4A8: one accumulator per exact K chunk (two of 16384 rows); with group factors as many 1024-row
  // chunks as tensor memory holds (512 columns)
  // With group factors and 128- or 256-token tiles every finished 1024-row chunk is drained by the
  // dequant warps into an int32 running sum (also in tensor memory, after the accumulators), so a K
  // slice may be any length.  128 tokens: the chunks take turns in two accumulators, the mmas fill one
  // while the other drains; 256 tokens: one accumulator, and the mmas of a chunk wait for the drain of
  // the one before.
  static constexpr bool kDrain = MODE == kModeW4A8G && NB == 1 && (BT == 128 || BT == 256);
  static constexpr int kAccSlots = BT == 128 ? 2 : 1;                 // drain mode
  static constexpr int kDrainLag = kAccSlots == 2 ? 4 : 0;           // k-steps into the next chunk
  static constexpr int kAccs = MODE == kModeW4A8 ? 2 : kDrain ? kAccSlots : MODE == kModeW4A8G ? 512 / (NB * BT) : 1;
  static constexpr int kSumCol = kAccs * NB * BT;  // drain mode: the int32 running sums
  static constexpr int kTmemCols = kDrain ? 512 : NB * kAccs * BT < 32 ? 32 : NB * kAccs * BT;
  // Warps: 0 copies activations, 1 issues the mmas (one thread), 2 copies packed weights, 16 dequantize.
  // With tiles of at most 64 tokens the mmas are short and their issue rate limits the k-step, so
  // the dequant warps skip the mma warp's sub-partition (warp % 4 == 1): 24 warps, of which 4..19 run
  // the epilogue (measured 10-12 % faster at 16-64 tokens, 3-5 % slower with larger tiles).
  static constexpr bool kSoloMma = BT <= 64;
  static constexpr int kWarps = kSoloMma ? 24 : 3 + kDqWarps;
  static constexpr int kThreads = kWarps * 32;
  // tcgen05 instruction descriptor, kind::f16: D f32, A/B both f16 or both bf16 (bits 7-9 / 10-12),
  // A MN-major, B K-major, M=128, N=BT
  static constexpr uint32_t kAB = kIsBF16<MODE> ? ((1u << 7) | (1u << 10)) : 0u;
  static constexpr uint32_t kIdesc = (1u << 4) | kAB | (1u << 15) | ((uint32_t)(BT >> 3) << 17) |
                                     ((uint32_t)(kBN >> 4) << 24);
  static_assert(kXStages >= 2 * kXSub, "activation ring");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  // the epilogue stages each M-block's output tile ([token][128 columns], 16-bit) in the idle rings
  static_assert(kXStages * kXSlotBytes + kWStages * kWBytes >= NB * BT * kBN * 2, "output staging");
  static_assert(kTmemCols <= 512, "tensor memory");
  static_assert(!kDrain || kSumCol + BT <= kTmemCols, "drain layout");
  static_assert(kDrainLag % 2 == 0, "the two dequant groups drain at one even and the next odd k-step");
};

// ------------------------------------------------------------------ tcgen05 mma (A, B from shared memory)
// Shared-memory descriptor of a K-major operand with 64-byte swizzle: rows of 64 bytes, 8-row groups
// 512 bytes apart (layout type 4).
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)(16 >> 4) << 16;
  d |= (uint64_t)(512 >> 4) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)4 << 61;  // 64-byte swizzle
  return d;
}
__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
// pair j of a packed word: (col 2j, col 2j+1) = nibble slots (j, j+4) as fp16 1024 + code
__device__ __forceinline__ uint32_t pair_magic(uint32_t w, int j) {
  return ((w >> (4 * j)) & 0x000F000Fu) | 0x64006400u;
}
// the same pair as bf16 128 + code (exact: 128..143 needs 8 significant bits)
__device__ __forceinline__ uint32_t pair_magic_bf16(uint32_t w, int j) {
  return ((w >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
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
// fp32 output value -> the layer's output format (fp16 or bf16), round to nearest even
template <int MODE>
__device__ __forceinline__ __half out_cvt(float v) {
  if constexpr (kIsBF16<MODE>) return __ushort_as_half(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
  else return __float2half_rn(v);
}

// ------------------------------------------------------------------ kernel
template <int BT, int NB, int MODE>
__global__ void __launch_bounds__(Cfg<BT, NB, MODE>::kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_q,
            const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_s,
            const __grid_constant__ CUtensorMap tm_y,
            __half* __restrict__ y, int32_t* __restrict__ acc_out, const float* __restrict__ s_tok,
            const __half* __restrict__ s_ch, void* __restrict__ part, int* __restrict__ counters,
            int* __restrict__ err, int M, int N, int K, int ksteps_per_split, int chunk_steps, int m_tiles,
            int band) {
  using C = Cfg<BT, NB, MODE>;
  // Accumulators in tensor memory: M-block b of K chunk c at column (c * NB + b) * BT.  W4A8 keeps one
  // per chunk of at most chunk_steps k-steps (16384 rows), each an exact integer in fp32; W4A16 uses
  // one per M-block for its whole K slice.
  constexpr int kTmemCols = C::kTmemCols;
  constexpr int kQStages = C::kQStages;
  constexpr int kWStages = C::kWStages;
  constexpr int kQStage = C::kQStage;
  constexpr int kQBytes = C::kQBytes;
  constexpr int kQWords = C::kQWords;
  constexpr int kWBytes = C::kWBytes;
  constexpr int SX = C::kXStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint8_t* xring = smem;                                   // SX slots of BT x 32 fp16 (1024-aligned)
  uint8_t* wring = xring + SX * C::kXSlotBytes;            // kWStages x NB x 16 KB (1024-aligned)
  uint8_t* qring = wring + kWStages * kWBytes;             // kQStages x kQStage (128-aligned)
  uint64_t* bars = reinterpret_cast<uint64_t*>(qring + kQStages * kQStage);
  // bars: fullx[SX] emptyx[SX] fullq[Q] emptyq[Q] wready[W] wempty[W] accf chunkfull[2] drained[2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * SX + 2 * kQStages + 2 * kWStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* last_flag = reinterpret_cast<int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // output tile of this CTA: bands of `band` token tiles, weight tiles in order within a band and the
  // band's token tiles fastest, so that the CTAs running at once share a few weight tiles and one
  // band of activation tiles (which stays in L2 while the band's weight tiles stream past)
  const int n_tiles = (int)(gridDim.x / (unsigned)m_tiles);
  const int band_id = (int)blockIdx.x / (band * n_tiles);
  const int in_band = (int)blockIdx.x - band_id * band * n_tiles;
  const int band_rows = min(band, m_tiles - band_id * band);
  const int tile_n = in_band / band_rows;
  const int tile_m = band_id * band + (in_band - tile_n * band_rows);
  const int tile_id = tile_m * n_tiles + tile_n;
  const int n0 = tile_n * (NB * kBN);
  const int m0 = tile_m * BT;
  const int total_steps = K / kBK;
  const int step0 = blockIdx.z * ksteps_per_split;
  const int nsteps = min(ksteps_per_split, total_steps - step0);

  auto fullx = [&](int s) { return smem_u32(bars + s); };
  auto emptyx = [&](int s) { return smem_u32(bars + SX + s); };
  auto fullq = [&](int s) { return smem_u32(bars + 2 * SX + s); };
  auto emptyq = [&](int s) { return smem_u32(bars + 2 * SX + kQStages + s); };
  auto wready = [&](int s) { return smem_u32(bars + 2 * SX + 2 * kQStages + s); };
  auto wempty = [&](int s) { return smem_u32(bars + 2 * SX + 2 * kQStages + kWStages + s); };
  const uint32_t accf_bar = smem_u32(bars + 2 * SX + 2 * kQStages + 2 * kWStages);
  // drain mode: an accumulator's chunk is complete (mma commit) / drained (all dequant warps)
  auto chunkfull = [&](int s) { return smem_u32(bars + 2 * SX + 2 * kQStages + 2 * kWStages + 1 + s); };
  auto drained = [&](int s) { return smem_u32(bars + 2 * SX + 2 * kQStages + 2 * kWStages + 3 + s); };
  // drain mode: every chunk but the slice's last is drained into the running sums (group g at its first
  // k-step from (c + 1) chunk_steps + kDrainLag on, or after its loop if it has none); the epilogue adds
  // the last chunk's accumulator
  const int n_chunks = kChunked<MODE> ? (nsteps + chunk_steps - 1) / chunk_steps : 1;
  constexpr int kS = C::kAccSlots;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SX; ++s) {
      mbar_init(fullx(s), 1);
      mbar_init(emptyx(s), 1);
    }
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(fullq(s), 1);
      mbar_init(emptyq(s), kDqGroupWarps);
    }
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(wready(s), kDqGroupWarps);
      mbar_init(wempty(s), 1);
    }
    mbar_init(accf_bar, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(chunkfull(s), 1);
      mbar_init(drained(s), kDqWarps);
    }
    *abort_flag = 0;
    *last_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"((uint32_t)kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched with programmatic dependent launch: the next kernel in the stream may launch now (it waits
  // for this grid before it touches shared data), and this grid's own setup and weight stream overlap
  // the previous kernel.  Only the activation copies (warp 0) and the epilogue, which writes every
  // global result and reads the per-token scales, wait for it.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------ TMA producers: activations (warp 0), weights (warp 2)
    if (lane == 0) {
      const bool is_x = warp == 0;
      if (is_x) asm volatile("griddepcontrol.wait;" ::: "memory");
      const int S = is_x ? SX : kQStages;
      const uint32_t tx = is_x ? (uint32_t)C::kXSlotBytes
                               : (uint32_t)(kQBytes + (kHasZeros<MODE> ? C::kZBytes : 0) +
                                            (kHasScales<MODE> ? C::kSBytes : 0));
      const int units = is_x ? nsteps * C::kXSub : nsteps;  // x: (k-step, 32-k half) slots
      int issued = 0;
      for (int j = 0; j < units; ++j, ++issued) {
        const int st = j % S;
        const uint32_t ph = (uint32_t)(j / S) & 1u;
        if (!wait_bounded(is_x ? emptyx(st) : emptyq(st), ph ^ 1u, abort_flag, err, is_x ? 101 : 102)) break;
        if (is_x) {
          mbar_arrive_tx(fullx(st), tx);
          tma_load_2d(smem_u32(xring + st * C::kXSlotBytes), &tm_x, step0 * kBK + j * C::kXK, m0, fullx(st));
        } else {
          const int kb = (step0 + j) * kBK;
          const int grp = kb / kGroup;
          uint8_t* qb = qring + st * kQStage;
          mbar_arrive_tx(fullq(st), tx);
          tma_load_2d(smem_u32(qb), &tm_q, n0 / 8, kb, fullq(st));
          if (kHasZeros<MODE>) tma_load_2d(smem_u32(qb + kQBytes), &tm_z, n0 / 8, grp, fullq(st));
          if (kHasScales<MODE>) tma_load_2d(smem_u32(qb + kQBytes + 128), &tm_s, n0, grp, fullq(st));
        }
      }
      // never leave the CTA with copies in flight
      volatile int no_abort = 0;
      for (int j = issued - S < 0 ? 0 : issued - S; j < issued; ++j)
        wait_bounded(is_x ? fullx(j % S) : fullq(j % S), (uint32_t)(j / S) & 1u, &no_abort, err, 103);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    // One thread shares its scheduler with four busy dequant warps, and with narrow token tiles its
    // mmas are short, so the loop keeps per-mma work to 64-bit adds on precomputed descriptors (the
    // start address is the low field, in 16-byte units) and tracks ring slots without division.
    if (lane == 0) {
      bool ok = true;
      const uint64_t adesc0 = smem_desc_sw128(smem_u32(wring), 1024, 2048);
      const uint64_t bdesc0 =
          C::kXK == 32 ? smem_desc_sw64(smem_u32(xring)) : smem_desc_sw128(smem_u32(xring), 16, 1024);
      int ws = 0, xs = 0, chunk = 0, within = 0;
      uint32_t wph = 0, xph = 0;
      for (int it = 0; it < nsteps && ok; ++it) {
        if (C::kDrain && within == 0 && chunk >= kS) {
          // the accumulator of chunk - kS must have been drained before this chunk overwrites it
          ok = wait_bounded(drained(chunk % kS), (uint32_t)((chunk - kS) / kS) & 1u, abort_flag, err, 204);
          if (!ok) break;
          tc_fence_after();
        }
        ok = wait_bounded(wready(ws), wph, abort_flag, err, 202);
        const uint64_t ad_s = adesc0 + (uint64_t)((ws * kWBytes) >> 4);
        for (int h = 0; h < C::kXSub && ok; ++h) {
          ok = wait_bounded(fullx(xs), xph, abort_flag, err, 201);
          if (!ok) break;
          tc_fence_after();
          const uint64_t bd_s = bdesc0 + (uint64_t)((xs * C::kXSlotBytes) >> 4);
#pragma unroll
          for (int k2 = 0; k2 < C::kXK / 16; ++k2) {
            const int kk = h * (C::kXK / 16) + k2;
            // B: activations, K-major; 16 k = 32 B inside the 64- or 128-byte swizzle row
            const uint64_t bd = bd_s + (uint64_t)(k2 * 2);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              // A: weights of M-block b, MN-major; 64-column atoms 1024 B apart (LBO), 8-row k groups
              // 2048 B apart (SBO); k16 step kk starts 4096 B further
              const uint64_t ad = ad_s + (uint64_t)((b * kWBlockBytes + kk * 4096) >> 4);
              const int acc = C::kDrain ? chunk % kS : chunk;
              mma_f16(tmem + (uint32_t)((acc * NB + b) * BT), ad, bd, C::kIdesc, (within > 0 || kk > 0) ? 1u : 0u);
            }
          }
          mma_commit(emptyx(xs));  // this part of the activation tile is free once its mmas have read it
          if (++xs == SX) {
            xs = 0;
            xph ^= 1u;
          }
        }
        if (ok) mma_commit(wempty(ws));
        if (++ws == kWStages) {
          ws = 0;
          wph ^= 1u;
        }
        ++within;  // k-steps accumulated into the current chunk (W4A16: one chunk)
        if (kChunked<MODE> && within == chunk_steps) {
          if (C::kDrain && chunk < n_chunks - 1) mma_commit(chunkfull(chunk % kS));  // to be drained
          within = 0;
          ++chunk;
        }
      }
      mma_commit(accf_bar);  // arrives once every issued mma has completed
      volatile int no_abort = 0;
      wait_bounded(accf_bar, 0, &no_abort, err, 203);
    }
  } else {
    // ------------------------------------------------ dequant warps (two groups, alternate k-steps)
    int group = (threadIdx.x - 96) / (kDqGroupWarps * 32);
    int d = (threadIdx.x - 96) % (kDqGroupWarps * 32);  // 0..255 within the group
    if (C::kSoloMma) {
      const int rk = dq_rank_solo(warp);
      group = rk / kDqGroupWarps;
      d = (rk % kDqGroupWarps) * 32 + lane;
    }
    constexpr int kRowsPerPass = kDqGroupWarps * 32 / kQWords;  // 16 (NB = 1) or 8 (NB = 2)
    constexpr int kPasses = kBK / kRowsPerPass;                   // rows per thread: 4 NB
    const int c = d % kQWords;       // packed word column within the tile (M-block c / 16)
    const int r0 = d / kQWords;      // first of the thread's rows (r0 + kRowsPerPass j)
    const int cw = c & 15;           // word column within its M-block
    const uint32_t blk_off = (uint32_t)((c >> 4) * kWBlockBytes);
    // drain mode: warp w adds its TMEM lane quarter (w % 4) of token quarter (w - 3) / 4 of chunk ch's
    // accumulator into the running sums, as exact integers, then arrives on drained
    int next_drain = 0;
    auto drain = [&](int ch) -> bool {
      if (!wait_bounded(chunkfull(ch % kS), (uint32_t)(ch / kS) & 1u, abort_flag, err, 303)) return false;
      tc_fence_after();
      const uint32_t lanes = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      const uint32_t col = (uint32_t)(((warp - 3) >> 2) * (BT / 4));
#pragma unroll
      for (int h = 0; h < BT / 64; ++h) {
        uint32_t v[16], s[16];
        tmem_ld16_nowait(lanes + (uint32_t)((ch % kS) * BT) + col + 16 * h, v);
        if (ch > 0) tmem_ld16_nowait(lanes + (uint32_t)C::kSumCol + col + 16 * h, s);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          s[j] = (uint32_t)((ch > 0 ? (int)s[j] : 0) + __float2int_rn(__uint_as_float(v[j])));
        tmem_st16(lanes + (uint32_t)C::kSumCol + col + 16 * h, s);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(drained(ch % kS));
      return true;
    };
    for (int it = (C::kSoloMma && warp % 4 == 1) ? nsteps : group; it < nsteps; it += kDqGroups) {
      const int qs = it % kQStages, ws = it % kWStages;
      if (!wait_bounded(fullq(qs), (uint32_t)(it / kQStages) & 1u, abort_flag, err, 301)) break;
      if (!wait_bounded(wempty(ws), ((uint32_t)(it / kWStages) & 1u) ^ 1u, abort_flag, err, 302)) break;
      const uint8_t* qb = qring + qs * kQStage;
      const uint32_t* qw = reinterpret_cast<const uint32_t*>(qb);
      uint8_t* wt = wring + ws * kWBytes;
      uint32_t zp[4], sp[4];
      if (kHasScales<MODE>) {
        const uint32_t zword = kHasZeros<MODE> ? reinterpret_cast<const uint32_t*>(qb + kQBytes)[c]
                                               : 0x88888888u;
        const uint4 sv = reinterpret_cast<const uint4*>(qb + kQBytes + 128)[c];
        sp[0] = sv.x; sp[1] = sv.y; sp[2] = sv.z; sp[3] = sv.w;
#pragma unroll
        for (int j = 0; j < 4; ++j) zp[j] = kIsBF16<MODE> ? pair_magic_bf16(zword, j) : pair_magic(zword, j);
      }
      uint32_t words[kPasses];
#pragma unroll
      for (int jr = 0; jr < kPasses; ++jr) words[jr] = qw[(r0 + kRowsPerPass * jr) * kQWords + c];
      __syncwarp();
      if (lane == 0) mbar_arrive(emptyq(qs));  // packed words are in registers: the slot can refill
#pragma unroll
      for (int jr = 0; jr < kPasses; ++jr) {
        const int r = r0 + kRowsPerPass * jr;
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if constexpr (kIsBF16<MODE>) {
            o[j] = bmul2(bsub2(pair_magic_bf16(words[jr], j), zp[j]), sp[j]);
          } else {
            const uint32_t h = pair_magic(words[jr], j);
            if constexpr (MODE == kModeW4A8G) o[j] = hmul2(hsub2(h, 0x64086408u), sp[j]);  // (u - 8) s3, exact
            else o[j] = kIsW4A8<MODE> ? hsub2(h, 0x64086408u) /* u - 8, exact */
                                      : hmul2(hsub2(h, zp[j]), sp[j]);
          }
        }
        const uint32_t off =
            blk_off + (uint32_t)((r >> 3) * 2048 + (cw >> 3) * 1024 + (r & 7) * 128 + (((cw & 7) ^ (r & 7)) << 4));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(wt + off)), "r"(o[0]), "r"(o[1]),
                     "r"(o[2]), "r"(o[3])
                     : "memory");
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(wready(ws));
      if constexpr (C::kDrain) {
        // chunk ch is drained by group 0 after it has dequantized k-step (ch + 1) chunk_steps + kDrainLag
        // and by group 1 after the step that follows (with one accumulator: after the first two k-steps
        // of the next chunk, whose mmas wait for the drain; their weights are then already in the ring)
        const int rel = it - C::kDrainLag - group;
        if (rel >= chunk_steps && rel % chunk_steps == 0 && rel / chunk_steps - 1 == next_drain &&
            next_drain < n_chunks - 1) {
          if (!drain(next_drain)) break;
          ++next_drain;
        }
      }
    }
    // drain mode: chunks whose drain step this warp's group never reached
    if constexpr (C::kDrain)
      while (next_drain < n_chunks - 1 && drain(next_drain)) ++next_drain;

    // ------------------------------------------------ epilogue (dequant group b reads M-block b)
    if (C::kSoloMma) {  // warps 4..19
      group = warp >= 4 ? (warp - 4) / kDqGroupWarps : NB;
      d = ((warp - 4) % kDqGroupWarps) * 32 + lane;
    }
    if (group < NB) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs, workspace and s_tok of the previous kernels
    bool have = wait_bounded(accf_bar, 0, abort_flag, err, 401);
    // drain mode: the running sums are complete once the slice's next-to-last chunk is drained
    if (C::kDrain && have && n_chunks > 1)
      have = wait_bounded(drained((n_chunks - 2) % kS), (uint32_t)((n_chunks - 2) / kS) & 1u, abort_flag, err, 402);
    tc_fence_after();
    const int lq = warp & 3;                 // TMEM lane quarter this warp may access
    const int half = ((warp - (C::kSoloMma ? 4 : 3)) & 7) >> 2;  // which half of the BT token columns
    const int nl = lq * 32 + lane;           // TMEM lane = weight column in the M-block
    const int n = n0 + group * kBN + nl;
    const uint32_t dcol = (uint32_t)(group * BT);  // this M-block's accumulator
    const bool n_ok = n < N;
    const int split = gridDim.z;
    constexpr int kHalf = BT / 2;
    float sch = 0.f;
    if (kIsW4A8<MODE> && n_ok) sch = __half2float(s_ch[n]);
    // without a K split the outputs are staged in the idle rings, [token][128 columns] per M-block, for
    // one tensor store per M-block
    __half* stg = reinterpret_cast<__half*>(xring) + (size_t)group * BT * kBN;
    if (have) {
#pragma unroll 1
      for (int cb = half * kHalf; cb < (half + 1) * kHalf; cb += 8) {
        float v[8];
        int vi[8];
        if constexpr (C::kDrain) {
          // the running sums of the drained chunks, then the accumulator of the slice's last chunk
          const uint32_t lanes = tmem + ((uint32_t)(lq * 32) << 16);
#pragma unroll
          for (int j = 0; j < 8; ++j) vi[j] = 0;
          if (n_chunks > 1) {
            tmem_ld8(lanes + (uint32_t)(C::kSumCol + cb), v);
#pragma unroll
            for (int j = 0; j < 8; ++j) vi[j] = __float_as_int(v[j]);
          }
          tmem_ld8(lanes + (uint32_t)(((n_chunks - 1) % kS) * BT + cb), v);
#pragma unroll
          for (int j = 0; j < 8; ++j) vi[j] += __float2int_rn(v[j]);
        } else {
          tmem_ld8(tmem + ((uint32_t)(lq * 32) << 16) + dcol + (uint32_t)cb, v);
          if (kIsW4A8<MODE>) {
#pragma unroll
            for (int j = 0; j < 8; ++j) vi[j] = __float2int_rn(v[j]);  // exact integers
            // the other chunks' accumulators, each an exact integer, added as int32
            for (int ch = 1; kChunked<MODE> && ch < C::kAccs && ch * chunk_steps < nsteps; ++ch) {
              float v2[8];
              tmem_ld8(tmem + ((uint32_t)(lq * 32) << 16) + dcol + (uint32_t)(ch * NB * BT + cb), v2);
#pragma unroll
              for (int j = 0; j < 8; ++j) vi[j] += __float2int_rn(v2[j]);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int m = m0 + cb + j;
          const bool in = n_ok && m < M;
          const size_t o = (size_t)m * N + n;
          if (split == 1) {
            __half hv;  // rows and columns beyond the tensor are staged too; the tensor store clips them
            if constexpr (kIsW4A8<MODE>) {
              if (acc_out && in) __stcs(acc_out + o, vi[j]);
              hv = __float2half_rn(in ? __fmul_rn(__fmul_rn((float)vi[j], s_tok[m]), sch) : 0.f);
            } else {
              hv = out_cvt<MODE>(v[j]);
            }
            stg[(cb + j) * kBN + nl] = hv;
          } else if (in) {
            if constexpr (kIsW4A8<MODE>) reinterpret_cast<int32_t*>(part)[(size_t)blockIdx.z * M * N + o] = vi[j];
            else reinterpret_cast<float*>(part)[(size_t)blockIdx.z * M * N + o] = v[j];
          }
        }
      }
    }
    if (split == 1) {
      // this group's tile out in one tensor store, after its staging writes are visible to the async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("bar.sync %0, %1;" ::"r"(2 + group), "r"(kDqGroupWarps * 32) : "memory");
      if (d == 0 && have) {
        tma_store_2d(&tm_y, smem_u32(stg), n0 + group * kBN, m0);
        bulk_commit();
        bulk_wait_read0();  // the staged tile has been read before this thread reaches the exit barrier
      }
    }
    if (split > 1) {
      __threadfence();
      asm volatile("bar.sync 1, %0;" ::"r"(NB * kDqGroupWarps * 32) : "memory");  // the epilogue groups
      if (group == 0 && d == 0) {
        const int ctr = tile_id;
        *last_flag = (atomicAdd(counters + ctr, 1) == split - 1);
      }
      asm volatile("bar.sync 1, %0;" ::"r"(NB * kDqGroupWarps * 32) : "memory");
      if (*last_flag) {
        __threadfence();
        // the split slices of kChunk tokens, two slices at a time, all their loads in flight together;
        // each sum still runs over the slices in order (0 + s0 + s1 + ...)
        constexpr int kChunk = kHalf < 8 ? kHalf : 8;
        using P = typename std::conditional<kIsW4A8<MODE>, int32_t, float>::type;
        const P* pp = reinterpret_cast<const P*>(part);
        const size_t slice = (size_t)M * N;
        for (int cb0 = half * kHalf; n_ok && cb0 < (half + 1) * kHalf && m0 + cb0 < M; cb0 += kChunk) {
          P a[kChunk];
#pragma unroll
          for (int j = 0; j < kChunk; ++j) a[j] = P(0);
          for (int sp = 0; sp < split; sp += 2) {
            P v0[kChunk], v1[kChunk];
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
              const int m = m0 + cb0 + j;
              const size_t o = (size_t)m * N + n;
              v0[j] = m < M ? __ldcg(pp + (size_t)sp * slice + o) : P(0);
              v1[j] = (m < M && sp + 1 < split) ? __ldcg(pp + (size_t)(sp + 1) * slice + o) : P(0);
            }
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
              a[j] += v0[j];
              if (sp + 1 < split) a[j] += v1[j];
            }
          }
#pragma unroll
          for (int j = 0; j < kChunk; ++j) {
            const int m = m0 + cb0 + j;
            if (m >= M) break;
            const size_t o = (size_t)m * N + n;
            if constexpr (kIsW4A8<MODE>) {
              if (acc_out) __stcs(acc_out + o, a[j]);
              __stcs(y + o, __float2half_rn(__fmul_rn(__fmul_rn((float)a[j], s_tok[m]), sch)));
            } else {
              __stcs(y + o, out_cvt<MODE>(a[j]));
            }
          }
        }
        if (group == 0 && d == 0) atomicExch(counters + tile_id, 0);
      }
    }
  }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host side

template <int BT, int NB, int MODE>
cudaError_t launch_t(const uint16_t* x16, const uint32_t* qw, const uint32_t* qz, const uint16_t* sc,
                     const float* s_tok, const uint16_t* s_ch, uint16_t* y, int32_t* acc_out, int64_t M,
                     int64_t K, int64_t N, const GemmPlan& p, void* part, int* counters, int* err,
                     cudaStream_t s) {
  using C = Cfg<BT, NB, MODE>;
  constexpr int kQWords = C::kQWords;
  CUtensorMap tx, tq, tz, ts, ty;
  const uint64_t nw = (uint64_t)N / 8, ng = (uint64_t)K / kGroup;
  constexpr CUtensorMapDataType kHalfType = kIsBF16<MODE> ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  bool ok = make_map_2d(&tx, kHalfType, 2, x16, (uint64_t)K, (uint64_t)M, C::kXK, BT,
                        C::kXK == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, qw, nw, (uint64_t)K, kQWords, kBK,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
  // zero-point and scale maps: dummies (the weight map) when the mode does not read them
  ok = ok && make_map_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, qz ? (const void*)qz : (const void*)qw, nw,
                         qz ? ng : (uint64_t)K, kQWords, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
  ok = ok && (!kHasScales<MODE>
                  ? make_map_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, qw, nw, (uint64_t)K, kQWords, 1,
                                CU_TENSOR_MAP_SWIZZLE_NONE)
                  : make_map_2d(&ts, kHalfType, 2, sc, (uint64_t)N, ng, NB * kBN, 1,
                                CU_TENSOR_MAP_SWIZZLE_NONE));
  // output map: [M, N] 16-bit, boxes of one M-block's 128 columns x BT tokens (the epilogue's tensor stores)
  ok = ok && make_map_2d(&ty, kHalfType, 2, y, (uint64_t)N, (uint64_t)M, kBN, BT, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!ok) return cudaErrorInvalidValue;
  auto kern = gemm_kernel<BT, NB, MODE>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), C::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)(p.n_tiles * p.m_tiles), 1, p.split);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, tx, tq, tz, ts, ty, reinterpret_cast<__half*>(y), acc_out, s_tok,
                         reinterpret_cast<const __half*>(s_ch), part, counters, err, (int)M, (int)N, (int)K,
                         p.ksteps, (MODE == kModeW4A8G ? kW4A8GroupChunk : kW4A8MaxKSlice) / kBK, p.m_tiles,
                         p.band);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_mode(const uint16_t* x16, const uint32_t* qw, const uint32_t* qz, const uint16_t* sc,
                        const float* s_tok, const uint16_t* s_ch, uint16_t* y, int32_t* acc_out, int64_t M,
                        int64_t K, int64_t N, const GemmPlan& p, void* part, int* counters, int* err,
                        cudaStream_t s) {
  if (p.nb == 2) {
    // W4A8 with two M-blocks: the plan keeps every K slice within one exact chunk
    constexpr int M2 = MODE == kModeW4A8 ? kModeW4A8One : MODE;
    if (MODE == kModeW4A8 && p.ksteps * kBK > kW4A8MaxKSlice) return cudaErrorInvalidValue;
    switch (p.bt) {
      case 64: return launch_t<64, 2, M2>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
      case 128: return launch_t<128, 2, M2>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
      case 256: return launch_t<256, 2, M2>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if (p.nb != 1) return cudaErrorInvalidValue;
  if constexpr (MODE == kModeW4A8G) {
    // token tiles of at most 64: 8 to 32 chunk accumulators hold a K slice; 128: two, drained in turn
    if (p.bt <= 64 && (int64_t)p.ksteps * kBK > (int64_t)(512 / p.bt) * kW4A8GroupChunk) return cudaErrorInvalidValue;
    switch (p.bt) {
      case 128: return launch_t<128, 1, MODE>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
      case 256: return launch_t<256, 1, MODE>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
      case 16: return launch_t<16, 1, MODE>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
      case 32: return launch_t<32, 1, MODE>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
      case 64: return launch_t<64, 1, MODE>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (p.bt) {
    case 16: return launch_t<16, 1, MODE>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
    case 32: return launch_t<32, 1, MODE>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
    case 64: return launch_t<64, 1, MODE>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
    case 128: return launch_t<128, 1, MODE>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
    case 256: return launch_t<256, 1, MODE>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

namespace {

// The split that fills one wave of 152 CTAs (largest split <= 8 with at least min_slice k-steps per
// slice), 1 if the unsplit grid already has a wave.
int fill_split(int64_t tiles, int total_k, int min_slice) {
  int sp = 1;
  if (tiles < 152 && tiles <= kMaxCounters)
    for (int s = 2; s <= 8; ++s)
      if (tiles * s <= 152 && total_k / s >= min_slice) sp = s;
  return sp;
}

// Modelled time (us) of a GEMM call: waves of one CTA per SM, each running its K slice at a per-k-step
// time that grows with the tile (128-column M-blocks x token tile), plus a fixed cost and, with a K
// split, the partials' reduction: a term that grows with the bytes each tile's last CTA reads, and the
// partials' DRAM time (written and read once at 6 TB/s).  The constants are a least-squares fit to
// timings of every (token tile, M-blocks, split) plan on the prefill and crossover shapes (K = 4096 /
// 14336, N = 4096 .. 28672, 64 .. 4096 tokens) on GB300; the plan picked by the fit was within 6.5 % of
// the best measured one on all of them, and picked the best measured plan for per-channel W4A8
// (K = 21760, N = 8192) at 256, 1024 and 4096 tokens.  The step of 64-token tiles with two M-blocks
// (0.62 us) was measured separately (gate_up, 64 tokens, one wave).
double gemm_plan_cost(int64_t M, int64_t N, int total, int bt, int nb, int split) {
  const int ks = (total + split - 1) / split;
  const int sp = (total + ks - 1) / ks;
  const int64_t tiles = ((N + (int64_t)nb * kBN - 1) / ((int64_t)nb * kBN)) * ((M + bt - 1) / bt);
  const int64_t waves = (tiles * sp + 151) / 152;
  double step = nb == 2 ? 0.62 : 0.358;  // 64 tokens
  if (bt == 128) step = nb == 2 ? 0.603 : 0.451;
  if (bt == 256) step = nb == 2 ? 0.804 : 0.560;
  double t = (double)waves * ks * step + 10.31;
  if (sp > 1) t += 7.43 + 7.05 * (sp - 1) * bt * nb / 512.0 + 2.0 * sp * (double)M * (double)N * 4.0 / 6.0e6;
  return t;
}

}  // namespace

GemmPlan gemm_plan(int64_t M, int64_t K, int64_t N, int split_k, int mode) {
  GemmPlan p;
  const int bt0 = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
  const int total = (int)(K / kBK);
  auto tiles = [&](int bt, int nb) {
    return ((N + (int64_t)nb * kBN - 1) / ((int64_t)nb * kBN)) * ((M + bt - 1) / bt);
  };
  // 128 weight columns per CTA; under one wave of 152 SMs, narrower token tiles (down to 64) before
  // splitting K
  p.nb = 1;
  p.bt = bt0;
  while (p.bt > 64 && tiles(p.bt, 1) < 114) p.bt /= 2;
  // with group factors: at most 64 tokens keep every 1024-row chunk accumulator of a K slice in tensor
  // memory (512 / 64 = 8); 128 and 256 tokens drain their chunks during the main loop
  // >= 128-token tiles: 256 weight columns per CTA (two M-blocks on one activation tile) whenever that
  // still fills about a wave.  W4A8 then has one exact accumulator per M-block, which holds K slices of
  // at most 16384 rows: taken here only when K fits one slice (the cost model below may still choose two
  // M-blocks with a K split: at K = 21760 and 4096 tokens that measured 1132 us against 1263 us for one
  // M-block with two accumulators)
  if (bt0 >= 128 && mode != kModeW4A8G && (mode != kModeW4A8 || K <= kW4A8MaxKSlice)) {
    int bt = bt0;
    while (bt > 128 && tiles(bt, 2) < 114) bt /= 2;
    // under a wave, a K split with slices of at least 32 k-steps may fill it (M = 256, K = 14336,
    // N = 4096: 104 -> 76 us); shorter slices measured slower than one M-block without a split
    // (K = 4096, N = 4096: 31 -> 37 us with slices of 16), except where one M-block needs a second
    // wave: W4A16 then takes slices of 16 (M = 256, K = 4096, N = 6144: 58 -> 39 us)
    const int64_t waves1 = (tiles(p.bt, 1) + 151) / 152;
    const int min_slice = (mode != kModeW4A8 && waves1 > 1) ? 16 : 32;
    const int sp_fill = split_k > 0 ? 1 : fill_split(tiles(bt, 2), total, min_slice);
    if (tiles(bt, 2) * sp_fill >= 114) {
      p.nb = 2;
      p.bt = bt;
    }
  }
  p.n_tiles = (int)((N + (int64_t)p.nb * kBN - 1) / ((int64_t)p.nb * kBN));
  p.m_tiles = (int)((M + p.bt - 1) / p.bt);
  // fill the 152 SMs: largest split (<= 8, >= 8 k-steps per slice) whose CTA count stays <= one wave,
  // if the unsplit grid is under one wave
  int split = split_k > 0 ? split_k : fill_split((int64_t)p.n_tiles * p.m_tiles, total, 8);
  if (mode == kModeW4A8 || (mode == kModeW4A8G && p.bt <= 64)) {
    // exact accumulators: each K slice spans at most 2 x 16384 rows with one M-block (two
    // accumulators), at most 16384 with two M-blocks (one each); with group factors and at most 64
    // tokens, 512 / bt chunks of 1024 rows
    const int64_t slice = mode == kModeW4A8G ? (int64_t)(512 / p.bt) * kW4A8GroupChunk
                                             : (p.nb == 2 ? kW4A8MaxKSlice : 2 * kW4A8MaxKSlice);
    const int min_split = (int)((K + slice - 1) / slice);
    if (split < min_split) split = min_split;
  }
  if (split > total) split = total;
  if (split < 1) split = 1;
  p.ksteps = (total + split - 1) / split;
  p.split = (total + p.ksteps - 1) / p.ksteps;
  // Above 64 tokens with an automatic split: the plan that the measured cost model (below) rates at
  // least 5 % faster replaces the one above; for per-channel W4A8 only plans whose K slices keep the
  // exact accumulators (16384 rows with two M-blocks, 2 x 16384 with one), with group factors only the
  // chunk-draining tiles (128 or 256 tokens, one M-block).  Up to 32 tokens the rules above stand (the
  // model knows tiles of 64 tokens and more).
  const bool w4a16 = mode == kModeZeroPoint || mode == kModeSymmetric || mode == kModeZeroPointBF16 ||
                     mode == kModeSymmetricBF16;
  if ((w4a16 || mode == kModeW4A8 || mode == kModeW4A8G) && split_k == 0 && M > 32) {
    const double cur = gemm_plan_cost(M, N, total, p.bt, p.nb, p.split);
    double best = cur;
    int bbt = p.bt, bnb = p.nb, bsp = p.split;
    for (int bt = 64; bt <= bt0; bt *= 2)
      for (int nb = 1; nb <= 2; ++nb)
        for (int sp = 1; sp <= 8; ++sp) {
          if (total / sp < 8) break;
          const int64_t tl = tiles(bt, nb);
          if (sp > 1 && tl > kMaxCounters) break;
          if (mode == kModeW4A8G && (bt < 128 || nb != 1)) continue;
          if (mode == kModeW4A8) {
            const int64_t rows = (int64_t)((total + sp - 1) / sp) * kBK;
            if (nb == 2 && rows > kW4A8MaxKSlice) continue;
            if (rows > 2 * kW4A8MaxKSlice) continue;
          }
          const double c = gemm_plan_cost(M, N, total, bt, nb, sp);
          if (c < best) {
            best = c;
            bbt = bt;
            bnb = nb;
            bsp = sp;
          }
        }
    if (best < 0.95 * cur) {
      p.bt = bbt;
      p.nb = bnb;
      p.n_tiles = (int)((N + (int64_t)p.nb * kBN - 1) / ((int64_t)p.nb * kBN));
      p.m_tiles = (int)((M + p.bt - 1) / p.bt);
      p.ksteps = (total + bsp - 1) / bsp;
      p.split = (total + p.ksteps - 1) / p.ksteps;
    }
  }
  // raster band: as many token tiles as keep their activation tiles (fp16, a K slice each) within about
  // a third of the 126 MB L2, so that they stay resident while the weight tiles stream past
  const int64_t x_tile = (int64_t)p.bt * p.ksteps * kBK * 2;
  int64_t band = kRasterBandBytes / (x_tile > 0 ? x_tile : 1);
  if (band > p.m_tiles) band = p.m_tiles;
  if (band < 1) band = 1;
  p.band = (int)band;
  return p;
}

// Workspace: [tile counters, kCounterBytes] [W4A8: fp16 copy of the codes] [split partials]
size_t gemm_workspace_bytes(const GemmPlan& p, int64_t M, int64_t K, int64_t N, int mode) {
  const size_t x16 = (mode == kModeW4A8 || mode == kModeW4A8G) ? align256((size_t)M * (size_t)K * 2) : 0;
  const size_t part = p.split > 1 ? align256((size_t)p.split * (size_t)M * (size_t)N * 4) : 0;
  if (x16 == 0 && part == 0) return 0;
  return kCounterBytes + x16 + part;
}

cudaError_t launch_gemm(int mode, const uint16_t* x16, const uint32_t* qw, const uint32_t* qz, const uint16_t* sc,
                        const float* s_tok, const uint16_t* s_ch, uint16_t* y, int32_t* acc_out, int64_t M,
                        int64_t K, int64_t N, const GemmPlan& p, void* part, int* counters, int* err,
                        cudaStream_t s) {
  switch (mode) {
    case kModeZeroPoint:
      return launch_mode<kModeZeroPoint>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
    case kModeSymmetric:
      return launch_mode<kModeSymmetric>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
    case kModeW4A8:
      return launch_mode<kModeW4A8>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
    case kModeW4A8G:
      return launch_mode<kModeW4A8G>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters, err, s);
    case kModeZeroPointBF16:
      return launch_mode<kModeZeroPointBF16>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters,
                                             err, s);
    case kModeSymmetricBF16:
      return launch_mode<kModeSymmetricBF16>(x16, qw, qz, sc, s_tok, s_ch, y, acc_out, M, K, N, p, part, counters,
                                             err, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace awq
