// Decode GEMV on a prepared copy of the weights: y[m, n] = sum_k x[m, k] * W[k, n] for M <= 8 tokens,
// plus the kernels that prepare that copy from the AWQ format and turn it back.
//
// Source of the operation: the M <= 8 branch of the AWQ dispatch snippet, gemv_forward_cuda(inputs,
// qweight, scales, qzeros, group_size) ("Speed up AWQ 2.5x with updated kernel"); the offline shuffle
// of the int4 weights so that each thread of a warp fetches what it needs ("Support W4A8 quantization
// for vllm", HandH1998 on the 8 INT4 weights of one INT32 shuffled offline).  The design is this
// library's own:
//
//  * Prepared layout (awq_prepack_gemv): one (256-column tile, 128-row group) unit per 17024-byte
//    block, units tile-major.  A block holds the group's codes as the words the mma lanes read
//    (16 KB: word (warp w, 16-row step i, lane l, column pair b) carries rows 2t, 2t+1, 2t+8, 2t+9 of
//    columns 64 w + 8 g + 2 b and + 1, g = l / 4, t = l % 4), then the zero points (one word of 8
//    nibbles per (w, g)) and the scales (8 halves per (w, g)) of the group in column order.  A CTA's
//    range of units is one contiguous run of memory, so every stage is a single bulk copy whatever
//    the tile width (the AWQ layout gives 128-byte row runs at this width), and a lane's 8 output
//    columns are consecutive.
//  * Each 32-bit word yields the four A registers of one m16n8k16 mma with four LOP3s and one
//    shift (no byte permutes): the low nibbles of its bytes are the even column, the high nibbles
//    the odd column (exact fp16 halves 1024 + q and 1024 + 16 q).  The group's zero point and scale
//    are applied once per group and column to fp32 sums, as in the AWQ-layout kernel:
//        sum_k (q - z) s x = s (sum_k (1024 + q) x - (1024 + z) sum_k x).
//  * Residency: 4 consumer warps (64 columns each) and 1 producer warp per CTA, a 5-stage ring of
//    19 KB, at most 168 registers: two CTAs fit on one SM.  Launched with programmatic dependent
//    launch, the next call's CTAs therefore become resident while this call's CTAs still run, and
//    stream their first two weight stages into shared memory before they wait for this call
//    (weights do not depend on it); only the activations, outputs and workspace wait.
//  * Split K as in the AWQ-layout kernel: a tile shared by several CTAs is completed by the CTA
//    holding its first group, which waits (bounded) for the others' fp32 partials and adds them in
//    contributor order (bit-reproducible).  256-column tiles give a quarter of the contributors per
//    tile and half the partial size of 512-column tiles.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "awq_internal.h"
#include "awq_host.h"
#include "awq_ptx.cuh"
#include "awq_gemv_common.cuh"

namespace awq {
namespace {

constexpr int kPpConsumers = 4;
constexpr int kPpThreads = (kPpConsumers + 1) * 32;
constexpr int kPpStages = 5;
// Stages whose weights are streamed before the wait on the previous kernel.  Two of the five: a deeper
// early stream competes with the previous call's split-K tail for the memory system (measured on the
// decode sweep, GB/s: 0 stages 2442, 1 2506, 2 2589, 3 2587, 4 2561, 5 2538).
constexpr int kPpPrefetch = 2;
static_assert(kPpPrefetch <= kPpStages, "early stages fit the ring");
constexpr uint32_t kPpProducerSleepNs = 500;
constexpr int kPpTileCols = kPrepackTileCols;        // 256
constexpr int kPpTileWords = kPpTileCols / 8;        // 32
constexpr int kPpQBytes = kGroup * kPpTileCols / 2;  // 16384
constexpr int kPpZBytes = kPpTileWords * 4;          // 128
constexpr int kPpSBytes = kPpTileCols * 2;           // 512
static_assert(kPpQBytes + kPpZBytes + kPpSBytes == kPrepackUnitBytes, "unit layout");
constexpr int kPpXBytes = 8 * kGroup * 2;            // 8 tokens x 128 k: two 1 KB 128-byte-swizzled boxes
constexpr int kPpStageBytes = (kPpXBytes + kPrepackUnitBytes + 1023) / 1024 * 1024;
constexpr int kPpSmem = kPpStages * kPpStageBytes + 1024 + 256;  // ring | alignment slack | barriers, flags
static_assert(kPpSmem <= 113 * 1024, "two CTAs per SM");
static_assert(8 * kPpTileCols * 4 <= kPpStageBytes, "a completer's own sums fit one ring slot");
// 10 warps on one SM (two CTAs): three on one sub-partition, a quarter of the 64 K registers
constexpr int kPpMaxRegs = (65536 / 4) / (3 * 32) / 8 * 8;
static_assert(kPpMaxRegs == 168, "two 5-warp CTAs per SM");

__device__ __forceinline__ void pp_consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kPpConsumers * 32) : "memory");
}
__device__ __forceinline__ bool pp_consumers_any(bool v) {
  uint32_t r;
  asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}"
               : "=r"(r) : "r"((uint32_t)v), "r"(kPpConsumers * 32) : "memory");
  return r != 0;
}

// fp32 factors of the fold for the lane's 8 consecutive columns c = 0..7 of one group: columns 2b
// (low nibbles: s, 1024 + z) and 2b + 1 (high nibbles: s / 16, 1024 + 16 z).  The zero-point word
// holds column c in nibble c, so byte b holds columns 2b and 2b + 1.
struct PpConsts {
  float sf[4][2], szc[4][2];
};

__device__ __forceinline__ void pp_consts(uint32_t zword, const uint4& sv, PpConsts& c) {
  const __half* sh = reinterpret_cast<const __half*>(&sv);
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    // 1024 + z and 1024 + 16 z as fp32 bit patterns: the nibbles of byte b land in the mantissa of
    // 1024.0f (whose last place is 2^-13) at bits 13..16 and 17..20, both from one shift
    const uint32_t zs = 8 * b <= 13 ? zword << (13 - 8 * b) : zword >> (8 * b - 13);
    const float zl = __uint_as_float(0x44800000u | (zs & 0x0001E000u));
    const float zh = __uint_as_float(0x44800000u | (zs & 0x001E0000u));
    c.sf[b][0] = __half2float(sh[2 * b]);
    c.sf[b][1] = __half2float(sh[2 * b + 1]) * 0.0625f;  // s / 16, exact
    c.szc[b][0] = c.sf[b][0] * zl;
    c.szc[b][1] = c.sf[b][1] * zh;
  }
}

__global__ void __maxnreg__(kPpMaxRegs)
gemv_pp_kernel(const __grid_constant__ CUtensorMap tm_x, const uint8_t* __restrict__ packed, __half* __restrict__ y,
               float* __restrict__ part, int* __restrict__ counters, int* __restrict__ err, int M, int N, int G,
               int tiles, int maxc) {
  // unit u = (tile u / G, group u % G); units < 2^31 (host check)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPpStages * kPpStageBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kPpStages);
  volatile int* ready_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int units = tiles * G;
  const int P = gridDim.x;
  const int p = blockIdx.x;
  const int u0 = (int)unit_begin(p, units, P);
  const int u1 = (int)unit_begin(p + 1, units, P);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + kPpStages + s); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPpStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kPpConsumers);
    }
    *abort_flag = 0;
    *ready_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    // the next kernel in the stream may launch now; it waits for this grid before touching shared data
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  __syncthreads();

  if (warp == kPpConsumers) {
    // ------------------------------------------------ copy producer
    if (lane == 0) {
      // the activations' tensor map is read by the first copy after the wait: fetch it now
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
      constexpr uint32_t kTx = (uint32_t)(kPrepackUnitBytes + kPpXBytes);
      auto issue_unit = [&](int st, int u) {
        bulk_load(smem_u32(smem + st * kPpStageBytes + kPpXBytes), packed + (size_t)u * kPrepackUnitBytes,
                  (uint32_t)kPrepackUnitBytes, full_bar(st));
      };
      auto issue_x = [&](int st, int grp) {
        uint8_t* sb = smem + st * kPpStageBytes;
        tma_load_2d(smem_u32(sb), &tm_x, grp * kGroup, 0, full_bar(st));
        tma_load_2d(smem_u32(sb + 1024), &tm_x, grp * kGroup + 64, 0, full_bar(st));
      };
      // the first stages' weights stream before the wait on the previous kernel
      int u = u0;
      int pre = 0;
      while (pre < kPpPrefetch && u < u1) {
        mbar_arrive_tx(full_bar(pre), kTx);
        issue_unit(pre, u);
        ++pre;
        ++u;
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      for (int i = 0; i < pre; ++i) issue_x(i, (u0 + i) % G);
      int issued = pre;
      for (; u < u1; ++u, ++issued) {
        const int st = issued % kPpStages;
        const uint32_t ph = (uint32_t)(issued / kPpStages) & 1u;
        if (!wait_backoff(empty_bar(st), ph ^ 1u, abort_flag, err, 511, kPpProducerSleepNs)) break;
        mbar_arrive_tx(full_bar(st), kTx);
        issue_unit(st, u);
        issue_x(st, u % G);
      }
      // never leave the CTA with copies in flight: the last stages issued must have landed
      volatile int no_abort = 0;
      for (int j = issued - kPpStages < 0 ? 0 : issued - kPpStages; j < issued; ++j)
        wait_bounded(full_bar(j % kPpStages), (uint32_t)(j / kPpStages) & 1u, &no_abort, err, 512);
    }
  } else {
    // ------------------------------------------------ consumer warps
    const int g = lane >> 2;       // mma group: A rows g / g+8 (columns 2b / 2b+1), B column (token) g
    const int t = lane & 3;        // mma thread-in-group
    const int wg = warp * 8 + g;   // this lane's 8-column word in the tile
    const uint32_t q_lane = (uint32_t)(kPpXBytes + ((warp * 8) * 32 + lane) * 16);  // + 512 per step
    const uint32_t z_lane = (uint32_t)(kPpXBytes + kPpQBytes + wg * 4);
    const uint32_t s_lane = (uint32_t)(kPpXBytes + kPpQBytes + kPpZBytes + wg * 16);
    uint32_t x_lane[4];  // activation pair k = 16 (i % 4) + 2t of token g in box i / 4
#pragma unroll
    for (int i = 0; i < 4; ++i) x_lane[i] = x_offset(g, 16 * i + 2 * t);

    bool waited = false;
    int part_tile = -1;     // a shared tile whose partial this CTA wrote (at most one)
    int own_tile = -1;      // the shared tile this CTA completes (it holds its first group)
    float hold[4][4];       // own_tile's sums, kept in registers for its reduction
    bool failed = false;
    int cst = 0;            // ring slot and phase of the next stage
    uint32_t cph = 0;
    int u = u0;
    int tile = u0 / G;
    int grp = u0 - tile * G;
    while (u < u1) {
      const int cur_tile = tile;
      float acc[4][4];
#pragma unroll
      for (int b = 0; b < 4; ++b)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[b][e] = 0.f;
      for (; u < u1 && tile == cur_tile;) {
        const int st = cst;
        const uint32_t ph = cph;
        if (++cst == kPpStages) {
          cst = 0;
          cph ^= 1u;
        }
        ++u;
        if (++grp == G) {
          grp = 0;
          ++tile;
        }
        const uint8_t* sb = smem + st * kPpStageBytes;
        if (!wait_bounded(full_bar(st), ph, abort_flag, err, 513)) {
          failed = true;
          break;
        }
        uint4 wv[8];
        uint32_t xb[8][2];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          wv[i] = *reinterpret_cast<const uint4*>(sb + q_lane + i * 512);
          const uint32_t xo = (uint32_t)((i >> 2) * 1024) + x_lane[i & 3];
          xb[i][0] = *reinterpret_cast<const uint32_t*>(sb + xo);
          xb[i][1] = *reinterpret_cast<const uint32_t*>(sb + (xo ^ 16u));  // k + 8: the next 16-byte chunk
        }
        const uint32_t zword = *reinterpret_cast<const uint32_t*>(sb + z_lane);
        const uint4 sv = *reinterpret_cast<const uint4*>(sb + s_lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(st));  // the slot is free once its data is in registers
        PpConsts gc;
        pp_consts(zword, sv, gc);
        float gacc[4][4], sx[4];  // this group's (1024 + q)^T x and sum_k x
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          sx[b] = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e) gacc[b][e] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t wd[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
          uint32_t a[4][4];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const uint32_t hi = wd[b] >> 8;
            a[b][0] = magic<0x000F000Fu>(wd[b]);  // column 2b, rows 2t / 2t+1
            a[b][1] = magic<0x00F000F0u>(wd[b]);  // column 2b+1 (x16), rows 2t / 2t+1
            a[b][2] = magic<0x000F000Fu>(hi);     // column 2b, rows 2t+8 / 2t+9
            a[b][3] = magic<0x00F000F0u>(hi);     // column 2b+1 (x16), rows 2t+8 / 2t+9
          }
#pragma unroll
          for (int b = 0; b < 4; ++b) mma16816(gacc[b], a[b][0], a[b][1], a[b][2], a[b][3], xb[i][0], xb[i][1]);
          mma16816(sx, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, xb[i][0], xb[i][1]);
        }
        // acc += s (gacc - (1024 + z) sx)  (odd columns: s / 16, 1024 + 16 z)
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            acc[b][e] = fmaf(gacc[b][e], gc.sf[b][e >> 1], fmaf(-gc.szc[b][e >> 1], sx[e & 1], acc[b][e]));
      }
      if (failed) break;

      // ---- flush: CTAs sharing the tile meet in the workspace
      if (!waited) {
        asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs and workspace of the previous kernel
        waited = true;
      }
      const int pf = (int)cta_of_unit(cur_tile * G, units, P);
      const int pl = (int)cta_of_unit((cur_tile + 1) * G - 1, units, P);
      // D fragment: acc[b][0/1] = column 2b, tokens 2t / 2t+1; acc[b][2/3] = column 2b+1: the lane holds
      // its 8 consecutive columns for tokens 2t and 2t+1
      const int n0 = cur_tile * kPpTileCols + wg * 8;
      if (pf == pl) {
#pragma unroll
        for (int par = 0; par < 2; ++par) {
          const int m = 2 * t + par;
          if (m < M && n0 < N) {  // N % 32 == 0: the lane's 8 columns are all in range
            uint32_t h[4];
#pragma unroll
            for (int c = 0; c < 8; c += 2) {
              __half2 v = __floats2half2_rn(acc[c >> 1][par], acc[c >> 1][2 + par]);
              h[c / 2] = *reinterpret_cast<uint32_t*>(&v);
            }
            *reinterpret_cast<uint4*>(y + (size_t)m * N + n0) = make_uint4(h[0], h[1], h[2], h[3]);
          }
        }
      } else if (p == pf) {
        // this CTA holds the tile's first group, so the tile is the last of its range
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int e = 0; e < 4; ++e) hold[b][e] = acc[b][e];
        own_tile = cur_tile;
      } else {
        float* slot = part + ((size_t)cur_tile * maxc + (size_t)(p - pf)) * 8 * kPpTileCols;
#pragma unroll
        for (int par = 0; par < 2; ++par) {
          const int m = 2 * t + par;
          if (m < M) {
            float4* dst = reinterpret_cast<float4*>(slot + m * kPpTileCols + wg * 8);
            dst[0] = make_float4(acc[0][par], acc[0][2 + par], acc[1][par], acc[1][2 + par]);
            dst[1] = make_float4(acc[2][par], acc[2][2 + par], acc[3][par], acc[3][2 + par]);
          }
        }
        part_tile = cur_tile;
      }
    }

    // ---- split K, after the whole range (see the AWQ-layout kernel: every wait ends because no CTA
    // waits before it has published its own partial)
    failed = pp_consumers_any(failed);
    if (!failed && part_tile >= 0) {
      pp_consumers_sync();  // every partial store of this CTA issued
      if (threadIdx.x == 0)
        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(counters + part_tile) : "memory");
    }
    if (!failed && own_tile >= 0) {
      const int nt = (int)cta_of_unit((own_tile + 1) * G - 1, units, P) - p + 1;
      if (threadIdx.x == 0) {
        int* cnt = counters + own_tile;
        const long long t0 = now_ns();
        bool ok = true;
        for (;;) {
          int c;
          asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(c) : "l"(cnt) : "memory");
          if (c == nt - 1) break;
          if (now_ns() - t0 > kWaitLimitNs) {
            if (err) atomicExch(err, 514);
            ok = false;
            break;
          }
        }
        if (ok) *reinterpret_cast<volatile int*>(cnt) = 0;  // every other contributor has counted
        *ready_flag = ok ? 1 : 0;
      }
      // the ring is idle now: its first slot takes this CTA's own sums, [token][256 columns] fp32
      float* own = reinterpret_cast<float*>(smem);
      pp_consumers_sync();
#pragma unroll
      for (int par = 0; par < 2; ++par) {
        const int m = 2 * t + par;
        if (m < M) {
          float4* dst = reinterpret_cast<float4*>(own + m * kPpTileCols + wg * 8);
          dst[0] = make_float4(hold[0][par], hold[0][2 + par], hold[1][par], hold[1][2 + par]);
          dst[1] = make_float4(hold[2][par], hold[2][2 + par], hold[3][par], hold[3][2 + par]);
        }
      }
      pp_consumers_sync();
      if (*ready_flag) {
        // items (token, 4 columns): four per thread, each with eight contributors' loads in flight
        constexpr int kQuads = kPpTileCols / 4;
        constexpr int kThreadsC = kPpConsumers * 32;
        const int items = M * kQuads;
        const float4* base = reinterpret_cast<const float4*>(part + (size_t)own_tile * maxc * 8 * kPpTileCols);
        constexpr size_t kSlotQuads = (size_t)8 * kQuads;
        for (int i0 = threadIdx.x; i0 < items; i0 += 4 * kThreadsC) {
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
            const int n = own_tile * kPpTileCols + (it - m * kQuads) * 4;
            if (n < N) {
              __half2* dst = reinterpret_cast<__half2*>(y + (size_t)m * N + n);
              dst[0] = __floats2half2_rn(s4[k].x, s4[k].y);
              dst[1] = __floats2half2_rn(s4[k].z, s4[k].w);
            }
          }
        }
      }
    }
  }
  __syncthreads();
}

// AWQ nibble of logical column `col` (0..7) in packed word `w`
__device__ __forceinline__ uint32_t awq_nib(uint32_t w, int col) { return (w >> (4 * slot_of_col(col))) & 0xFu; }

// One thread per (unit, warp w, step i, lane l): the lane's four code words; the threads with i = 0 and
// t = 0 also write the (w, g) zero-point word and scale vector.
__global__ void prepack_kernel(const uint32_t* __restrict__ qw, const uint32_t* __restrict__ qz,
                               const __half* __restrict__ sc, uint8_t* __restrict__ out, int64_t N, int G,
                               int64_t total) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int64_t unit = idx >> 10;
  const int r = (int)(idx & 1023);
  const int w = r >> 8, i = (r >> 5) & 7, l = r & 31;
  const int g = l >> 2, t = l & 3;
  const int64_t tile = unit / G;
  const int grp = (int)(unit - tile * G);
  const int64_t nw = N / 8;
  const int64_t cw = tile * kPpTileWords + w * 8 + g;  // AWQ word column of the lane's 8 columns
  const bool in = cw < nw;
  const int64_t k0 = (int64_t)grp * kGroup + 16 * i + 2 * t;
  const uint32_t r0 = in ? qw[k0 * nw + cw] : 0u, r1 = in ? qw[(k0 + 1) * nw + cw] : 0u;
  const uint32_t r8 = in ? qw[(k0 + 8) * nw + cw] : 0u, r9 = in ? qw[(k0 + 9) * nw + cw] : 0u;
  uint32_t o[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int ce = 2 * b, co = 2 * b + 1;
    o[b] = awq_nib(r0, ce) | awq_nib(r0, co) << 4 | awq_nib(r8, ce) << 8 | awq_nib(r8, co) << 12 |
           awq_nib(r1, ce) << 16 | awq_nib(r1, co) << 20 | awq_nib(r9, ce) << 24 | awq_nib(r9, co) << 28;
  }
  uint8_t* ub = out + unit * kPrepackUnitBytes;
  *reinterpret_cast<uint4*>(ub + ((w * 8 + i) * 32 + l) * 16) = make_uint4(o[0], o[1], o[2], o[3]);
  if (i == 0 && t == 0) {
    const int wg = w * 8 + g;
    uint32_t zw = 0;
    uint32_t sv[4] = {0, 0, 0, 0};
    if (in) {
      const uint32_t zaw = qz ? qz[(int64_t)grp * nw + cw] : 0x88888888u;
#pragma unroll
      for (int c = 0; c < 8; ++c) zw |= awq_nib(zaw, c) << (4 * c);
      const uint4 s8 = *reinterpret_cast<const uint4*>(sc + (int64_t)grp * N + cw * 8);
      sv[0] = s8.x; sv[1] = s8.y; sv[2] = s8.z; sv[3] = s8.w;
    }
    *reinterpret_cast<uint32_t*>(ub + kPpQBytes + wg * 4) = zw;
    *reinterpret_cast<uint4*>(ub + kPpQBytes + kPpZBytes + wg * 16) = make_uint4(sv[0], sv[1], sv[2], sv[3]);
  }
}

// The inverse: one thread per (unit, w, i, l) writes the four AWQ words (rows 2t, 2t+1, 2t+8, 2t+9 of its
// 8 columns) that its code words hold; threads with i = 0 and t = 0 write the group's zero-point word and
// scales of those columns.  Padding columns (beyond N) are not written.
__global__ void unprepack_kernel(const uint8_t* __restrict__ in, uint32_t* __restrict__ qw, uint32_t* __restrict__ qz,
                                 __half* __restrict__ sc, int64_t N, int G, int64_t total) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int64_t unit = idx >> 10;
  const int r = (int)(idx & 1023);
  const int w = r >> 8, i = (r >> 5) & 7, l = r & 31;
  const int g = l >> 2, t = l & 3;
  const int64_t tile = unit / G;
  const int grp = (int)(unit - tile * G);
  const int64_t nw = N / 8;
  const int64_t cw = tile * kPpTileWords + w * 8 + g;
  if (cw >= nw) return;
  const uint8_t* ub = in + unit * kPrepackUnitBytes;
  const uint4 v = *reinterpret_cast<const uint4*>(ub + ((w * 8 + i) * 32 + l) * 16);
  const uint32_t o[4] = {v.x, v.y, v.z, v.w};
  // nibble position p of word b: rows (2t, 2t, 2t+8, 2t+8, 2t+1, 2t+1, 2t+9, 2t+9), columns 2b (even p), 2b+1
  uint32_t rw[4] = {0, 0, 0, 0};  // rows 2t, 2t+1, 2t+8, 2t+9
#pragma unroll
  for (int b = 0; b < 4; ++b)
#pragma unroll
    for (int pos = 0; pos < 8; ++pos) {
      const int col = 2 * b + (pos & 1);
      const int row = ((pos >> 1) & 1) * 2 + (pos >> 2);  // positions 0,1 -> 2t; 2,3 -> 2t+8; 4,5 -> 2t+1; 6,7 -> 2t+9
      rw[row] |= ((o[b] >> (4 * pos)) & 0xFu) << (4 * slot_of_col(col));
    }
  const int64_t k0 = (int64_t)grp * kGroup + 16 * i + 2 * t;
  qw[k0 * nw + cw] = rw[0];
  qw[(k0 + 1) * nw + cw] = rw[1];
  qw[(k0 + 8) * nw + cw] = rw[2];
  qw[(k0 + 9) * nw + cw] = rw[3];
  if (i == 0 && t == 0) {
    const int wg = w * 8 + g;
    if (qz) {
      const uint32_t zw = *reinterpret_cast<const uint32_t*>(ub + kPpQBytes + wg * 4);
      uint32_t zaw = 0;
#pragma unroll
      for (int c = 0; c < 8; ++c) zaw |= ((zw >> (4 * c)) & 0xFu) << (4 * slot_of_col(c));
      qz[(int64_t)grp * nw + cw] = zaw;
    }
    *reinterpret_cast<uint4*>(sc + (int64_t)grp * N + cw * 8) =
        *reinterpret_cast<const uint4*>(ub + kPpQBytes + kPpZBytes + wg * 16);
  }
}

}  // namespace

size_t prepacked_bytes(int64_t K, int64_t N) {
  const int64_t tiles = (N + kPpTileCols - 1) / kPpTileCols;
  return (size_t)tiles * (size_t)(K / kGroup) * (size_t)kPrepackUnitBytes;
}

cudaError_t launch_prepack(const uint32_t* qw, const uint32_t* qz, const uint16_t* sc, int64_t K, int64_t N,
                           uint8_t* out, cudaStream_t s) {
  const int64_t tiles = (N + kPpTileCols - 1) / kPpTileCols;
  const int64_t total = tiles * (K / kGroup) * 1024;
  const int64_t blocks = (total + 255) / 256;
  prepack_kernel<<<(unsigned)blocks, 256, 0, s>>>(qw, qz, reinterpret_cast<const __half*>(sc), out, N,
                                                  (int)(K / kGroup), total);
  return cudaGetLastError();
}

cudaError_t launch_unprepack(const uint8_t* in, int64_t K, int64_t N, uint32_t* qw, uint32_t* qz, uint16_t* sc,
                             cudaStream_t s) {
  const int64_t tiles = (N + kPpTileCols - 1) / kPpTileCols;
  const int64_t total = tiles * (K / kGroup) * 1024;
  const int64_t blocks = (total + 255) / 256;
  unprepack_kernel<<<(unsigned)blocks, 256, 0, s>>>(in, qw, qz, reinterpret_cast<__half*>(sc), N,
                                                    (int)(K / kGroup), total);
  return cudaGetLastError();
}

GemvPlan gemv_pp_plan(int64_t M, int64_t K, int64_t N, int split_k) {
  (void)M;
  GemvPlan p;
  p.tiles = (int)((N + kPpTileCols - 1) / kPpTileCols);
  p.groups = (int)(K / kGroup);
  const int64_t units = (int64_t)p.tiles * p.groups;
  const int64_t sms = device_sm_count();
  int64_t ctas;
  if (split_k == 1) {
    ctas = p.tiles;  // one CTA per tile: no tile is shared, so no CTA waits for another
  } else {
    // one CTA per SM for each call: with two per SM, twice the contributors per tile made the split-K
    // tail longer than the better balance saved (measured on the decode sweep)
    ctas = split_k > 1 ? (int64_t)p.tiles * split_k : sms;
    if (ctas > sms) ctas = sms;
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

size_t gemv_pp_workspace_bytes(const GemvPlan& p) {
  if (p.maxc <= 1) return 0;
  return kCounterBytes + align256((size_t)p.tiles * p.maxc * 8 * kPpTileCols * sizeof(float));
}

cudaError_t launch_gemv_prepacked(const uint16_t* x, const uint8_t* packed, uint16_t* y, int64_t M, int64_t K,
                                  int64_t N, const GemvPlan& p, void* ws, int* err, cudaStream_t s) {
  if ((int64_t)p.tiles * p.groups >= ((int64_t)1 << 31) || M < 1 || M > 8) return cudaErrorInvalidValue;
  float* part = nullptr;
  int* counters = nullptr;
  if (p.maxc > 1) {
    counters = static_cast<int*>(ws);
    part = reinterpret_cast<float*>(static_cast<char*>(ws) + kCounterBytes);
  }
  CUtensorMap tx;
  if (!make_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x, (uint64_t)K, (uint64_t)M, 64, 8,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(gemv_pp_kernel), kPpSmem);
  if (e != cudaSuccess) return e;
  // two CTAs per SM need the largest shared-memory carveout (2 x 97 KB)
  static int carveout_set[64] = {0};
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !carveout_set[dev]) {
    e = cudaFuncSetAttribute(reinterpret_cast<const void*>(gemv_pp_kernel),
                             cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    carveout_set[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)p.ctas);
  cfg.blockDim = dim3(kPpThreads);
  cfg.dynamicSmemBytes = kPpSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemv_pp_kernel, tx, packed, reinterpret_cast<__half*>(y), part, counters, err,
                         (int)M, (int)N, (int)(K / kGroup), p.tiles, p.maxc);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace awq
