// Decode GEMV (M <= 8 tokens): y[m, n] = sum_k x[m, k] * W[k, n], W dequantized in registers.
//
// Source of the operation: the M <= 8 branch of the AWQ dispatch snippet,
// gemv_forward_cuda(inputs, qweight, scales, qzeros, group_size) ("Speed up AWQ
// 2.5x with updated kernel").  The kernel design is this library's own:
//
//  * HBM-bound: every packed word is read exactly once.  Measured on GB300, a TMA
//    stream only approaches the copy bandwidth with 256-byte-or-longer runs per row and
//    ~200 KB in flight per SM (loaded DRAM latency is several microseconds), and a decode
//    GEMV of a 7B-model layer moves only 8-47 MB, so per-call latency (first bytes, the
//    cross-CTA reduction, the launch) matters as much as the streaming rate.  The kernel
//    therefore uses at most half of an SM: one persistent CTA per SM per call, a
//    producer warp streaming 16 KB stages (64 rows x 512 columns of packed words as two
//    128-byte-swizzled TMA boxes, plus the group's zero-point / scale rows and the 64
//    activations of every token) through a 5-deep ring, and 8 consumer warps (one
//    64-column slice each) that copy their share of a stage into registers and release
//    the slot at once.  The other half of every SM takes the next call's CTA, which
//    programmatic dependent launch starts early: it streams its weights while this call
//    finishes, so consecutive calls overlap their latencies.
//  * Persistent, evenly balanced grid: the (512-column tile, 64-row block) units are cut
//    into equal contiguous ranges, one per SM.  A tile finished by one CTA is written
//    directly; a tile shared by several CTAs leaves one fp32 partial per CTA in the
//    workspace and the last of them (atomic ticket) sums the partials in contributor
//    order and rounds once to fp16, so results are bit-reproducible.
//  * Programmatic dependent launch: the GEMV starts streaming its weights before waiting
//    for the previous kernel, and touches activations, outputs and the workspace only
//    after that wait.
//  * The multiply runs on the tensor pipe: mma.sync m16n8k16 with the dequantized
//    weights as the A operand (16 output columns x 16 k) and the activations as B
//    (16 k x 8 tokens), fp32 accumulation.  The mma wants k-pairs in each 32-bit A
//    register while a packed word holds 8 columns of one k, so a PRMT takes the same
//    byte of two consecutive rows, and a LOP3 with the fp16 magic 0x6400 turns its low /
//    high nibbles into (1024 + q) / (1024 + 16 q) halves.  HSUB2 of the zero (same
//    magic) then HMUL2 by the scale (s, or s / 16 for the high nibble) give
//    fp16_RN((q - z) * s), the same value the dequant kernel writes.
//  * Lane (g, t) of the mma reads rows 2t, 2t+1 (+8) of each 16-row step; with the
//    128-byte swizzle those 32-bit shared-memory loads, and the activation loads, are
//    free of bank conflicts, and every address is a lane constant plus an immediate.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "awq_internal.h"
#include "awq_ptx.cuh"

namespace awq {
namespace {

constexpr int kConsumers = 8;                  // consumer warps, one 64-column slice of the tile each
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kCtasPerSm = 2;                  // this call's CTA and the next call's
constexpr int kStages = 5;
constexpr int kRows = 64;                      // rows per stage (half a quantization group)
constexpr int kTileWords = 64;                 // packed words per tile row = 512 output columns
constexpr int kTileCols = kTileWords * 8;
constexpr int kBoxWords = 32;                  // one 128-byte-swizzled TMA box is 32 words wide
constexpr int kBoxBytes = kRows * kBoxWords * 4;   // 8 KB
constexpr int kQBytes = kRows * kTileWords * 4;    // 16 KB (two boxes)
constexpr int kXBytes = kGemvMaxM * kRows * 2;     // 1 KB (one 128B-swizzled box, 8 tokens x 64)
constexpr int kZBytes = kTileWords * 4;            // 256 B
constexpr int kSBytes = kTileCols * 2;             // 1 KB
constexpr int kXOff = kQBytes;
constexpr int kZOff = kXOff + kXBytes;
constexpr int kSOff = kZOff + kZBytes;
constexpr int kStageBytes = ((kSOff + kSBytes) + 1023) / 1024 * 1024;
constexpr int kSmemBytes = kStages * kStageBytes + 256 + 1024;
static_assert(kSmemBytes * kCtasPerSm <= 227 * 1024, "shared memory budget: two CTAs per SM");
static_assert(kTileWords == kConsumers * 8, "one 8-word slice per consumer warp");

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
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
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

__device__ __forceinline__ void consumers_sync() {  // the consumer warps only (named barrier 1)
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
}

// 32-bit word `word` (0..63) of packed row `row` in the stage tile: two 128-byte-swizzled
// boxes of 32 words x 64 rows.
__device__ __forceinline__ uint32_t q_offset(int row, int word) {
  return (uint32_t)((word >> 5) * kBoxBytes + row * 128 + (((((word & 31) >> 2) ^ (row & 7))) << 4) +
                    (word & 3) * 4);
}
// Activation pair (k, k+1), k even (0..62), of token g in the 128-byte-swizzled 1 KB box.
__device__ __forceinline__ uint32_t x_offset(int g, int k) {
  return (uint32_t)(g * 128 + ((((k >> 3) ^ g)) << 4) + (k & 7) * 2);
}

// Lane-constant parts of the shared-memory addresses a consumer lane reads; every load of a
// stage is then one of these plus a compile-time row offset.
struct LaneOffsets {
  uint32_t q[2];  // packed word of row 2t + c, c = 0, 1 (rows +8 are +1024 bytes)
  uint32_t x[4];  // activation pair k = 16i + 2t of token g for the four 16-row steps i
};

__device__ __forceinline__ LaneOffsets lane_offsets(int word, int g, int t) {
  LaneOffsets o;
#pragma unroll
  for (int c = 0; c < 2; ++c) o.q[c] = q_offset(2 * t + c, word);
#pragma unroll
  for (int i = 0; i < 4; ++i) o.x[i] = kXOff + x_offset(g, 16 * i + 2 * t);
  return o;
}

// A consumer lane's share of one stage, copied out of shared memory so the slot can be
// released before the arithmetic starts.
struct StageRegs {
  uint32_t r[4][4];  // [16-row step][rows 2t, 2t+1, 2t+8, 2t+9]
  uint32_t b[4][2];  // [16-row step][activation pairs k = 2t, 2t+8]
  uint32_t zword;
  uint4 sv;
};

__device__ __forceinline__ void load_stage(const uint8_t* sb, bool has_z, int word, const LaneOffsets& lo,
                                           StageRegs& sr) {
  sr.zword = has_z ? reinterpret_cast<const uint32_t*>(sb + kZOff)[word] : 0x88888888u;
  sr.sv = reinterpret_cast<const uint4*>(sb + kSOff)[word];
  const uint8_t* q0 = sb + lo.q[0];
  const uint8_t* q1 = sb + lo.q[1];
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int base = 16 * it;  // (base + 2t + c) & 7 == (2t + c) & 7
    sr.r[it][0] = *reinterpret_cast<const uint32_t*>(q0 + base * 128);
    sr.r[it][1] = *reinterpret_cast<const uint32_t*>(q1 + base * 128);
    sr.r[it][2] = *reinterpret_cast<const uint32_t*>(q0 + (base + 8) * 128);
    sr.r[it][3] = *reinterpret_cast<const uint32_t*>(q1 + (base + 8) * 128);
    // k + 8 is the neighbouring 16-byte chunk: physical chunk ^ 1, address ^ 16
    sr.b[it][0] = *reinterpret_cast<const uint32_t*>(sb + lo.x[it]);
    sr.b[it][1] = *reinterpret_cast<const uint32_t*>(sb + (lo.x[it] ^ 16u));
  }
}

// acc += W^T x over the 64 rows held in `sr` (this lane's packed word column, 8 tokens).
__device__ __forceinline__ void compute_stage(const StageRegs& sr, float (&acc)[4][4]) {
  uint32_t zlo[4], zhi[4], slo[4], shi[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t zb = prmt(sr.zword, sr.zword, byte_sel(b));
    zlo[b] = magic<0x000F000Fu>(zb);  // 1024 + z(slot 2b)
    zhi[b] = magic<0x00F000F0u>(zb);  // 1024 + 16 z(slot 2b+1)
    slo[b] = bcast_half(sr.sv, order_map(2 * b));
    shi[b] = hmul2(bcast_half(sr.sv, order_map(2 * b + 1)), 0x2C002C00u);  // s / 16
  }
#pragma unroll
  for (int it = 0; it < 4; ++it) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t p01 = prmt(sr.r[it][0], sr.r[it][1], byte_sel(b));
      const uint32_t p23 = prmt(sr.r[it][2], sr.r[it][3], byte_sel(b));
      const uint32_t a0 = hmul2(hsub2(magic<0x000F000Fu>(p01), zlo[b]), slo[b]);
      const uint32_t a1 = hmul2(hsub2(magic<0x00F000F0u>(p01), zhi[b]), shi[b]);
      const uint32_t a2 = hmul2(hsub2(magic<0x000F000Fu>(p23), zlo[b]), slo[b]);
      const uint32_t a3 = hmul2(hsub2(magic<0x00F000F0u>(p23), zhi[b]), shi[b]);
      mma16816(acc[b], a0, a1, a2, a3, sr.b[it][0], sr.b[it][1]);
    }
  }
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
gemv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_x,
            const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_s, int has_z,
            __half* __restrict__ y, float* __restrict__ part, int* __restrict__ counters, int* __restrict__ err,
            int M, int N, int RB, int tiles, int maxc) {
  // RB = K / 64 row blocks per tile; unit u = (tile u / RB, row block u % RB)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kStages);
  int* last_flag = reinterpret_cast<int*>(bars + 2 * kStages) + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t units = (int64_t)tiles * RB;
  const int64_t P = gridDim.x;
  const int64_t p = blockIdx.x;
  const int64_t u0 = unit_begin(p, units, P);
  const int64_t u1 = unit_begin(p + 1, units, P);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + kStages + s); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kConsumers);
    }
    *abort_flag = 0;
    *last_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    // the next kernel in the stream may launch now; it waits for this grid before touching shared data
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t tx = kQBytes + kXBytes + (has_z ? kZBytes : 0) + kSBytes;
      auto issue_weights = [&](int st, int64_t u) {
        const int tile = (int)(u / RB);
        const int rb = (int)(u - (int64_t)tile * RB);
        const int grp = rb / (kGroup / kRows);
        uint8_t* sb = smem + st * kStageBytes;
#pragma unroll
        for (int bx = 0; bx < kTileWords / kBoxWords; ++bx)
          tma_load_2d(smem_u32(sb + bx * kBoxBytes), &tm_q, tile * kTileWords + bx * kBoxWords, rb * kRows,
                      full_bar(st));
        if (has_z) tma_load_2d(smem_u32(sb + kZOff), &tm_z, tile * kTileWords, grp, full_bar(st));
        // scales viewed as int32 pairs: 512 columns = one 256-pair box
        tma_load_2d(smem_u32(sb + kSOff), &tm_s, tile * (kTileCols / 2), grp, full_bar(st));
      };
      auto issue_x = [&](int st, int64_t u) {
        const int rb = (int)(u % RB);
        tma_load_2d(smem_u32(smem + st * kStageBytes + kXOff), &tm_x, rb * kRows, 0, full_bar(st));
      };
      const int64_t n = u1 - u0;
      const int pre = (int)(n < kStages ? n : kStages);
      // weights of the first stages stream before the wait on the previous kernel
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_tx(full_bar(i), tx);
        issue_weights(i, u0 + i);
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      for (int i = 0; i < pre; ++i) issue_x(i, u0 + i);
      int issued = pre;
      for (int64_t u = u0 + pre; u < u1; ++u, ++issued) {
        const int st = issued % kStages;
        const uint32_t ph = (uint32_t)(issued / kStages) & 1u;
        if (!wait_bounded(empty_bar(st), ph ^ 1u, abort_flag, err, 501)) break;
        mbar_arrive_tx(full_bar(st), tx);
        issue_weights(st, u);
        issue_x(st, u);
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
    const LaneOffsets lo = lane_offsets(word, g, t);
    bool waited = false;
    int64_t i = 0;                    // stage counter, identical to the producer's
    for (int64_t seg = u0; seg < u1;) {
      const int tile = (int)(seg / RB);
      const int64_t seg_end = min(u1, (int64_t)(tile + 1) * RB);
      float acc[4][4];
#pragma unroll
      for (int b = 0; b < 4; ++b)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[b][e] = 0.f;
      for (int64_t u = seg; u < seg_end; ++u, ++i) {
        const int st = (int)(i % kStages);
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        StageRegs sr;
        const bool ok = wait_bounded(full_bar(st), ph, abort_flag, err, 503);
        if (ok) load_stage(smem + st * kStageBytes, has_z != 0, word, lo, sr);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(st));  // slot free before the arithmetic
        if (ok) compute_stage(sr, acc);
      }

      // ---- flush: this warp owns its 64 columns; CTAs sharing the tile meet in the workspace
      if (!waited) {
        asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs and workspace of the previous kernel
        waited = true;
      }
      const int64_t pf = cta_of_unit((int64_t)tile * RB, units, P);
      const int64_t pl = cta_of_unit((int64_t)(tile + 1) * RB - 1, units, P);
      const int nt = (int)(pl - pf + 1);
      // D fragment: acc[b][0/1] = (column lo of byte b, tokens 2t / 2t+1), acc[b][2/3] = column hi
      if (nt == 1) {
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m = 2 * t + (e & 1);
            const int n = tile * kTileCols + word * 8 + order_map(2 * b + (e >> 1));
            if (m < M && n < N) y[(size_t)m * N + n] = __float2half_rn(acc[b][e]);
          }
      } else {
        float* slot = part + ((size_t)tile * maxc + (size_t)(p - pf)) * kGemvMaxM * kTileCols;
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m = 2 * t + (e & 1);
            if (m < M) slot[m * kTileCols + word * 8 + order_map(2 * b + (e >> 1))] = acc[b][e];
          }
        __threadfence();
        consumers_sync();
        if (threadIdx.x == 0) *last_flag = (atomicAdd(counters + tile, 1) == nt - 1);
        consumers_sync();
        if (*last_flag) {
          __threadfence();
          // contributor-ordered sum, eight partials in flight per step
          const float4* base = reinterpret_cast<const float4*>(part + (size_t)tile * maxc * kGemvMaxM * kTileCols);
          constexpr int kQuads = kTileCols / 4;
          constexpr size_t kSlotQuads = (size_t)kGemvMaxM * kQuads;
          for (int q = threadIdx.x; q < M * kQuads; q += kConsumers * 32) {
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j0 = 0; j0 < nt; j0 += 8) {
              float4 v[8];
#pragma unroll
              for (int jj = 0; jj < 8; ++jj)
                v[jj] = (j0 + jj < nt) ? __ldcg(base + (size_t)(j0 + jj) * kSlotQuads + q)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                s.x += v[jj].x; s.y += v[jj].y; s.z += v[jj].z; s.w += v[jj].w;
              }
            }
            const int m = q / kQuads;
            const int n = tile * kTileCols + (q - m * kQuads) * 4;
            if (n < N) {  // N % 32 == 0: all four outputs are in range
              __half2* dst = reinterpret_cast<__half2*>(y + (size_t)m * N + n);
              dst[0] = __floats2half2_rn(s.x, s.y);
              dst[1] = __floats2half2_rn(s.z, s.w);
            }
          }
          if (threadIdx.x == 0) atomicExch(counters + tile, 0);  // leave the ticket at zero for the next call
        }
        consumers_sync();  // last_flag is reused by the next tile
      }
      seg = seg_end;
    }
  }
  __syncthreads();
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t inner,
                 uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  const auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * (uint64_t)elem_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

GemvPlan gemv_plan(int64_t M, int64_t K, int64_t N, int split_k) {
  (void)M;
  GemvPlan p;
  p.tiles = (int)((N / 8 + kTileWords - 1) / kTileWords);
  p.groups = (int)(K / kRows);  // row blocks of 64 (two per quantization group)
  const int64_t units = (int64_t)p.tiles * p.groups;
  int64_t ctas = split_k > 0 ? (int64_t)p.tiles * split_k : (int64_t)kNumSMs;
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
  (void)M;
  (void)N;
  if (p.maxc <= 1) return 0;
  return kCounterBytes + align256((size_t)p.tiles * p.maxc * kGemvMaxM * kTileCols * sizeof(float));
}

cudaError_t launch_gemv(const uint16_t* x, const uint32_t* qw, const uint32_t* qz, const uint16_t* sc,
                        uint16_t* y, int64_t M, int64_t K, int64_t N, const GemvPlan& p, void* ws,
                        int* err, cudaStream_t s) {
  float* part = nullptr;
  int* counters = nullptr;
  if (p.maxc > 1) {
    counters = static_cast<int*>(ws);
    part = reinterpret_cast<float*>(static_cast<char*>(ws) + kCounterBytes);
  }
  const uint64_t nw = (uint64_t)N / 8;
  const uint64_t ng = (uint64_t)K / kGroup;
  CUtensorMap tq, tx, tz, ts;
  const bool ok =
      make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, qw, nw, (uint64_t)K, kBoxWords, kRows,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
      make_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x, (uint64_t)K, (uint64_t)M, kRows, kGemvMaxM,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
      make_map_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, qz ? (const void*)qz : (const void*)qw, nw,
                  qz ? ng : (uint64_t)K, kTileWords, 1, CU_TENSOR_MAP_SWIZZLE_NONE) &&
      make_map_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, sc, (uint64_t)N / 2, ng, kTileCols / 2, 1,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!ok) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
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
  e = cudaLaunchKernelEx(&cfg, gemv_kernel, tq, tx, tz, ts, qz ? 1 : 0, reinterpret_cast<__half*>(y), part, counters,
                         err, (int)M, (int)N, (int)(K / kRows), p.tiles, p.maxc);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace awq
