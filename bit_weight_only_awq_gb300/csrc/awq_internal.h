// Private declarations shared by the translation units of libawq.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace awq {

// Order map of the older AWQ format: nibble slot i holds logical column
// order_map(i), map = [0, 2, 4, 6, 1, 3, 5, 7].
// Source: "Speed up AWQ 2.5x with updated kernel", casper-hansen's format differences.
__host__ __device__ constexpr int order_map(int slot) { return 2 * (slot & 3) + (slot >> 2); }
// Inverse: logical column j lives in nibble slot slot_of_col(j) = [0, 4, 1, 5, 2, 6, 3, 7][j].
__host__ __device__ constexpr int slot_of_col(int col) { return (col >> 1) + 4 * (col & 1); }
static_assert(order_map(0) == 0 && order_map(1) == 2 && order_map(3) == 6 && order_map(4) == 1 &&
                  order_map(7) == 7 && slot_of_col(order_map(5)) == 5 && slot_of_col(1) == 4,
              "AWQ order map");

constexpr int kGroup = 128;          // GPU path group size (input channels per scale)
constexpr int kGemvMaxM = 16;        // decode path handles up to 16 tokens (two 8-token halves above 8)
constexpr int kW4A8MaxKSlice = 16384;  // exact-integer bound of an fp32 tensor-core sum

// Workspace layout shared by every split-K call: a fixed 64 KB block of tile
// counters at offset 0 (so that a zeroed workspace stays valid across calls of
// any shape: each call returns its counters to zero), then call-specific data.
constexpr size_t kCounterBytes = 65536;
constexpr int kMaxCounters = (int)(kCounterBytes / sizeof(int));
inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

// Device error word (one per device, inside the library): kernels record the id
// of a bounded wait that expired; the host reads and clears it.
int* device_error_ptr();  // nullptr if the symbol address could not be obtained

// ---- elementwise kernels (awq_elementwise.cu)
// new_order: the new format's order map [0..7] (else the older [0, 2, 4, 6, 1, 3, 5, 7])
cudaError_t launch_pack(const uint8_t* q, int64_t rows, int64_t n, uint32_t* packed, cudaStream_t s,
                        bool new_order = false);
cudaError_t launch_unpack(const uint32_t* packed, int64_t rows, int64_t n, uint8_t* q, cudaStream_t s,
                          bool new_order = false);
// bf16: bf16 scales and output (else fp16)
cudaError_t launch_dequant(const uint32_t* qw, const uint32_t* qz, const uint16_t* scales, int64_t K,
                           int64_t N, int group, uint16_t* w, cudaStream_t s, bool bf16 = false);

// ---- decode GEMV (awq_gemv.cu)
constexpr int kNumSMs = 152;  // GB300

// Work partition of the decode GEMV: units are (512-column tile, 64-row block) pairs in tile-major
// order; CTA p of P owns units [unit_begin(p), unit_begin(p + 1)).
__host__ __device__ inline int64_t unit_begin(int64_t p, int64_t units, int64_t ctas) {
  return p * units / ctas;
}
// The CTA whose range contains unit u.
__host__ __device__ inline int64_t cta_of_unit(int64_t u, int64_t units, int64_t ctas) {
  return ((u + 1) * ctas + units - 1) / units - 1;
}

struct GemvPlan {
  int tiles;   // 512-column tiles
  int groups;  // 64-row blocks per tile (K / 64)
  int ctas;    // grid size P
  int maxc;    // most CTAs contributing to one tile (1 = no cross-CTA reduction)
  int split;   // effective K split (ceil(ctas / tiles)), the knob callers pass as split_k
};
GemvPlan gemv_plan(int64_t M, int64_t K, int64_t N, int split_k);
size_t gemv_workspace_bytes(const GemvPlan& p, int64_t M, int64_t N);
// bf16: bf16 activations, scales and output on the 8- or 16-token instance (workspace rows as for M = 16)
cudaError_t launch_gemv(const uint16_t* x, const uint32_t* qw, const uint32_t* qz, const uint16_t* sc,
                        uint16_t* y, int64_t M, int64_t K, int64_t N, const GemvPlan& p, void* ws,
                        int* err, cudaStream_t s, bool bf16 = false);
// W4A8 on the GEMV (M <= 16; 8- or 16-token instance): x16 = the int8 codes widened to fp16,
// wq = AWQ-packed u = q + 8, exact int32 accumulators.  gemv_w4a8_ok: the plan keeps every CTA's rows
// of a tile within 16384.
bool gemv_w4a8_ok(const GemvPlan& p, int64_t M);
cudaError_t launch_gemv_w4a8(const uint16_t* x16, const uint32_t* wq, const float* s_tok, const uint16_t* s_ch,
                             uint16_t* y, int32_t* acc_out, int64_t M, int64_t K, int64_t N, const GemvPlan& p,
                             void* ws, int* err, cudaStream_t s);

// SMs of the current device (GB300's count when it cannot be queried)
int device_sm_count();

// ---- decode GEMV on the prepared layout (awq_gemv_pp.cu)
constexpr int kPrepackTileCols = 256;   // output columns per unit
constexpr int kPrepackUnitBytes = kGroup * kPrepackTileCols / 2 + kPrepackTileCols / 2 + 2 * kPrepackTileCols;
static_assert(kPrepackUnitBytes == 17024 && kPrepackUnitBytes % 16 == 0, "prepared unit: codes | zeros | scales");
size_t prepacked_bytes(int64_t K, int64_t N);
cudaError_t launch_prepack(const uint32_t* qw, const uint32_t* qz, const uint16_t* sc, int64_t K, int64_t N,
                           uint8_t* out, cudaStream_t s);
cudaError_t launch_unprepack(const uint8_t* in, int64_t K, int64_t N, uint32_t* qw, uint32_t* qz, uint16_t* sc,
                             cudaStream_t s);
GemvPlan gemv_pp_plan(int64_t M, int64_t K, int64_t N, int split_k);
size_t gemv_pp_workspace_bytes(const GemvPlan& p);
cudaError_t launch_gemv_prepacked(const uint16_t* x, const uint8_t* packed, uint16_t* y, int64_t M, int64_t K,
                                  int64_t N, const GemvPlan& p, void* ws, int* err, cudaStream_t s);

// ---- tensor-core GEMM (awq_gemm_tc.cu)
// kModeW4A8One is the W4A8 kernel for K slices of at most 16384 rows (kW4A8MaxKSlice): one exact
// accumulator per M-block instead of two, which leaves tensor memory for two M-blocks of 256 tokens.
// The plan picks it; callers pass kModeW4A8.
// kModeZeroPointBF16 / kModeSymmetricBF16: the W4A16 modes with bf16 activations, scales and output.
enum GemmMode {
  kModeZeroPoint = 0,
  kModeSymmetric = 1,
  kModeW4A8 = 2,
  kModeW4A8One = 3,
  kModeZeroPointBF16 = 4,
  kModeSymmetricBF16 = 5,
  kModeW4A8G = 6  // W4A8 with per-group integer weight factors s3: weights (u - 8) * s3
};
// W4A8 with per-group factors: |code| <= 128 times |weight| <= 128, so an fp32 sum stays an exact integer
// over 1024 rows (2^24); each tensor-memory accumulator holds one such chunk.
constexpr int kW4A8GroupChunk = 1024;
struct GemmPlan {
  int bt;        // token tile (MMA N): 16, 32, 64, 128 or 256
  int split;     // K slices (grid.z)
  int ksteps;    // 64-row k-steps per slice
  int nb;        // 128-column M-blocks per CTA (1, or 2 for W4A16 with >= 128-token tiles)
  int n_tiles;   // (128 nb)-column weight tiles
  int m_tiles;   // token tiles
  int band;      // token tiles per raster band (the CTA order: bands, then weight tiles, then token tiles)
};
constexpr int64_t kRasterBandBytes = 40ll << 20;
GemmPlan gemm_plan(int64_t M, int64_t K, int64_t N, int split_k, int mode);
size_t gemm_workspace_bytes(const GemmPlan& p, int64_t M, int64_t K, int64_t N, int mode);
// x16: fp16 activations [M, K] (for W4A8 the fp16 copy of the int8 codes).
cudaError_t launch_gemm(int mode, const uint16_t* x16, const uint32_t* qw, const uint32_t* qz,
                        const uint16_t* sc, const float* s_tok, const uint16_t* s_ch, uint16_t* y,
                        int32_t* acc_out, int64_t M, int64_t K, int64_t N, const GemmPlan& p,
                        void* ws_partials, int* counters, int* err, cudaStream_t s);

// ---- W4A8 activation kernels (w4a8_act.cu)
// xq (int8 codes) and x16 (the codes widened to fp16) are each written when not null
cudaError_t launch_quant_act(const uint16_t* x, int8_t* xq, float* s_tok, int64_t M, int64_t K,
                             cudaStream_t s, uint16_t* x16 = nullptr);
cudaError_t launch_i8_to_f16(const int8_t* xq, uint16_t* x16, int64_t count, cudaStream_t s);

}  // namespace awq
