// C ABI of libawq: argument checks, workspace planning, dispatch to the kernels.
// Declarations and the meaning of every argument: include/awq.h.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/awq.h"
#include "awq_internal.h"

namespace awq {
namespace {

__device__ int g_device_error = 0;  // id of the last bounded device wait that expired (0 = none)

constexpr int kMaxDevices = 64;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Compute capability 10.3 check, cached per device.
awq_status check_arch() {
  static int cached[kMaxDevices] = {0};  // 0 unknown, 1 ok, -1 wrong arch
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return AWQ_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return AWQ_ECUDA;
  if (cached[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return AWQ_ECUDA;
    cached[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return cached[dev] == 1 ? AWQ_OK : AWQ_EARCH;
}

awq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? AWQ_OK : AWQ_ECUDA; }

awq_status check_workspace(size_t need, const void* ws, size_t have) {
  if (need == 0) return AWQ_OK;
  if (ws == nullptr || have < need) return AWQ_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return AWQ_EALIGN;
  return AWQ_OK;
}

}  // namespace

int* device_error_ptr() {
  static int* ptrs[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

}  // namespace awq

using namespace awq;

extern "C" {

const char* awq_status_string(awq_status status) {
  switch (status) {
    case AWQ_OK: return "AWQ_OK";
    case AWQ_EINVAL: return "AWQ_EINVAL: size or shape argument out of range";
    case AWQ_EALIGN: return "AWQ_EALIGN: pointer not 16-byte aligned (workspace: 256-byte)";
    case AWQ_EARCH: return "AWQ_EARCH: current device is not compute capability 10.3";
    case AWQ_ECUDA: return "AWQ_ECUDA: CUDA runtime call or kernel launch failed";
    case AWQ_ETIMEOUT: return "AWQ_ETIMEOUT: a bounded device-side wait expired";
    case AWQ_EWORKSPACE: return "AWQ_EWORKSPACE: workspace missing or too small";
    case AWQ_ENULL: return "AWQ_ENULL: required pointer is NULL";
    default: return "AWQ: unknown status";
  }
}

awq_status awq_pack(const uint8_t* q, int64_t rows, int64_t n, int32_t* packed, awq_stream_t stream) {
  if (rows < 0 || n < 0 || n % 8 != 0) return AWQ_EINVAL;
  if (rows == 0 || n == 0) return AWQ_OK;
  if (!q || !packed) return AWQ_ENULL;
  if (!aligned16(q) || !aligned16(packed)) return AWQ_EALIGN;
  awq_status st = check_arch();
  if (st != AWQ_OK) return st;
  return from_cuda(launch_pack(q, rows, n, reinterpret_cast<uint32_t*>(packed), (cudaStream_t)stream));
}

awq_status awq_unpack(const int32_t* packed, int64_t rows, int64_t n, uint8_t* q, awq_stream_t stream) {
  if (rows < 0 || n < 0 || n % 8 != 0) return AWQ_EINVAL;
  if (rows == 0 || n == 0) return AWQ_OK;
  if (!q || !packed) return AWQ_ENULL;
  if (!aligned16(q) || !aligned16(packed)) return AWQ_EALIGN;
  awq_status st = check_arch();
  if (st != AWQ_OK) return st;
  return from_cuda(launch_unpack(reinterpret_cast<const uint32_t*>(packed), rows, n, q, (cudaStream_t)stream));
}

awq_status awq_pack_order(const uint8_t* q, int64_t rows, int64_t n, awq_order order, int32_t* packed,
                          awq_stream_t stream) {
  if (order != AWQ_ORDER_OLD && order != AWQ_ORDER_NEW) return AWQ_EINVAL;
  if (rows < 0 || n < 0 || n % 8 != 0) return AWQ_EINVAL;
  if (rows == 0 || n == 0) return AWQ_OK;
  if (!q || !packed) return AWQ_ENULL;
  if (!aligned16(q) || !aligned16(packed)) return AWQ_EALIGN;
  awq_status st = check_arch();
  if (st != AWQ_OK) return st;
  return from_cuda(launch_pack(q, rows, n, reinterpret_cast<uint32_t*>(packed), (cudaStream_t)stream,
                               order == AWQ_ORDER_NEW));
}

awq_status awq_unpack_order(const int32_t* packed, int64_t rows, int64_t n, awq_order order, uint8_t* q,
                            awq_stream_t stream) {
  if (order != AWQ_ORDER_OLD && order != AWQ_ORDER_NEW) return AWQ_EINVAL;
  if (rows < 0 || n < 0 || n % 8 != 0) return AWQ_EINVAL;
  if (rows == 0 || n == 0) return AWQ_OK;
  if (!q || !packed) return AWQ_ENULL;
  if (!aligned16(q) || !aligned16(packed)) return AWQ_EALIGN;
  awq_status st = check_arch();
  if (st != AWQ_OK) return st;
  return from_cuda(launch_unpack(reinterpret_cast<const uint32_t*>(packed), rows, n, q, (cudaStream_t)stream,
                                 order == AWQ_ORDER_NEW));
}

awq_status awq_dequant(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales, int64_t K,
                       int64_t N, int32_t group_size, uint16_t* w, awq_stream_t stream) {
  if (group_size != 32 && group_size != 64 && group_size != 128 && group_size != 256) return AWQ_EINVAL;
  if (K < 0 || N < 0 || K % group_size != 0 || N % 8 != 0) return AWQ_EINVAL;
  if (K == 0 || N == 0) return AWQ_OK;
  if (!qweight || !scales || !w) return AWQ_ENULL;
  if (!aligned16(qweight) || !aligned16(scales) || !aligned16(w) || (qzeros && !aligned16(qzeros)))
    return AWQ_EALIGN;
  awq_status st = check_arch();
  if (st != AWQ_OK) return st;
  return from_cuda(launch_dequant(reinterpret_cast<const uint32_t*>(qweight),
                                  reinterpret_cast<const uint32_t*>(qzeros), scales, K, N, group_size, w,
                                  (cudaStream_t)stream));
}

awq_status awq_dequant_bf16(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales, int64_t K,
                            int64_t N, int32_t group_size, uint16_t* w, awq_stream_t stream) {
  if (group_size != 32 && group_size != 64 && group_size != 128 && group_size != 256) return AWQ_EINVAL;
  if (K < 0 || N < 0 || K % group_size != 0 || N % 8 != 0) return AWQ_EINVAL;
  if (K == 0 || N == 0) return AWQ_OK;
  if (!qweight || !scales || !w) return AWQ_ENULL;
  if (!aligned16(qweight) || !aligned16(scales) || !aligned16(w) || (qzeros && !aligned16(qzeros)))
    return AWQ_EALIGN;
  awq_status st = check_arch();
  if (st != AWQ_OK) return st;
  return from_cuda(launch_dequant(reinterpret_cast<const uint32_t*>(qweight),
                                  reinterpret_cast<const uint32_t*>(qzeros), scales, K, N, group_size, w,
                                  (cudaStream_t)stream, true));
}

static bool gemv_shape_ok(int64_t M, int64_t K, int64_t N, int32_t group_size, int32_t split_k) {
  return M >= 0 && M <= kGemvMaxM && K > 0 && K % kGroup == 0 && N > 0 && N % 32 == 0 && group_size == kGroup &&
         split_k >= 0 && K <= (int64_t)1 << 30 && N <= (int64_t)1 << 30;
}
static bool gemm_shape_ok(int64_t M, int64_t K, int64_t N, int32_t split_k) {
  return M >= 0 && M <= (int64_t)1 << 24 && K > 0 && K % kGroup == 0 && K <= (int64_t)1 << 30 && N > 0 &&
         N % 32 == 0 && N <= (int64_t)1 << 30 && split_k >= 0 && M * N < ((int64_t)1 << 40);
}

// W4A8 with at most 16 tokens runs on the GEMV (exact products, int32 reduction) when its plan
// keeps every CTA's rows of a tile within 16384; otherwise, and for more tokens, on the GEMM.
static bool w4a8_on_gemv(int64_t M, int64_t K, int64_t N, int32_t split_k, GemvPlan* plan) {
  if (M < 1 || M > kGemvMaxM) return false;
  *plan = gemv_plan(M, K, N, split_k);
  return gemv_w4a8_ok(*plan, M);
}
// counters | fp16 copy of the codes | GEMV partials (16 token rows per slot; the 8-token instance uses 8)
static size_t w4a8_gemv_workspace_bytes(const GemvPlan& p, int64_t M, int64_t K, int64_t N) {
  const size_t part = gemv_workspace_bytes(p, 16, N);
  return kCounterBytes + align256((size_t)M * (size_t)K * 2) + (part ? part - kCounterBytes : 0);
}

size_t awq_workspace_bytes(awq_op op, int64_t M, int64_t K, int64_t N, int32_t split_k) {
  switch (op) {
    case AWQ_OP_GEMV:
      if (!gemv_shape_ok(M, K, N, kGroup, split_k) || M == 0) return 0;
      return gemv_workspace_bytes(gemv_plan(M, K, N, split_k), M, N);
    case AWQ_OP_GEMM:
      if (!gemm_shape_ok(M, K, N, split_k) || M == 0) return 0;
      return gemm_workspace_bytes(gemm_plan(M, K, N, split_k, kModeZeroPoint), M, K, N, kModeZeroPoint);
    case AWQ_OP_GEMV_BF16:  // sized for the 16-token instance's partials (the 8-token one needs half)
      if (!gemv_shape_ok(M, K, N, kGroup, split_k) || M == 0) return 0;
      return gemv_workspace_bytes(gemv_plan(M, K, N, split_k), 16, N);
    case AWQ_OP_GEMM_BF16:
      if (!gemm_shape_ok(M, K, N, split_k) || M == 0) return 0;
      return gemm_workspace_bytes(gemm_plan(M, K, N, split_k, kModeZeroPointBF16), M, K, N, kModeZeroPointBF16);
    case AWQ_OP_W4A8_GROUPED:
      if (!gemm_shape_ok(M, K, N, split_k) || M == 0) return 0;
      return gemm_workspace_bytes(gemm_plan(M, K, N, split_k, kModeW4A8G), M, K, N, kModeW4A8G);
    case AWQ_OP_GEMV_PREPACKED:
      if (!gemv_shape_ok(M, K, N, kGroup, split_k) || M == 0 || M > 8) return 0;
      return gemv_pp_workspace_bytes(gemv_pp_plan(M, K, N, split_k));
    case AWQ_OP_W4A8_GEMM: {
      if (!gemm_shape_ok(M, K, N, split_k) || M == 0) return 0;
      GemvPlan gp;
      if (w4a8_on_gemv(M, K, N, split_k, &gp)) return w4a8_gemv_workspace_bytes(gp, M, K, N);
      return gemm_workspace_bytes(gemm_plan(M, K, N, split_k, kModeW4A8), M, K, N, kModeW4A8);
    }
    default:
      return 0;
  }
}

awq_status awq_gemv(const uint16_t* x, const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales,
                    uint16_t* y, int64_t M, int64_t K, int64_t N, int32_t group_size, int32_t split_k,
                    void* workspace, size_t workspace_bytes, awq_stream_t stream) {
  if (!gemv_shape_ok(M, K, N, group_size, split_k)) return AWQ_EINVAL;
  if (M == 0) return AWQ_OK;
  if (!x || !qweight || !scales || !y) return AWQ_ENULL;
  if (!aligned16(x) || !aligned16(qweight) || !aligned16(scales) || !aligned16(y) || (qzeros && !aligned16(qzeros)))
    return AWQ_EALIGN;
  const GemvPlan plan = gemv_plan(M, K, N, split_k);
  awq_status st = check_workspace(gemv_workspace_bytes(plan, M, N), workspace, workspace_bytes);
  if (st != AWQ_OK) return st;
  st = check_arch();
  if (st != AWQ_OK) return st;
  int* err = device_error_ptr();
  if (!err) return AWQ_ECUDA;
  return from_cuda(launch_gemv(x, reinterpret_cast<const uint32_t*>(qweight), reinterpret_cast<const uint32_t*>(qzeros),
                               scales, y, M, K, N, plan, workspace, err, (cudaStream_t)stream));
}

size_t awq_prepacked_bytes(int64_t K, int64_t N) {
  if (!gemv_shape_ok(1, K, N, kGroup, 0)) return 0;
  return prepacked_bytes(K, N);
}

awq_status awq_prepack_gemv(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales, int64_t K,
                            int64_t N, int32_t group_size, void* packed, size_t packed_bytes, awq_stream_t stream) {
  if (!gemv_shape_ok(1, K, N, group_size, 0)) return AWQ_EINVAL;
  if (!qweight || !scales || !packed) return AWQ_ENULL;
  if (!aligned16(qweight) || !aligned16(scales) || !aligned16(packed) || (qzeros && !aligned16(qzeros)))
    return AWQ_EALIGN;
  if (packed_bytes < prepacked_bytes(K, N)) return AWQ_EINVAL;
  awq_status st = check_arch();
  if (st != AWQ_OK) return st;
  return from_cuda(launch_prepack(reinterpret_cast<const uint32_t*>(qweight), reinterpret_cast<const uint32_t*>(qzeros),
                                  scales, K, N, static_cast<uint8_t*>(packed), (cudaStream_t)stream));
}

awq_status awq_unprepack_gemv(const void* packed, int64_t K, int64_t N, int32_t* qweight, int32_t* qzeros,
                              uint16_t* scales, awq_stream_t stream) {
  if (!gemv_shape_ok(1, K, N, kGroup, 0)) return AWQ_EINVAL;
  if (!packed || !qweight || !scales) return AWQ_ENULL;
  if (!aligned16(packed) || !aligned16(qweight) || !aligned16(scales) || (qzeros && !aligned16(qzeros)))
    return AWQ_EALIGN;
  awq_status st = check_arch();
  if (st != AWQ_OK) return st;
  return from_cuda(launch_unprepack(static_cast<const uint8_t*>(packed), K, N, reinterpret_cast<uint32_t*>(qweight),
                                    reinterpret_cast<uint32_t*>(qzeros), scales, (cudaStream_t)stream));
}

awq_status awq_gemv_prepacked(const uint16_t* x, const void* packed, uint16_t* y, int64_t M, int64_t K, int64_t N,
                              int32_t split_k, void* workspace, size_t workspace_bytes, awq_stream_t stream) {
  if (!gemv_shape_ok(M, K, N, kGroup, split_k) || M > 8) return AWQ_EINVAL;
  if (M == 0) return AWQ_OK;
  if (!x || !packed || !y) return AWQ_ENULL;
  if (!aligned16(x) || !aligned16(packed) || !aligned16(y)) return AWQ_EALIGN;
  const GemvPlan plan = gemv_pp_plan(M, K, N, split_k);
  awq_status st = check_workspace(gemv_pp_workspace_bytes(plan), workspace, workspace_bytes);
  if (st != AWQ_OK) return st;
  st = check_arch();
  if (st != AWQ_OK) return st;
  int* err = device_error_ptr();
  if (!err) return AWQ_ECUDA;
  return from_cuda(launch_gemv_prepacked(x, static_cast<const uint8_t*>(packed), y, M, K, N, plan, workspace, err,
                                         (cudaStream_t)stream));
}

awq_status awq_gemv_bf16(const uint16_t* x, const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales,
                         uint16_t* y, int64_t M, int64_t K, int64_t N, int32_t group_size, int32_t split_k,
                         void* workspace, size_t workspace_bytes, awq_stream_t stream) {
  if (!gemv_shape_ok(M, K, N, group_size, split_k)) return AWQ_EINVAL;
  if (M == 0) return AWQ_OK;
  if (!x || !qweight || !scales || !y) return AWQ_ENULL;
  if (!aligned16(x) || !aligned16(qweight) || !aligned16(scales) || !aligned16(y) || (qzeros && !aligned16(qzeros)))
    return AWQ_EALIGN;
  const GemvPlan plan = gemv_plan(M, K, N, split_k);
  awq_status st = check_workspace(gemv_workspace_bytes(plan, 16, N), workspace, workspace_bytes);
  if (st != AWQ_OK) return st;
  st = check_arch();
  if (st != AWQ_OK) return st;
  int* err = device_error_ptr();
  if (!err) return AWQ_ECUDA;
  return from_cuda(launch_gemv(x, reinterpret_cast<const uint32_t*>(qweight), reinterpret_cast<const uint32_t*>(qzeros),
                               scales, y, M, K, N, plan, workspace, err, (cudaStream_t)stream, true));
}

awq_status awq_gemm_bf16(const uint16_t* x, const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales,
                         uint16_t* y, int64_t M, int64_t K, int64_t N, int32_t group_size, int32_t split_k,
                         void* workspace, size_t workspace_bytes, awq_stream_t stream) {
  if (!gemm_shape_ok(M, K, N, split_k) || group_size != kGroup) return AWQ_EINVAL;
  if (M == 0) return AWQ_OK;
  if (!x || !qweight || !scales || !y) return AWQ_ENULL;
  if (!aligned16(x) || !aligned16(qweight) || !aligned16(scales) || !aligned16(y) || (qzeros && !aligned16(qzeros)))
    return AWQ_EALIGN;
  const int mode = qzeros ? kModeZeroPointBF16 : kModeSymmetricBF16;
  const GemmPlan plan = gemm_plan(M, K, N, split_k, mode);
  awq_status st = check_workspace(gemm_workspace_bytes(plan, M, K, N, mode), workspace, workspace_bytes);
  if (st != AWQ_OK) return st;
  st = check_arch();
  if (st != AWQ_OK) return st;
  int* err = device_error_ptr();
  if (!err) return AWQ_ECUDA;
  void* part = nullptr;
  int* counters = nullptr;
  if (plan.split > 1) {
    if ((int64_t)plan.n_tiles * plan.m_tiles > kMaxCounters) return AWQ_EINVAL;
    counters = static_cast<int*>(workspace);
    part = static_cast<char*>(workspace) + kCounterBytes;
  }
  return from_cuda(launch_gemm(mode, x, reinterpret_cast<const uint32_t*>(qweight),
                               reinterpret_cast<const uint32_t*>(qzeros), scales, nullptr, nullptr, y, nullptr, M,
                               K, N, plan, part, counters, err, (cudaStream_t)stream));
}

awq_status awq_gemm(const uint16_t* x, const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales,
                    uint16_t* y, int64_t M, int64_t K, int64_t N, int32_t group_size, int32_t split_k,
                    void* workspace, size_t workspace_bytes, awq_stream_t stream) {
  if (!gemm_shape_ok(M, K, N, split_k) || group_size != kGroup) return AWQ_EINVAL;
  if (M == 0) return AWQ_OK;
  if (!x || !qweight || !scales || !y) return AWQ_ENULL;
  if (!aligned16(x) || !aligned16(qweight) || !aligned16(scales) || !aligned16(y) || (qzeros && !aligned16(qzeros)))
    return AWQ_EALIGN;
  const int mode = qzeros ? kModeZeroPoint : kModeSymmetric;
  const GemmPlan plan = gemm_plan(M, K, N, split_k, mode);
  awq_status st = check_workspace(gemm_workspace_bytes(plan, M, K, N, mode), workspace, workspace_bytes);
  if (st != AWQ_OK) return st;
  st = check_arch();
  if (st != AWQ_OK) return st;
  int* err = device_error_ptr();
  if (!err) return AWQ_ECUDA;
  void* part = nullptr;
  int* counters = nullptr;
  if (plan.split > 1) {
    if ((int64_t)plan.n_tiles * plan.m_tiles > kMaxCounters) return AWQ_EINVAL;
    counters = static_cast<int*>(workspace);
    part = static_cast<char*>(workspace) + kCounterBytes;
  }
  return from_cuda(launch_gemm(mode, x, reinterpret_cast<const uint32_t*>(qweight),
                               reinterpret_cast<const uint32_t*>(qzeros), scales, nullptr, nullptr, y, nullptr, M,
                               K, N, plan, part, counters, err, (cudaStream_t)stream));
}

awq_status w4a8_quant_act(const uint16_t* x, int8_t* xq, float* s_tok, int64_t M, int64_t K, awq_stream_t stream) {
  if (M < 0 || K <= 0 || K % 8 != 0 || M > 0x7FFFFFFF || K > ((int64_t)1 << 30)) return AWQ_EINVAL;
  if (M == 0) return AWQ_OK;
  if (!x || !xq || !s_tok) return AWQ_ENULL;
  if (!aligned16(x) || !aligned16(xq)) return AWQ_EALIGN;
  awq_status st = check_arch();
  if (st != AWQ_OK) return st;
  return from_cuda(launch_quant_act(x, xq, s_tok, M, K, (cudaStream_t)stream));
}

}  // extern "C"

// The W4A8 product once `fill` has written the fp16 codes of the activations into the workspace
// (from int8 codes, or by quantizing fp16 activations): the GEMV (up to 16 tokens) or the GEMM, as planned.
template <class Fill>
static awq_status w4a8_product(Fill fill, const float* s_tok, const int32_t* wq, const uint16_t* s_ch, uint16_t* y,
                               int32_t* acc_out, int64_t M, int64_t K, int64_t N, int32_t split_k, void* workspace,
                               size_t workspace_bytes, awq_stream_t stream) {
  GemvPlan gp;
  const bool on_gemv = w4a8_on_gemv(M, K, N, split_k, &gp);
  const GemmPlan plan = gemm_plan(M, K, N, split_k, kModeW4A8);
  const size_t need = on_gemv ? w4a8_gemv_workspace_bytes(gp, M, K, N) : gemm_workspace_bytes(plan, M, K, N, kModeW4A8);
  awq_status st = check_workspace(need, workspace, workspace_bytes);
  if (st != AWQ_OK) return st;
  if (!on_gemv && plan.split > 1 && (int64_t)plan.n_tiles * plan.m_tiles > kMaxCounters) return AWQ_EINVAL;
  st = check_arch();
  if (st != AWQ_OK) return st;
  int* err = device_error_ptr();
  if (!err) return AWQ_ECUDA;
  char* ws = static_cast<char*>(workspace);
  uint16_t* x16 = reinterpret_cast<uint16_t*>(ws + kCounterBytes);
  const cudaStream_t s = (cudaStream_t)stream;
  if (fill(x16, s) != cudaSuccess) return AWQ_ECUDA;
  const uint32_t* w = reinterpret_cast<const uint32_t*>(wq);
  if (on_gemv) return from_cuda(launch_gemv_w4a8(x16, w, s_tok, s_ch, y, acc_out, M, K, N, gp, workspace, err, s));
  void* part = nullptr;
  int* counters = nullptr;
  if (plan.split > 1) {
    counters = reinterpret_cast<int*>(ws);
    part = ws + kCounterBytes + align256((size_t)M * (size_t)K * 2);
  }
  return from_cuda(launch_gemm(kModeW4A8, x16, w, nullptr, nullptr, s_tok, s_ch, y, acc_out, M, K, N, plan, part,
                               counters, err, s));
}

extern "C" {

awq_status w4a8_gemm(const int8_t* xq, const float* s_tok, const int32_t* wq, const uint16_t* s_ch, uint16_t* y,
                     int32_t* acc_out, int64_t M, int64_t K, int64_t N, int32_t split_k, void* workspace,
                     size_t workspace_bytes, awq_stream_t stream) {
  if (!gemm_shape_ok(M, K, N, split_k)) return AWQ_EINVAL;
  if (M == 0) return AWQ_OK;
  if (!xq || !s_tok || !wq || !s_ch || !y) return AWQ_ENULL;
  if (!aligned16(xq) || !aligned16(wq) || !aligned16(s_ch) || !aligned16(y) || (acc_out && !aligned16(acc_out)))
    return AWQ_EALIGN;
  auto widen = [&](uint16_t* x16, cudaStream_t s) { return launch_i8_to_f16(xq, x16, M * K, s); };
  return w4a8_product(widen, s_tok, wq, s_ch, y, acc_out, M, K, N, split_k, workspace, workspace_bytes, stream);
}

awq_status w4a8_linear(const uint16_t* x, const int32_t* wq, const uint16_t* s_ch, uint16_t* y, int32_t* acc_out,
                       int8_t* xq_out, float* s_tok, int64_t M, int64_t K, int64_t N, int32_t split_k,
                       void* workspace, size_t workspace_bytes, awq_stream_t stream) {
  if (!gemm_shape_ok(M, K, N, split_k)) return AWQ_EINVAL;
  if (M == 0) return AWQ_OK;
  if (!x || !s_tok || !wq || !s_ch || !y) return AWQ_ENULL;
  if (!aligned16(x) || !aligned16(wq) || !aligned16(s_ch) || !aligned16(y) || (acc_out && !aligned16(acc_out)) ||
      (xq_out && !aligned16(xq_out)))
    return AWQ_EALIGN;
  auto quantize = [&](uint16_t* x16, cudaStream_t s) { return launch_quant_act(x, xq_out, s_tok, M, K, s, x16); };
  return w4a8_product(quantize, s_tok, wq, s_ch, y, acc_out, M, K, N, split_k, workspace, workspace_bytes, stream);
}

}  // extern "C"

// The per-group W4A8 product once `fill` has written the fp16 codes of the activations into the workspace:
// the tensor-core GEMM with 1024-row exact chunks (every token count).
template <class Fill>
static awq_status w4a8_grouped_product(Fill fill, const float* s_tok, const int32_t* wq, const uint16_t* s3,
                                       const uint16_t* s2, uint16_t* y, int32_t* acc_out, int64_t M, int64_t K,
                                       int64_t N, int32_t split_k, void* workspace, size_t workspace_bytes,
                                       awq_stream_t stream) {
  const GemmPlan plan = gemm_plan(M, K, N, split_k, kModeW4A8G);
  awq_status st = check_workspace(gemm_workspace_bytes(plan, M, K, N, kModeW4A8G), workspace, workspace_bytes);
  if (st != AWQ_OK) return st;
  if (plan.split > 1 && (int64_t)plan.n_tiles * plan.m_tiles > kMaxCounters) return AWQ_EINVAL;
  st = check_arch();
  if (st != AWQ_OK) return st;
  int* err = device_error_ptr();
  if (!err) return AWQ_ECUDA;
  char* ws = static_cast<char*>(workspace);
  uint16_t* x16 = reinterpret_cast<uint16_t*>(ws + kCounterBytes);
  const cudaStream_t s = (cudaStream_t)stream;
  if (fill(x16, s) != cudaSuccess) return AWQ_ECUDA;
  void* part = nullptr;
  int* counters = nullptr;
  if (plan.split > 1) {
    counters = reinterpret_cast<int*>(ws);
    part = ws + kCounterBytes + align256((size_t)M * (size_t)K * 2);
  }
  return from_cuda(launch_gemm(kModeW4A8G, x16, reinterpret_cast<const uint32_t*>(wq), nullptr, s3, s_tok, s2, y,
                               acc_out, M, K, N, plan, part, counters, err, s));
}

extern "C" {

awq_status w4a8_gemm_grouped(const int8_t* xq, const float* s_tok, const int32_t* wq, const uint16_t* s3,
                             const uint16_t* s2, uint16_t* y, int32_t* acc_out, int64_t M, int64_t K, int64_t N,
                             int32_t group_size, int32_t split_k, void* workspace, size_t workspace_bytes,
                             awq_stream_t stream) {
  if (!gemm_shape_ok(M, K, N, split_k) || group_size != kGroup) return AWQ_EINVAL;
  if (M == 0) return AWQ_OK;
  if (!xq || !s_tok || !wq || !s3 || !s2 || !y) return AWQ_ENULL;
  if (!aligned16(xq) || !aligned16(wq) || !aligned16(s3) || !aligned16(s2) || !aligned16(y) ||
      (acc_out && !aligned16(acc_out)))
    return AWQ_EALIGN;
  auto widen = [&](uint16_t* x16, cudaStream_t s) { return launch_i8_to_f16(xq, x16, M * K, s); };
  return w4a8_grouped_product(widen, s_tok, wq, s3, s2, y, acc_out, M, K, N, split_k, workspace, workspace_bytes,
                              stream);
}

awq_status w4a8_linear_grouped(const uint16_t* x, const int32_t* wq, const uint16_t* s3, const uint16_t* s2,
                               uint16_t* y, int32_t* acc_out, int8_t* xq_out, float* s_tok, int64_t M, int64_t K,
                               int64_t N, int32_t group_size, int32_t split_k, void* workspace,
                               size_t workspace_bytes, awq_stream_t stream) {
  if (!gemm_shape_ok(M, K, N, split_k) || group_size != kGroup) return AWQ_EINVAL;
  if (M == 0) return AWQ_OK;
  if (!x || !s_tok || !wq || !s3 || !s2 || !y) return AWQ_ENULL;
  if (!aligned16(x) || !aligned16(wq) || !aligned16(s3) || !aligned16(s2) || !aligned16(y) ||
      (acc_out && !aligned16(acc_out)) || (xq_out && !aligned16(xq_out)))
    return AWQ_EALIGN;
  auto quantize = [&](uint16_t* x16, cudaStream_t s) { return launch_quant_act(x, xq_out, s_tok, M, K, s, x16); };
  return w4a8_grouped_product(quantize, s_tok, wq, s3, s2, y, acc_out, M, K, N, split_k, workspace, workspace_bytes,
                              stream);
}

awq_status awq_last_device_error(int32_t* code) {
  if (!code) return AWQ_ENULL;
  *code = 0;
  int* p = device_error_ptr();
  if (!p) return AWQ_ECUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return AWQ_ECUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return AWQ_ECUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return AWQ_ECUDA;
  }
  *code = v;
  return v ? AWQ_ETIMEOUT : AWQ_OK;
}

}  // extern "C"
