// Host-side launch helpers shared by the kernels' translation units: 2-D tiled TMA descriptors
// and the dynamic shared-memory attribute, both kept from one call to the next so that a call
// with the same tensors (the usual case for model weights and for a decode loop's buffers)
// skips the driver work.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

namespace awq {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// Row-major [outer][inner] tensor of elem_bytes-sized elements at `base`, copied in boxes of
// box_outer x box_inner with swizzle `sw`, 256-byte L2 promotion, zero fill out of bounds.
// A descriptor depends only on these arguments, so a small per-thread cache returns the one
// encoded for an identical argument set.
inline bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t inner,
                        uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  struct Key {
    const void* base;
    uint64_t inner, outer;
    uint32_t box_inner, box_outer;
    int32_t dt, elem_bytes, sw, pad;
  };
  struct Entry {
    Key key;
    CUtensorMap map;
    bool valid;
  };
  static thread_local Entry cache[64];
  Key key;
  std::memset(&key, 0, sizeof key);
  key.base = base;
  key.inner = inner;
  key.outer = outer;
  key.box_inner = box_inner;
  key.box_outer = box_outer;
  key.dt = (int32_t)dt;
  key.elem_bytes = elem_bytes;
  key.sw = (int32_t)sw;
  uint64_t h = reinterpret_cast<uintptr_t>(base) >> 4;
  h = h * 0x9E3779B97F4A7C15ull ^ (inner * 31 + outer) ^ ((uint64_t)box_inner << 20) ^ ((uint64_t)box_outer << 40) ^
      ((uint64_t)key.dt << 8) ^ ((uint64_t)key.sw << 16);
  Entry& e = cache[(h ^ (h >> 29)) & 63];
  if (e.valid && std::memcmp(&e.key, &key, sizeof key) == 0) {
    *map = e.map;
    return true;
  }
  const auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * (uint64_t)elem_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  e.key = key;
  e.map = *map;
  e.valid = true;
  return true;
}

// cudaFuncSetAttribute(func, MaxDynamicSharedMemorySize, bytes) once per (kernel, device, size).
inline cudaError_t set_smem_once(const void* func, int bytes) {
  struct Done {
    const void* func;
    int dev, bytes;
  };
  static std::mutex mu;
  static Done done[128];
  static int n = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
      if (done[i].func == func && done[i].dev == dev && done[i].bytes == bytes) return cudaSuccess;
  }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (n < 128) done[n++] = Done{func, dev, bytes};
  return cudaSuccess;
}

}  // namespace awq
