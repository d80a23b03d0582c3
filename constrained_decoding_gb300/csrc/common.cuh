// Shared definitions of the PCD CUDA library: error words, bf16 helpers and
// the host-side launch helpers every kernel file uses.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace pcd {

// Device-side error word (one int per model, in device memory).  Kernels
// record the first failure with atomicCAS; the host reads it after a sync.
enum DeviceError : int {
  DEV_OK = 0,
  DEV_WAIT_TIMEOUT_PRODUCER = 1,
  DEV_WAIT_TIMEOUT_MMA = 2,
  DEV_WAIT_TIMEOUT_EPILOGUE = 3,
  DEV_WAIT_TIMEOUT_DRAIN = 4,
  DEV_BAD_INDEX = 5,
};

__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ __nv_bfloat16 f2bf(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace pcd
