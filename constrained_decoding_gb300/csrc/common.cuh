// Shared definitions of the PCD CUDA library: error words, the operand
// element type and its conversions.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <cstdlib>

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
  DEV_WAIT_TIMEOUT_PROBE = 6,
};

__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Bound on the waits of an abort path for copies and MMAs that were already
// issued.  Those complete on their own, so their drain does not take the
// configurable pipeline limit (which a caller may shrink far below a copy's
// latency); it only guards against a lost completion.
constexpr uint64_t kDrainWaitNs = 4000000000ull;

// Element type of every tensor-core operand and stored activation: fp16.
// The model's weights are bf16 numbers; they are carried as fp16 (every bf16
// value of magnitude >= 2^-17 is exact in fp16, smaller ones land on the
// fp16 subnormal grid, error <= 2^-25).  fp16 rounds activations 8x finer
// than bf16, which the 28-layer decoders need to stay within the parity
// tolerance of the fp32 reference.
using act_t = __half;

__device__ __forceinline__ float a2f(act_t x) { return __half2float(x); }
__device__ __forceinline__ act_t f2a(float x) { return __float2half_rn(x); }

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// silu(g) = g * sigmoid(g) with the fast exponential and division intrinsics
// (a few ulp in fp32; the product is rounded to fp16 right after).  For
// g < -87 the denominator exceeds 2^126 and the quotient flushes to 0, the
// limit of g * e^g.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Programmatic dependent launch: a kernel lets the next one in the stream be
// scheduled early (its prologue overlaps this kernel's tail) and waits for
// the previous one's results before touching memory it produced or reads.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launches `kern` on `stream` with the programmatic-serialisation attribute
// (when enabled), so it may start while the previous kernel finishes.
bool pdl_enabled();
template <class Kern, class... Args>
cudaError_t launch_k(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace pcd
