// extern "C" kernel-level entry points (include/pcd_kernels.h).
#include <cuda_runtime.h>

#include "gemm.h"
#include "pcd_kernels.h"

namespace {
int device_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}
}  // namespace

extern "C" int pcd_k_gemm(const void* a, int M, int lda, const void* b, int N, int ldb, int K, int epi, void* out,
                          int ldo, int mt, int bn, int splits, int* dev_err, void* stream) {
  if (!a || !b || !out || M < 0 || N <= 0 || K <= 0) return -1;
  if (epi < PCD_EPI_BF16 || epi > PCD_EPI_SWIGLU) return -1;
  const int sms = device_sms();
  pcd::GemmTiling t;
  if (mt == 0) {
    t = pcd::choose_tiling(M, N, K, epi, sms);
  } else {
    t.mt = mt;
    t.bn = bn;
    t.splits = splits < 1 ? 1 : splits;
  }
  pcd::GemmShape s{a, M, lda, b, N, ldb, K};
  pcd::EpiArgs e;
  e.out = out;
  e.ldo = ldo;
  const int r = pcd::launch_gemm(s, epi, e, t, static_cast<cudaStream_t>(stream), dev_err, 2000000000ull, sms);
  return r == 0 ? 0 : (r < 0 ? -1 : -10);
}
