// extern "C" kernel-level entry points (include/pcd_kernels.h).
#include <cuda_runtime.h>

#include <cstring>
#include <string>

#include "gemm.h"
#include "pcd_kernels.h"
#include "plan.h"

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

extern "C" int pcd_plan_inspect(const void* fields, int n_fields, int vocab, int32_t* sizes, int32_t* const* arrays) {
  if (!sizes || vocab < 1) return PCD_ERR_INVALID_ARG;
  pcd::HostPlan p;
  std::string msg;
  const int rc = pcd::compile_fields(static_cast<const pcd_field*>(fields), n_fields, vocab, &p, &msg);
  if (rc != PCD_OK) return rc;
  sizes[0] = p.T;
  sizes[1] = p.R;
  sizes[2] = p.n_children;
  sizes[3] = p.n_labels;
  sizes[4] = p.n_path;
  sizes[5] = static_cast<int32_t>(p.anc_idx.size());
  sizes[6] = p.n_fields;
  if (arrays) {
    const std::vector<int32_t>* src[12] = {&p.tok,     &p.rel,       &p.anc_off, &p.anc_idx, &p.ro_tok,  &p.row_ch,
                                          &p.ch_tok,  &p.child_row, &p.lab_off, &p.path,    &p.fld_lab, &p.fld_root};
    for (int i = 0; i < 12; ++i)
      if (arrays[i] && !src[i]->empty()) std::memcpy(arrays[i], src[i]->data(), src[i]->size() * sizeof(int32_t));
  }
  return PCD_OK;
}
