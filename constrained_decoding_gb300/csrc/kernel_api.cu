// extern "C" kernel-level entry points (include/pcd_kernels.h).
#include <cuda_runtime.h>

#include <cstring>
#include <string>

#include <algorithm>
#include <vector>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "pcd.h"
#include "pcd_kernels.h"
#include "plan.h"
#include "ptx.cuh"

namespace {
// One thread waits, with the pipelines' bounded wait, on a shared-memory
// mbarrier whose single expected arrival never comes.
__global__ void wait_probe_kernel(uint64_t limit_ns, int* err, int64_t* elapsed_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  pcd::mbar_init(&bar, 1);
  pcd::fence_mbar_init();
  const uint64_t t0 = pcd::globaltimer_ns();
  const bool done = pcd::mbar_wait(&bar, 0, limit_ns);
  const uint64_t t1 = pcd::globaltimer_ns();
  if (!done) pcd::record_error(err, pcd::DEV_WAIT_TIMEOUT_PROBE);
  if (elapsed_ns) *elapsed_ns = static_cast<int64_t>(t1 - t0);
}

int device_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}
}  // namespace

extern "C" int pcd_k_gemm(const void* a, int M, int lda, const void* b, int N, int ldb, int K, int epi, void* out,
                          int ldo, int mt, int bn, int splits, int* dev_err, void* stream) {
  // mt = 3 asks for a CTA pair sharing one MMA (see the header)
  bool pair = false;
  if (mt == 3) {
    pair = true;
    mt = 1;
  }
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
    t.pair = pair;
  }
  pcd::GemmShape s{a, M, lda, b, N, ldb, K};
  pcd::EpiArgs e;
  e.out = out;
  e.ldo = ldo;
  const int r = pcd::launch_gemm(s, epi, e, t, static_cast<cudaStream_t>(stream), dev_err, 2000000000ull, sms);
  return r == 0 ? 0 : (r < 0 ? -1 : -10);
}

extern "C" int pcd_k_gemm_split(const void* a_hi, const void* a_lo, int M, int lda, const void* b, int N, int ldb,
                                int K, int epi, void* out, int ldo, int bn, int splits, int* dev_err, void* stream) {
  if (!a_hi || !a_lo || !b || !out || M < 0 || N <= 0 || K <= 0) return -1;
  if (epi != PCD_EPI_F32_ADD && epi != PCD_EPI_F32_ATOMIC && epi != PCD_EPI_SWIGLU) return -1;
  pcd::GemmTiling t;
  t.mt = 1;
  t.bn = bn;
  t.splits = splits < 1 ? 1 : splits;
  pcd::GemmShape s{a_hi, M, lda, b, N, ldb, K, a_lo};
  pcd::EpiArgs e;
  e.out = out;
  e.ldo = ldo;
  const int r = pcd::launch_gemm(s, epi, e, t, static_cast<cudaStream_t>(stream), dev_err, 2000000000ull, device_sms());
  return r == 0 ? 0 : (r < 0 ? -1 : -10);
}

namespace {
// Scratch layout of the readout: partials [n_tiles][R] float2, then the gather
// CSR [n_tiles + 1] int32, then the gather entries [n_cand] int4.  Sized for
// the smallest N tile (the most tiles) so any tiling fits.
int64_t readout_scratch_bytes(int R, int V, int n_cand) {
  const int64_t tiles = (V + 127) / 128;
  const int64_t part = tiles * R * 8;
  const int64_t off = ((tiles + 1) * 4 + 15) / 16 * 16;
  return (part + 255) / 256 * 256 + off + static_cast<int64_t>(n_cand) * 16 + 256;
}

int readout_into(const void* h, int R, const void* w, int V, int d, const int32_t* cand_row, const int32_t* cand_tok,
                 int n_cand, float* lse, float* z_out, void* scratch, int64_t scratch_bytes, int* dev_err,
                 cudaStream_t st) {
  if (!h || !w || !lse || R < 1 || V < 32 || V % 32 || d < 64 || d % 64 || n_cand < 0) return PCD_ERR_INVALID_ARG;
  if (n_cand > 0 && (!cand_row || !cand_tok || !z_out)) return PCD_ERR_INVALID_ARG;
  if (!scratch || scratch_bytes < readout_scratch_bytes(R, V, n_cand)) return PCD_ERR_INVALID_ARG;
  // the gather list is copied from a host vector that lives only until this
  // call returns, so a stream being captured into a graph is refused
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) {
    cudaGetLastError();
    return PCD_ERR_INVALID_ARG;
  }
  if (cap != cudaStreamCaptureStatusNone) return PCD_ERR_INVALID_ARG;
  for (int i = 0; i < n_cand; ++i)
    if (cand_row[i] < 0 || cand_row[i] >= R || cand_tok[i] < 0 || cand_tok[i] >= V) return PCD_ERR_TOKEN_RANGE;
  const int sms = device_sms();
  pcd::GemmTiling t = pcd::choose_tiling(R, V, d, pcd::EPI_READOUT, sms);
  t.splits = 1;
  const int tiles = pcd::gemm_n_tiles(V, t);
  // host: gather entries sorted by vocabulary tile
  std::vector<int> order(n_cand);
  for (int i = 0; i < n_cand; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cand_tok[a] / t.bn < cand_tok[b] / t.bn; });
  const int64_t part_bytes = (static_cast<int64_t>(tiles) * R * 8 + 255) / 256 * 256;
  const int64_t off_bytes = ((static_cast<int64_t>(tiles) + 1) * 4 + 15) / 16 * 16;
  std::vector<int32_t> host(static_cast<size_t>(off_bytes / 4 + 4 * n_cand), 0);
  for (int i : order) host[cand_tok[i] / t.bn + 1]++;
  for (int i = 0; i < tiles; ++i) host[i + 1] += host[i];
  int32_t* g = host.data() + off_bytes / 4;
  for (size_t k = 0; k < order.size(); ++k) {
    const int i = order[k];
    g[4 * k + 0] = cand_tok[i] % t.bn;
    g[4 * k + 1] = cand_row[i];
    g[4 * k + 2] = i;
    g[4 * k + 3] = 0;
  }
  uint8_t* base = static_cast<uint8_t*>(scratch);
  float2* part = reinterpret_cast<float2*>(base);
  int32_t* dev_lists = reinterpret_cast<int32_t*>(base + part_bytes);
  if (cudaMemcpyAsync(dev_lists, host.data(), host.size() * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return PCD_ERR_CUDA;
  pcd::GemmShape s{h, R, d, w, V, d, d};
  pcd::EpiArgs e;
  e.part = part;
  e.gather_off = dev_lists;
  e.gather = reinterpret_cast<const int4*>(dev_lists + off_bytes / 4);
  e.z_out = z_out;
  int r = pcd::launch_gemm(s, pcd::EPI_READOUT, e, t, st, dev_err, 2000000000ull, sms);
  if (r != 0) return r < 0 ? PCD_ERR_INVALID_ARG : PCD_ERR_CUDA;
  r = pcd::launch_lse_combine(part, tiles, R, lse, st);
  return r == 0 ? PCD_OK : PCD_ERR_CUDA;
}
}  // namespace

extern "C" int64_t pcd_k_readout_scratch_bytes(int R, int V, int n_cand) {
  if (R < 1 || V < 1 || n_cand < 0) return 0;
  return readout_scratch_bytes(R, V, n_cand);
}

extern "C" int pcd_k_readout(const void* h, int R, const void* w, int V, int d, const int32_t* cand_row,
                             const int32_t* cand_tok, int n_cand, float* lse, float* z_out, void* scratch,
                             int64_t scratch_bytes, int* dev_err, void* stream) {
  return readout_into(h, R, w, V, d, cand_row, cand_tok, n_cand, lse, z_out, scratch, scratch_bytes, dev_err,
                      static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------ allocation-free readout
// The readout's scratch for callers that cannot allocate: a fixed array in
// device global memory, shared by every call on a device.  Host code may not
// use the symbol's address directly (in host code it names a host-side
// stand-in), so every call looks up its device address with the caller's
// device current.  Looking it up each time (a host-side table lookup that
// allocates nothing) keeps the address right after cudaDeviceReset or a
// re-created primary context, when the module is loaded again elsewhere.
static __device__ __align__(256) unsigned char g_readout_scratch[PCD_K_READOUT_NOALLOC_MAX_BYTES];

namespace {
int noalloc_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_readout_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return PCD_ERR_CUDA;
  }
  *out = p;
  return PCD_OK;
}
}  // namespace

extern "C" int pcd_k_readout_noalloc(const void* h, int R, const void* w, int V, int d, const int32_t* cand_row,
                                     const int32_t* cand_tok, int n_cand, float* lse, float* z_out, int* dev_err,
                                     void* stream) {
  if (R < 1 || V < 1 || n_cand < 0) return PCD_ERR_INVALID_ARG;
  const int64_t need = readout_scratch_bytes(R, V, n_cand);
  if (need > static_cast<int64_t>(PCD_K_READOUT_NOALLOC_MAX_BYTES)) return PCD_ERR_OOM;
  void* scratch = nullptr;
  const int rc = noalloc_scratch(&scratch);
  if (rc != PCD_OK) return rc;
  return readout_into(h, R, w, V, d, cand_row, cand_tok, n_cand, lse, z_out, scratch,
                      static_cast<int64_t>(PCD_K_READOUT_NOALLOC_MAX_BYTES), dev_err, static_cast<cudaStream_t>(stream));
}

extern "C" int pcd_answer_line(const void* field, int label, const int32_t* sep, int n_sep, int32_t* out, int cap) {
  if (!field || cap < 0) return PCD_ERR_INVALID_ARG;
  std::vector<int32_t> line;
  const int rc = pcd::answer_line(*static_cast<const pcd_field*>(field), label, sep, n_sep, &line);
  if (rc != PCD_OK) return rc;
  for (int i = 0; out && i < cap && i < static_cast<int>(line.size()); ++i) out[i] = line[i];
  return static_cast<int>(line.size());
}

extern "C" int pcd_plan_inspect(const void* fields, int n_fields, int vocab, int32_t* sizes, int32_t* const* arrays,
                                const int32_t* ctx, int n_ctx) {
  if (!sizes || vocab < 1) return PCD_ERR_INVALID_ARG;
  pcd::HostPlan p;
  std::string msg;
  const int rc = pcd::compile_fields(static_cast<const pcd_field*>(fields), n_fields, vocab, &p, &msg, ctx, n_ctx);
  if (rc != PCD_OK) return rc;
  sizes[0] = p.T;
  sizes[1] = p.R;
  sizes[2] = p.n_children;
  sizes[3] = p.n_labels;
  sizes[4] = p.n_path;
  sizes[5] = static_cast<int32_t>(p.anc_idx.size());
  sizes[6] = p.n_fields;
  sizes[7] = p.n_out;
  if (arrays) {
    const std::vector<int32_t>* src[15] = {&p.tok,     &p.rel,       &p.anc_off,    &p.anc_idx, &p.ro_tok,
                                          &p.row_ch,  &p.ch_tok,    &p.child_row,  &p.lab_off, &p.path,
                                          &p.fld_lab, &p.fld_root,  &p.cand_label, &p.fld_out, &p.scoring};
    for (int i = 0; i < 15; ++i)
      if (arrays[i] && !src[i]->empty()) std::memcpy(arrays[i], src[i]->data(), src[i]->size() * sizeof(int32_t));
  }
  return PCD_OK;
}

extern "C" int pcd_k_wait_probe(int64_t limit_ns, int* dev_err, int64_t* elapsed_ns, void* stream) {
  if (limit_ns < 0 || limit_ns > 10000000000ll || !dev_err) return -1;
  wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint64_t>(limit_ns), dev_err,
                                                                    elapsed_ns);
  return cudaGetLastError() == cudaSuccess ? 0 : -10;
}

extern "C" int pcd_k_gemm_swap(const void* a, const void* a_lo, int M, int lda, const void* b, int N, int ldb, int K,
                               int epi, void* out, int ldo, int splits, int* dev_err, void* stream) {
  if (!a || !b || !out || M < 0 || N <= 0 || K <= 0) return -1;
  if (epi != PCD_EPI_F32_ADD && epi != PCD_EPI_F32_ATOMIC && epi != PCD_EPI_SWIGLU) return -1;
  const int sms = device_sms();
  if (splits < 1) splits = pcd::swap_splits(N, K, epi, sms);
  pcd::SwapShape s{b, N, ldb, a, M, lda, K, a_lo, false};
  pcd::EpiArgs e;
  e.out = out;
  e.ldo = ldo;
  const int r = pcd::launch_gemm_swap(s, epi, e, splits, static_cast<cudaStream_t>(stream), dev_err, 2000000000ull, sms);
  return r == 0 ? 0 : (r < 0 ? -1 : -10);
}
