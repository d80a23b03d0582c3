// Host interface of the tcgen05 GEMM: D = A . B^T with A [M][K] and B [N][K]
// 16-bit, both K-contiguous, fp32 accumulation in tensor memory, and one of a
// few fused epilogues.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace pcd {

using act_t_storage = __half;

enum EpiKind : int {
  EPI_BF16 = 0,        // out 16-bit [M][ldo] = D
  EPI_F32_ADD = 1,     // out f32 [M][ldo] += D (one K split: plain read-modify-write)
  EPI_F32_ATOMIC = 2,  // out f32 [M][ldo] += D with atomics (any number of K splits)
  EPI_SWIGLU = 3,      // D columns (2f, 2f+1) = (gate_f, up_f); out 16-bit [M][ldo]: silu(gate) * up
  EPI_READOUT = 4,     // vocabulary readout: per (row, N tile) max and sum-exp, plus gathered logits
  EPI_F32_STORE = 5,   // out f32 [M][ldo] = D (one K split)
  EPI_QKV_ROPE = 6,    // q/k/v projection (head dim 128): rotary embedding applied, q to q_out, k/v to
                       // the cache (rows < split_row) or the branch scratch (rows >= split_row)
};

struct GemmShape {
  const void* a; int a_rows; int a_ld;   // A: a_rows x K, leading dim in elements
  const void* b; int b_rows; int b_ld;   // B: b_rows x K
  int K;
  const void* a_lo = nullptr;            // optional low half of A (same layout): D = (A + A_lo) . B^T
  int lo_row0 = 0;                       // 128-row tiles entirely below this row skip the low half
  bool b_const = false;                  // B is never written by an earlier kernel in the stream (weights):
                                         // its first tiles may load before the programmatic dependency wait
};

struct EpiArgs {
  void* out = nullptr;            // output base (16-bit or f32)
  int ldo = 0;                    // leading dimension of out, in elements
  void* out_lo = nullptr;         // EPI_SWIGLU: optional fp16 rounding remainder of out (same layout)
  float2* part = nullptr;         // EPI_READOUT: [n_tiles_n][M] (max, sum exp(z - max))
  const int* gather_off = nullptr;  // EPI_READOUT: [n_tiles_n + 1] CSR over gather entries
  const int4* gather = nullptr;   // EPI_READOUT: (column in tile, row, output index, 0)
  float* z_out = nullptr;         // EPI_READOUT: gathered logits
  // EPI_QKV_ROPE: D columns are Hq query heads, then Hkv key heads, then Hkv value heads of 128
  act_t_storage* q_out = nullptr;  // [M][Hq * 128]
  int n_q_heads = 0, n_kv_heads = 0;
  const float2* rope_cs = nullptr;  // [64][max_pos] (cos, sin) of pair i at position pos: rope_cs[i * max_pos + pos]
  int max_pos = 0;
  int split_row = 0;              // rows < split_row use destination 0, the rest destination 1
  act_t_storage* kv_k[2] = {nullptr, nullptr};  // key of (head h, row r') at kv_k[d] + (h * kv_stride[d] + kv_row0[d] + r') * 128
  act_t_storage* kv_v[2] = {nullptr, nullptr};
  // optional fp16 rounding remainders of q, k and v (same layouts as q_out, kv_k, kv_v)
  act_t_storage* q_lo = nullptr;
  act_t_storage* kv_k_lo[2] = {nullptr, nullptr};
  act_t_storage* kv_v_lo[2] = {nullptr, nullptr};
  int64_t kv_stride[2] = {0, 0};
  int kv_row0[2] = {0, 0};
  int pos_base[2] = {0, 0};       // position = pos_base[d] + (pos_rel[d] ? pos_rel[d][r'] : r'), r' = row - (d ? split_row : 0)
  const int32_t* pos_rel[2] = {nullptr, nullptr};
  int* err = nullptr;
};

struct GemmTiling {
  int mt = 1;       // 128-row M tiles per CTA work unit (1, 2 or 4)
  int bn = 256;     // N tile (128 or 256)
  int splits = 1;   // K splits (EPI_F32_ATOMIC only when > 1)
  bool pair = false;  // a CTA pair (cta_group::2 MMA, M = 256) per work unit; mt = 1
};

// Picks a tiling for the shape and epilogue on an `sms`-SM device.
GemmTiling choose_tiling(int M, int N, int K, int epi, int sms);

// Number of N tiles for a tiling (the readout partial array's first dimension).
inline int gemm_n_tiles(int N, const GemmTiling& t) { return (N + t.bn - 1) / t.bn; }

// Launches D = A . B^T with the epilogue on `stream`.  Returns a cudaError_t
// value (0 on success); -1 for an invalid shape or tiling.
int launch_gemm(const GemmShape& s, int epi, const EpiArgs& e, const GemmTiling& t, cudaStream_t stream,
                int* dev_err, uint64_t wait_ns, int sms);

// ---------------------------------------------------------------- weight-streaming form
// D^T = W . X^T for at most kSwapMaxRows token rows: the weights are the
// 256-row side of a CTA-pair MMA and the tokens its N side, so every weight
// tile is read once (instead of once per 128-token tile).
constexpr int kSwapMaxRows = 512;
struct SwapShape {
  const void* w; int w_rows; int w_ld;   // weights [w_rows][K] (output features), leading dim in elements
  const void* x; int x_rows; int x_ld;   // activations [x_rows][K]
  int K;
  const void* x_lo = nullptr;            // optional activation remainder (same layout): D = W . (X + X_lo)^T
  bool w_const = false;                  // W is never written by an earlier kernel in the stream
};
// K splits for the shape (1 unless epi is EPI_F32_ATOMIC).
int swap_splits(int w_rows, int K, int epi, int sms);
// Launches the weight-streaming GEMM; epi is EPI_F32_ADD (splits 1),
// EPI_F32_ATOMIC or EPI_SWIGLU (splits 1), writing out[t][n] (n a weight row;
// SwiGLU: out[t][f] from rows 2f, 2f+1).  Returns a cudaError_t value, -1 for
// an invalid shape.
int launch_gemm_swap(const SwapShape& s, int epi, const EpiArgs& e, int splits, cudaStream_t stream, int* dev_err,
                     uint64_t wait_ns, int sms);

// Loads cuTensorMapEncodeTiled from the driver; false if it is unavailable.
bool tma_init();
// 2-D tensor map of a 16-bit row-major matrix [rows][>= cols] (leading dim
// `ld` elements), box 64 columns x box_rows rows, 128-byte swizzle; cached.
bool make_tile_map(CUtensorMap* m, const void* ptr, int rows, int cols, int ld, int box_rows);
// Tensor map over a 16-bit KV cache laid out [layer][head][row][dh] (head
// stride head_rows rows, layer stride layer_elems elements): dimensions
// {dh, n_rows, n_heads, n_layers}, so rows at or past n_rows read as zero;
// box {64, 64, 1, 1} with 128-byte swizzling.  Cached by its arguments.
bool make_kv_map(CUtensorMap* m, const void* base, int dh, int n_rows, int n_heads, int64_t head_rows, int n_layers,
                 int64_t layer_elems);
// 3-D map of a row-major [n_rows][n_heads][dh] fp16 tensor (q: a token's
// heads side by side) with boxes of 64 x box_heads x box_rows, 128-byte
// swizzle: the rows land as box_rows x box_heads consecutive 128-byte rows of
// one 64-column half.  Cached by its arguments.
bool make_q_map(CUtensorMap* m, const void* base, int dh, int n_heads, int n_rows, int box_heads, int box_rows);

}  // namespace pcd
