// Host launchers of the non-GEMM device steps of the PCD hot path.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace pcd {

using act_t = __half;  // same as common.cuh

// x[t][0..d) = E[ids[t]][0..d) as fp32 (the residual stream starts here).
int launch_embed(const int32_t* ids, int n, const act_t* E, int d, int vocab, float* x, int* err, cudaStream_t s);

// out[r] = fp16( x[src] / sqrt(mean(x[src]^2) + eps) * gain ), src = rows ? rows[r] : r;
// out_lo (optional) receives the rounding remainder fp16(y - out), so out + out_lo ~ y.
int launch_rmsnorm(const float* x, int ldx, const int32_t* rows, int n, int d, const float* gain, float eps, act_t* out,
                   int ldo, cudaStream_t s, act_t* out_lo = nullptr);

struct RopeArgs {
  const float* qkv;       // [n][ldqkv] fp32: q heads, then k heads, then v heads
  int ldqkv, n, Hq, Hkv, DH;
  const float2* cs;       // [max_pos][DH/2] (cos, sin)
  int max_pos;
  const int32_t* rel;     // position of token t = base + (rel ? rel[t] : t)
  int base;
  act_t* q;                // [n][Hq][DH]
  act_t* k_dst;            // K row of token t: k_dst + (h * kv_head_stride + kv_row0 + t) * DH
  act_t* v_dst;
  int64_t kv_head_stride; // elements between KV heads
  int kv_row0;
  int* err;
  int clear_qkv = 0;      // zero the consumed qkv values (the next split-K projection accumulates into them)
  act_t* q_lo = nullptr;  // optional fp16 rounding remainders of q, k and v (same layouts)
  act_t* k_lo = nullptr;
  act_t* v_lo = nullptr;
};
int launch_rope_kv(const RopeArgs& a, cudaStream_t s);

struct AttnArgs {
  const act_t* q;            // [tok0 + n_tok][Hq][DH]: this launch's query tokens are tok0 .. tok0+n_tok-1
  int n_tok, Hq, Hkv, DH;
  int tok0;                 // first token (also offsets rel, out and the partial rows)
  int part_rows;            // rows of the partial arrays per (split, KV head): all tokens x G
  const act_t* k;            // this layer's keys: k + (h * kv_head_stride + j) * DH, j < n_keys
  const act_t* v;
  int64_t kv_head_stride;
  int n_keys;
  const int32_t* rel;       // query position = base + (rel ? rel[t] : t); key j is visible iff j <= position
  int base;
  int n_splits, split_len;  // keys are cut into n_splits ranges of split_len (a multiple of 64)
  float scale_log2;         // log2(e) / sqrt(DH)
  act_t* out;                // n_splits == 1 and !partial: out[t][h * DH + d] (normalised)
  int ld_out;
  float* part_o;            // partial: [split][Hkv][part_rows][DH] normalised by the split's own l
  float2* part_ml;          // partial: [split][Hkv][part_rows] (max, sum) in log2 units
  int partial;
  int causal_heavy_first;   // schedule the row blocks with the most keys first
};
int launch_attention(const AttnArgs& a, cudaStream_t s);

struct MergeArgs {
  const act_t* q;            // [n_tok][Hq][DH]
  int n_tok, Hq, Hkv, DH;
  const float* part_o;      // prefix partials from launch_attention (partial = 1)
  const float2* part_ml;
  int n_splits;
  const act_t* kb;           // branch keys/values [Hkv][n_tok][DH]
  const act_t* vb;
  const int32_t* anc_off;   // [n_tok + 1]: ancestors (incl. itself) of token t in the branch batch;
                            // nullptr: only combine the key splits (split prefill attention)
  const int32_t* anc_idx;
  float scale_log2;
  act_t* out;                // out[t][h * DH + d]
  int ld_out;
  act_t* out_lo = nullptr;   // optional fp16 rounding remainder of out
};
int launch_branch_merge(const MergeArgs& a, cudaStream_t s);

// Tree attention: every query of a pass in one launch, normalised output
// written directly.  Prefix queries are causal (query t sees prefix keys
// 0..t); branch queries see every prefix key plus their own ancestors in the
// branch batch (scaffold chain and trie path, themselves included).  Queries
// are tiled by whole tokens (tpt tokens x G query heads <= 64 rows per tile);
// a branch tile's ancestor keys are the ascending union of its tokens'
// ancestor lists, cut into 64-key chunks, with a 64-bit visibility mask per
// (chunk, token of the tile).  csk CTAs (a thread-block cluster) share one
// (tile, KV head) and split its key blocks; they combine their partial
// softmax states through distributed shared memory.
// The prefix cache of one request of a batch (tensor-core tree attention):
// layer l's keys of KV head h at k + ((l * Hkv + h) * cap + j) * DH, j < n_keys.
struct SegKV {
  const act_t* k;
  const act_t* v;
  const act_t* k_lo;  // remainders, or nullptr
  const act_t* v_lo;
  int64_t cap;
  int32_t n_keys;
  int32_t pad;
};

struct TreeAttnArgs {
  const act_t* q;               // [rows][Hq][DH]: prefix queries at rows 0..n_pf-1, branch queries at br_row0..
  act_t* out;                   // out[row][h * DH + d]
  act_t* out_lo = nullptr;      // optional fp16 rounding remainder of out
  int ld_out;
  int Hq, Hkv, DH;
  int tpt;                      // query tokens per tile
  int n_pf, n_pf_tiles;         // causal prefix queries: query i sits at position pf_pos0 + i, sees keys 0 .. that
  int pf_pos0 = 0;
  int n_br, n_br_tiles, br_row0;
  const act_t* k;               // this layer's prefix keys: k + (h * kv_head_stride + j) * DH, j < n_keys
  const act_t* v;
  int64_t kv_head_stride;
  int n_keys;
  const act_t* kb;              // branch keys/values [Hkv][n_br][DH]
  const act_t* vb;
  const act_t* q_lo = nullptr;   // fp16 remainders of q, kb, vb (tensor-core kernel only), or nullptr
  const act_t* kb_lo = nullptr;
  const act_t* vb_lo = nullptr;
  const int32_t* tile_tok;                  // [n_br_tiles][3]: first branch token, tokens, request of each tile
  const SegKV* segs = nullptr;              // per request of a batch (branch tiles read their request's
                                            // prefix keys by cp.async), or nullptr: k / v / n_keys above
  int layer = 0;                            // layer of segs' caches
  const int32_t* tile_chunk_off;            // [n_br_tiles + 1] ancestor chunks of each branch tile
  const int32_t* tile_keys;                 // [chunks][64] branch key index, -1 past the union's end
  const unsigned long long* tile_mask;      // [chunks][tpt] bit i: key i of the chunk is visible to the token
  float scale_log2;                         // log2(e) / sqrt(DH)
  int csk;                                  // CTAs (cluster size) per (tile, KV head): 1 .. 8
  int lo_terms = 3;                         // with remainders: 1 = S takes Q K_lo + Q_lo K, 2 = O takes
                                            // P V_lo + P_lo V
};
int launch_tree_attention(const TreeAttnArgs& a, cudaStream_t s);
// The same on the tcgen05 tensor cores, head dim 128, tiles of tpt x G <= 128
// rows.  tmK / tmV map the prefix cache (make_kv_map: rows past n_keys read
// as zero); `layer` selects its layer.  With q_lo set, q, k, v and the
// attention weights carry their fp16 remainders (tmKlo / tmVlo map the
// cache's, kb_lo / vb_lo hold the branch keys').  Pipeline waits give up
// after wait_ns and record an error code in *err.
int launch_tree_attention_tc(const TreeAttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const CUtensorMap* tmKlo, const CUtensorMap* tmVlo, int layer, uint64_t wait_ns, int* err,
                             cudaStream_t s);
// CTAs per (tile, KV head) for the warp-MMA (tc = false) or tensor-core
// kernel: the key blocks of the heaviest tile (max_blocks) against the waves
// of CTAs the cluster split adds.
int tree_attention_csk(int tiles, int Hkv, int max_blocks, int sms, bool tc);
// CTAs of the tensor-core tree attention that can be resident at once when
// launched in clusters of csk (1..8); 0 if the query fails.
int tree_attention_tc_slots(int csk);

// lse[r] = log sum_tiles sum exp(z) from per-tile (max, sum exp(z - max)).
int launch_lse_combine(const float2* part, int n_tiles, int R, float* lse, cudaStream_t s);

struct ScoreArgs {
  const float* z;           // gathered candidate logits, one per child entry
  const float* lse;         // [R]
  const int32_t* child_row; // readout row of each child entry
  const int32_t* lab_off;   // [n_paths_total + 1] CSR into path_entries
  const int32_t* path;      // child entry of every step of every label path
  const int32_t* fld_lab;   // [n_fields + 1] candidate paths of each field
  const int32_t* fld_root;  // root readout row of each field
  const int32_t* row_ch;    // [R + 1] child entries of each readout row
  const float* temp;        // [n_fields]
  const int32_t* scoring;   // [n_fields] PCD_SCORE_SUM / _MEAN / _LEVEL
  const int32_t* cand_label;  // [n_paths_total] label (within its field) each candidate path spells
  const int32_t* fld_out;   // [n_fields + 1] outputs (labels) of each field
  int n_fields;
  float* out_field;         // [n_fields][8]: label, mass, log_mass, margin, first_mass, n_labels, 0, 0
  float* out_probs;         // [n_labels_total]
  float* out_logprobs;      // [n_labels_total]
};
int launch_score(const ScoreArgs& a, cudaStream_t s);

}  // namespace pcd
