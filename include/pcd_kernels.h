/* Kernel-level entry points of the PCD library, for testing one device step
 * in isolation against the CPU oracle.  Every pointer is a DEVICE pointer the
 * caller owns; nothing is allocated or freed here.  Each call is enqueued on
 * `stream` (a cudaStream_t, NULL = legacy default stream) and returns without
 * synchronising.  Return value: 0 on success, a negative PCD_ERR_* code
 * (pcd.h) for invalid arguments, or PCD_ERR_CUDA when the launch fails.
 */
#ifndef PCD_KERNELS_H
#define PCD_KERNELS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Epilogue kinds of pcd_k_gemm. */
#define PCD_EPI_BF16 0       /* out fp16 [M][ldo] = A.B^T (16-bit store)                    */
#define PCD_EPI_F32_ADD 1    /* out f32 [M][ldo] += A.B^T (splits must be 1)                */
#define PCD_EPI_F32_ATOMIC 2 /* out f32 [M][ldo] += A.B^T with atomics (any splits)         */
#define PCD_EPI_SWIGLU 3     /* out fp16 [M][ldo]: col f = silu(D[:,2f]) * D[:,2f+1]        */

/* Dense projection on the tensor cores: D[M][N] = A[M][K] . B[N][K]^T with
 * fp16 A and B (row-major, K contiguous, leading dimensions lda/ldb in
 * elements, multiples of 8), fp32 accumulation and a fused epilogue.  This is
 * the contraction of every QKV, output and SwiGLU projection of the decoder
 * (configs: nn.Linear weights [out][in] as B, activations [tokens][in] as A).
 * K must be a multiple of 64, N a multiple of 32.  mt/bn/splits force a
 * tiling (mt in {1,2,4}, bn in {128,256}); mt = 0 lets the library choose;
 * mt = 3 runs CTA pairs that share one tensor-core MMA of 256 rows (each CTA
 * loads its 128 rows of A and half of the B tile).
 * `dev_err` (device int, may be NULL) receives a nonzero code if a pipeline
 * wait times out. */
int pcd_k_gemm(const void* a, int M, int lda, const void* b, int N, int ldb, int K, int epi, void* out, int ldo,
               int mt, int bn, int splits, int* dev_err, void* stream);

/* pcd_k_gemm with A given as two fp16 halves, a_hi + a_lo (a_lo the rounding
 * remainder of an fp32 activation): D = (A_hi + A_lo) . B^T, both products
 * accumulated in one fp32 accumulator from one read of B.  One 128-row tile
 * per CTA; epi PCD_EPI_F32_ADD, PCD_EPI_F32_ATOMIC or PCD_EPI_SWIGLU; bn in
 * {128, 256}. */
int pcd_k_gemm_split(const void* a_hi, const void* a_lo, int M, int lda, const void* b, int N, int ldb, int K, int epi,
                     void* out, int ldo, int bn, int splits, int* dev_err, void* stream);

/* pcd_k_gemm in the weight-streaming form for short activations (M <= 512
 * token rows: the branch rows of one request, How TypeSafe's Jev Might Work,
 * "One forward pass for all fields"): the same D[M][N] = (A + A_lo)[M][K] .
 * B[N][K]^T, computed with B (the weights) as the 256-row side of a tensor-core
 * MMA shared by a pair of CTAs and A as its N side, so every weight tile is
 * read from HBM once.  a_lo (may be NULL) is A's fp16 rounding remainder.
 * epi PCD_EPI_F32_ADD (splits 1), PCD_EPI_F32_ATOMIC (splits >= 1; 0 lets the
 * library choose) or PCD_EPI_SWIGLU (splits 1; B rows 2f, 2f+1 are gate f and
 * up f, out[M][ldo] fp16).  K a multiple of 64, N a multiple of 32, lda/ldb
 * multiples of 8.  Returns 0, -1 for an invalid shape, -10 for a launch
 * error; `dev_err` as in pcd_k_gemm. */
int pcd_k_gemm_swap(const void* a, const void* a_lo, int M, int lda, const void* b, int N, int ldb, int K, int epi,
                    void* out, int ldo, int splits, int* dev_err, void* stream);

/* Fused vocabulary readout: the LM-head contraction z = h . W^T run tile by
 * tile on the tensor cores with an online log-sum-exp over the whole
 * vocabulary and a gather of selected logits, so the [R][V] logits are never
 * written (PCD: A Technical Reference, section 4, stages 3-4: read only the
 * candidate logits; the log-sum-exp turns them into full-vocabulary
 * log-probs).  h [R][d] and w [V][d] are fp16 device matrices (K
 * contiguous, d a multiple of 64, V a multiple of 32).  The gathered pairs are
 * HOST arrays cand_row/cand_tok[n_cand] (row < R, token < V).  Outputs
 * (device): lse[R] = log sum_v exp(z[r][v]) and z_out[n_cand] =
 * z[cand_row][cand_tok], fp32.  `scratch` is a device buffer of at least
 * pcd_k_readout_scratch_bytes(R, V, n_cand) bytes that the call overwrites
 * (per-tile partial maxima and sums, the tile-sorted gather list).  Enqueued
 * on `stream`; the gather list is copied from host memory first, from a
 * buffer that lives only until the call returns, so a call made while
 * `stream` is being captured into a CUDA graph returns PCD_ERR_INVALID_ARG
 * without enqueueing anything. */
int64_t pcd_k_readout_scratch_bytes(int R, int V, int n_cand);
int pcd_k_readout(const void* h, int R, const void* w, int V, int d, const int32_t* cand_row, const int32_t* cand_tok,
                  int n_cand, float* lse, float* z_out, void* scratch, int64_t scratch_bytes, int* dev_err,
                  void* stream);

/* pcd_k_readout without a scratch argument, for callers that cannot allocate
 * device memory: a serving loop whose GPU memory is already reserved by its
 * own pool (a fresh cudaMalloc would fail or fragment it), or code on a
 * latency-critical stream where cudaMalloc / cudaFree would synchronise the
 * device and stall every other stream.  (The pages have no counterpart: it is
 * a property of this library's interface, not of the method.)
 * The scratch is one file-scope __device__ array of
 * PCD_K_READOUT_NOALLOC_MAX_BYTES bytes that every GPU loading the library
 * holds until the process exits.  Inputs, outputs and errors are those of
 * pcd_k_readout; a problem whose pcd_k_readout_scratch_bytes(R, V, n_cand)
 * exceeds the array returns PCD_ERR_OOM without launching anything.  Every
 * call looks up the array's device address (cudaGetSymbolAddress) with the
 * caller's device current; the first call on a device also loads the
 * library's device code there, so make that first call before any stream
 * capture.  No call allocates or frees memory.  Every call
 * shares the one array and leaves its contents behind; each call writes every
 * scratch element it reads before reading it, so nothing needs clearing, but
 * calls that overlap on the GPU (other streams, other threads) race on the
 * array and must be serialised by the caller. */
#define PCD_K_READOUT_NOALLOC_MAX_BYTES (8 * 1024 * 1024)
int pcd_k_readout_noalloc(const void* h, int R, const void* w, int V, int d, const int32_t* cand_row,
                          const int32_t* cand_tok, int n_cand, float* lse, float* z_out, int* dev_err, void* stream);

/* Bounded-wait check (the pages have no counterpart: it exercises this
 * library's failure path, a pipeline partner that never arrives, without
 * faulting or hanging the GPU).  One thread waits on a shared-memory mbarrier
 * that nothing ever arrives on, with the bounded wait every pipeline of the
 * library uses, and gives up once `limit_ns` (0 .. 10^10) has passed: it
 * then records a nonzero code in `dev_err` (a device int, which it never
 * clears) and writes the wait's duration in ns, by the device's global timer,
 * to `elapsed_ns` (a device int64, may be NULL).  Enqueued on `stream`;
 * returns 0, -1 for a bad argument (nothing enqueued) or -10 for a launch
 * error. */
int pcd_k_wait_probe(int64_t limit_ns, int* dev_err, int64_t* elapsed_ns, void* stream);

/* Host-only view of the branch compiler (no GPU needed): compiles `fields`
 * (pcd.h) for a vocabulary of `vocab` tokens into the packed branch batch the
 * branch pass runs (How TypeSafe's Jev Might Work, "When one token is not
 * enough": scaffold tokens plus every internal node of the label trie).
 * sizes[0..7] receives T (branch tokens), R (readout rows), C (child
 * entries), NL (candidate paths), NP (path steps), NA (ancestor entries),
 * NF (fields), NO (labels the paths spell).  When `arrays` is non-NULL,
 * arrays[i] (caller-allocated, sized from a first call with arrays == NULL;
 * a NULL entry is skipped) receives:
 *  0 tok[T], 1 rel[T] (position after the prefix end), 2 anc_off[T+1],
 *  3 anc_idx[NA] (ancestors of each token, itself included, same field),
 *  4 ro_tok[R] (branch token read at each readout row), 5 row_ch[R+1],
 *  6 ch_tok[C] (candidate next token of each child entry), 7 child_row[C],
 *  8 lab_off[NL+1], 9 path[NP] (child entry of each step of each label),
 *  10 fld_lab[NF+1], 11 fld_root[NF] (readout row of each scaffold end),
 *  12 cand_label[NL] (label, within its field, each path spells),
 *  13 fld_out[NF+1] (labels of each field), 14 scoring[NF] (PCD_SCORE_*).
 * ctx[0..n_ctx) (NULL / 0 for none): context tokens written before every
 * field (first field first's answer line), compiled as the first branch
 * tokens.  Returns 0 or the PCD_ERR_* validation code pcd_score would return. */
int pcd_plan_inspect(const void* fields, int n_fields, int vocab, int32_t* sizes, int32_t* const* arrays,
                     const int32_t* ctx, int n_ctx);

/* Host only, no GPU: the answer line first field first writes for `field`
 * (a pcd_field, pcd.h) decided as `label`: its scaffold, the first listed
 * candidate path that spells the label, then sep[0..n_sep) (How TypeSafe's
 * Jev Might Work, "The first key of a JSON object is a special position").
 * Writes at most cap tokens to out (may be NULL with cap = 0) and returns the
 * line's length, or PCD_ERR_INVALID_ARG when no path spells the label. */
int pcd_answer_line(const void* field, int label, const int32_t* sep, int n_sep, int32_t* out, int cap);

#ifdef __cplusplus
}
#endif
#endif
