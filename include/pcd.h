/* pcd.h -- C ABI of the GB300 parallel constrained decoding (PCD) library.
 *
 * The method (How TypeSafe's Jev Might Work: Parallel Constrained Decoding
 * from Scratch, "The idea: parallel constrained decoding"; PCD: A Technical
 * Reference, section 4 "The algorithm"): a decoder LM prefills a shared
 * prompt once into a KV cache; each boolean or enum field of a closed schema
 * becomes a short branch row (its scaffold tokens, then the candidate label
 * tokens laid out as a trie); all rows run in ONE batched forward pass that
 * attends to the shared prefix KV plus each row's own causal ancestors; at
 * every readout position the full-vocabulary logits give candidate log-probs,
 * and each label's score is the sum of its tokens' log-probs
 * (How TypeSafe's Jev Might Work, "When one token is not enough").  The
 * field's answer is the candidate-only softmax of the label scores at
 * temperature T, its argmax (first declared label on ties, the rule PCD: A
 * Technical Reference suggests in its FAQ) and the candidate mass
 * ("And you get confidence for free").  Tokenisation and JSON assembly stay
 * with the caller.
 *
 * Conventions
 *  - Every call returns PCD_OK (0) or a negative PCD_ERR_* code; outputs are
 *    untouched on error.  pcd_last_error() gives a thread-local detail string.
 *  - Host pointers unless a name ends in _device.  Inputs are borrowed for the
 *    duration of the call only (copied).  Result arrays are caller-allocated.
 *    Handles are freed only by pcd_*_free.
 *  - A model owns one CUDA stream (the one given at load; for NULL the
 *    library creates a blocking stream, which is ordered with the legacy
 *    default stream); every call is ordered on it.  Passes run as CUDA
 *    graphs captured on first use (environment PCD_GRAPHS=0 disables them).  Calls that return host
 *    results synchronise that stream; *_device calls only enqueue.
 *  - A cache is immutable once created: it may be scored many times and
 *    extended into new caches.
 *  - There is no CPU fallback: without an sm_100-family GPU (sm_103a code)
 *    pcd_load_weights fails with PCD_ERR_CUDA.
 *  - A model is not thread-safe: serialise calls on one model.
 */
#ifndef PCD_H
#define PCD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
#define PCD_OK 0
#define PCD_ERR_INVALID_ARG -1
#define PCD_ERR_TOO_MANY_CANDIDATES -2 /* > 255 labels in a field (PCD: A Technical Reference, section 6) */
#define PCD_ERR_TOO_FEW_CANDIDATES -3  /* < 2 labels (its pre-deployment checklist, 13.1)               */
#define PCD_ERR_EMPTY_LABEL -4         /* a label with no tokens                                         */
#define PCD_ERR_DUPLICATE_LABEL -5     /* two labels with the same token path                            */
#define PCD_ERR_PREFIX_LABEL -6        /* a label's path is a strict prefix of another's                 */
#define PCD_ERR_TOKEN_RANGE -7         /* a token id outside [0, vocab)                                  */
#define PCD_ERR_SHAPE_MISMATCH -8      /* cache of another model, or a shape the kernels do not support  */
#define PCD_ERR_OOM -9                 /* device or pinned-host allocation failed                        */
#define PCD_ERR_CUDA -10               /* a CUDA call failed, or no suitable GPU                         */
#define PCD_ERR_DEVICE_TIMEOUT -11     /* a kernel's bounded pipeline wait expired                       */
#define PCD_ERR_BAD_WEIGHTS -12        /* weight file missing, truncated or inconsistent                 */
#define PCD_ERR_TOO_LONG -13           /* a position beyond the model's max_positions                    */

/* dtypes of pcd_load_weights_host matrices.  On the device every matrix is
 * carried as fp16 (round to nearest even): bf16 values of magnitude >= 2^-17
 * convert exactly, smaller ones within 2^-25.  Activations and the KV cache
 * are fp16 too; accumulation and the residual stream are fp32. */
#define PCD_DTYPE_F32 1
#define PCD_DTYPE_BF16 2

typedef struct pcd_model pcd_model; /* opaque, library-owned */
typedef struct pcd_cache pcd_cache; /* opaque: the prefix KV snapshot */
typedef struct pcd_plan pcd_plan;   /* opaque: a compiled, device-resident branch batch */

/* Decoder shape (a Qwen2.5-style pre-norm decoder: RMSNorm, bias-free q/k/v/o,
 * rotate-half RoPE, grouped-query attention, SwiGLU MLP, final RMSNorm). */
typedef struct {
  int n_layers, d_model, n_q_heads, n_kv_heads, head_dim, d_ff, vocab;
  float rms_eps, rope_theta;
  int tied_embedding; /* 1: the LM head is the embedding matrix */
  int max_positions;  /* RoPE table size; 0 = 32768 */
} pcd_model_config;

/* One field of a closed schema (PCD: A Technical Reference, section 6:
 * boolean or enum, 2..255 choices, flat).
 *  scaffold[n_scaffold]: the row's tokens up to the readout, n_scaffold >= 1;
 *    its last token predicts each label's first token ("Tokens are not
 *    characters", How TypeSafe's Jev Might Work: end the row where the
 *    labels diverge).
 *  cand_tokens / cand_offsets: label c is cand_tokens[cand_offsets[c] ..
 *    cand_offsets[c+1]), n_cands + 1 offsets, cand_offsets[0] = 0.  Labels
 *    may share prefixes (scored through the trie) but no label may be a
 *    strict prefix of another: append the terminator token the tokenizer
 *    writes after a value.
 *  temperature: T > 0 divides the label scores before the softmax; 0 means 1.
 *  scoring: how a label's token log-probs make its score s_c
 *    PCD_SCORE_SUM   their sum, log P(label) (default, zero-initialised);
 *    PCD_SCORE_MEAN  their mean, sum / n_tokens (PCD From First Principles,
 *                    "Multi-token candidates": length-normalised);
 *    PCD_SCORE_LEVEL the log of the product, over the trie levels on the
 *                    label's path, of the next token's probability
 *                    renormalised over the tokens the field allows there
 *                    (PCD: A Technical Reference, "Resolve shared prefixes
 *                    level by level").
 *    Any other value is PCD_ERR_INVALID_ARG.
 *  cand_label / n_labels: NULL / ignored when every candidate path is its
 *    own label.  Otherwise cand_label[c] in [0, n_labels) names the label
 *    that path c spells, so one label may have several spellings ("Small
 *    models quote their booleans", How TypeSafe's Jev Might Work: a bare and
 *    a quoted value are one answer); every label needs at least one path,
 *    2 <= n_labels <= n_cands.  Each path is scored by the rule above and a
 *    label's score is the log-sum-exp of its paths' scores. */
#define PCD_SCORE_SUM 0
#define PCD_SCORE_MEAN 1
#define PCD_SCORE_LEVEL 2
typedef struct {
  const int32_t* scaffold;
  int n_scaffold;
  const int32_t* cand_tokens;
  const int32_t* cand_offsets;
  int n_cands;
  float temperature;
  int scoring;
  const int32_t* cand_label;
  int n_labels;
} pcd_field;

/* Per-field result.  probs / logprobs are caller-owned arrays of one float
 * per label (n_cands, or n_labels with cand_label; may be NULL to skip).
 * logprobs[c] = s_c, the label's score under the field's scoring rule (PCD_SCORE_SUM: the sum of its full-vocabulary
 * token log-probs); probs[c] = softmax(s / T)[c]; label = argmax (lowest
 * index on exact ties); margin = s_top1 - s_top2.  Whatever the rule,
 * mass = sum over the candidate paths of the full-vocabulary product of the
 * path's token probabilities, log_mass = log(mass), and first_mass =
 * probability that the next token after the scaffold starts any allowed
 * path. */
typedef struct {
  float* probs;
  float* logprobs;
  int32_t label;
  float mass, log_mass, margin, first_mass;
} pcd_field_result;

/* Phase timings (CUDA events on the model stream; when the branch pass runs
 * as a CUDA graph, branch_ms covers the readout too and readout_ms is 0) and
 * the true number of sequential forward passes (PCD From First Principles, "Where the two real
 * implementations disagree": count what ran, do not hard-code it). */
typedef struct {
  float prefill_ms, compile_ms, branch_ms, readout_ms, total_ms;
  int forward_passes;
  int branch_tokens, readout_rows;
  int64_t h2d_bytes, d2h_bytes; /* host<->device bytes this call copied */
} pcd_stats;

/* ------------------------------------------------------------------ models */
/* Loads a .pcdw weight file: a 64-byte header (b"PCDW", u32 version = 1,
 * u32 dtype 1=f32/2=bf16, u32 n_layers, d_model, n_q_heads, n_kv_heads,
 * head_dim, d_ff, vocab, tied, reserved, f32 rms_eps, f32 rope_theta), then
 * embed [V][d]; per layer attn_norm [d] f32, wq [Hq*dh][d], wk [Hkv*dh][d],
 * wv [Hkv*dh][d], wo [d][Hq*dh], mlp_norm [d] f32, w_gate [F][d],
 * w_up [F][d], w_down [d][F]; final_norm [d] f32; lm_head [V][d] if untied.
 * `cfg` may be NULL (the header's shape is used) or must match the header.
 * `stream` is a cudaStream_t the model keeps.  Errors: PCD_ERR_BAD_WEIGHTS,
 * PCD_ERR_SHAPE_MISMATCH, PCD_ERR_OOM, PCD_ERR_CUDA. */
int pcd_load_weights(const pcd_model_config* cfg, const char* path, void* stream, pcd_model** out);

/* Same, from host arrays in the order above: tensors[0] = embed, then per
 * layer 9 pointers (attn_norm, wq, wk, wv, wo, mlp_norm, w_gate, w_up,
 * w_down), then final_norm, then lm_head if untied.  Matrices are `dtype`
 * (PCD_DTYPE_F32 or PCD_DTYPE_BF16 bit patterns), norm gains always f32. */
int pcd_load_weights_host(const pcd_model_config* cfg, const void* const* tensors, int dtype, void* stream,
                          pcd_model** out);

void pcd_model_free(pcd_model* m);

/* Device bytes of one token's K and V over all layers: layers x 2 x KV heads
 * x head dim x 2 for 16-bit k and v ("The piece of plumbing you need: the KV
 * cache", How TypeSafe's Jev Might Work), twice that when the cache also
 * keeps their fp16 rounding remainders (head dim 128 with the default
 * precision: PCD_SPLIT_ACT bit 256). */
int64_t pcd_kv_bytes_per_token(const pcd_model* m);

/* ------------------------------------------------------------------ prefill */
/* Prefills the shared prompt ids[0..n) (host) at positions 0..n-1 into a new
 * cache ("The idea", step 1; PCD: A Technical Reference, stage 1 "Broadcast
 * prefill").  Enqueued on the model stream; the cache is usable by later
 * calls at once.  Errors: INVALID_ARG (n < 1), TOKEN_RANGE, TOO_LONG, OOM, CUDA. */
int pcd_prefill(pcd_model* m, const int32_t* ids, int n, pcd_cache** out);
/* Same with ids already in device memory.  They are not checked on the host:
 * an id outside [0, vocab) is read as id 0 and the next pcd_sync reports
 * PCD_ERR_TOKEN_RANGE. */
int pcd_prefill_device(pcd_model* m, const int32_t* ids_device, int n, pcd_cache** out);

/* Warm mode: a new cache = `head` (e.g. the cached instructions and schema
 * catalogue, How TypeSafe's Jev Might Work, "The idea": "its KV state is
 * computed once and cached") followed by ids[0..n) at positions
 * head_len .. head_len+n-1.  `head` is not modified. */
int pcd_prefill_extend(pcd_model* m, const pcd_cache* head, const int32_t* ids, int n, pcd_cache** out);

int pcd_cache_length(const pcd_cache* c);
void pcd_cache_free(pcd_cache* c);

/* --------------------------------------------------------------------- score */
/* Scores every field against the prefix in one batched branch pass (stages
 * 2-5 of PCD: A Technical Reference, section 4, with the multi-token stage
 * done as exact scoring through the candidate trie) and writes out[f] for
 * each field.  Synchronises the model stream.  stats may be NULL.
 * Errors: the validation codes above, SHAPE_MISMATCH, TOO_LONG, OOM, CUDA,
 * DEVICE_TIMEOUT. */
int pcd_score(pcd_model* m, const pcd_cache* cache, const pcd_field* fields, int n_fields, pcd_field_result* out,
              pcd_stats* stats);

/* Batched serving: requests r = 0..n_requests-1, each with its own cache and
 * fields, scored in one branch pass (the weights are streamed once for all). */
int pcd_score_batch(pcd_model* m, const pcd_cache* const* caches, const pcd_field* const* fields, const int* n_fields,
                    int n_requests, pcd_field_result* const* out, pcd_stats* stats);

/* Compiles fields once into a device-resident plan (the per-schema
 * compilation the stephanj README's CompiledSchema does once).  The plan does
 * not depend on the prefix length. */
int pcd_plan_create(pcd_model* m, const pcd_field* fields, int n_fields, pcd_plan** out);
void pcd_plan_free(pcd_plan* p);
/* Floats of the device result blob of a plan: n_fields * 8 (label, mass,
 * log_mass, margin, first_mass, labels of the field, 0, 0), then probs[total labels],
 * then logprobs[total labels], labels in field order. */
int pcd_plan_result_floats(const pcd_plan* p);
/* Scores a compiled plan against a cache; results go to a device buffer of
 * pcd_plan_result_floats(p) floats.  Only enqueues (no synchronisation). */
int pcd_score_plan_device(pcd_model* m, const pcd_cache* cache, const pcd_plan* p, float* result_device);

/* Single-pass request (the stephanj README's single-pass mode): the prefix
 * ids[0..n) and every field's branch rows run in ONE forward pass -- each
 * layer writes the prefix keys/values and the branch rows attend to them in
 * the same layer -- so the weights stream once per request instead of twice.
 * The results equal pcd_prefill + pcd_score's (same arithmetic, rows
 * batched differently).  `cache_out` (nullable) receives the prefix cache for
 * later pcd_score / pcd_prefill_extend calls.  Synchronises the model
 * stream. */
int pcd_prefill_score(pcd_model* m, const int32_t* ids, int n, const pcd_field* fields, int n_fields,
                      pcd_field_result* out, pcd_stats* stats, pcd_cache** cache_out);
/* Same with device-resident ids and a compiled plan; only enqueues. */
int pcd_prefill_score_plan_device(pcd_model* m, const int32_t* ids_device, int n, const pcd_plan* plan,
                                  float* result_device, pcd_cache** cache_out);

/* First field first (How TypeSafe's Jev Might Work, "The first key of a JSON
 * object is a special position": every row of the batched pass otherwise
 * asks its field as if it were the object's first key).  Scores fields[0]
 * alone against `cache`; its answer line -- fields[0].scaffold, the first
 * listed path of its winning label, then sep[0..n_sep) (the tokens that
 * close the value, e.g. quote, comma, newline) -- then stands between the
 * prefix and every other field, and fields[1..n_fields) are scored after it
 * in one batched branch pass.  out[f] is written for every field.
 * With cache_out == NULL the line runs as branch tokens ahead of the other
 * fields inside that pass (two passes in all).  With cache_out the line is
 * written after a copy of the prefix by an extension pass first (three
 * passes) and *cache_out receives that extended prefix, owned by the caller
 * (NULL is stored with a single field, where no line is written).  `cache`
 * is not modified.  stats (may be NULL) adds up the passes of this call:
 * forward_passes counted, branch_tokens and readout_rows summed, prefill_ms
 * the extension pass, total_ms the call.  All fields are validated before
 * the first pass.  Synchronises the model stream after the first decision
 * (the line depends on it).  Errors: as pcd_score and pcd_prefill_extend;
 * sep tokens out of range are PCD_ERR_TOKEN_RANGE, n_sep < 0 or sep NULL
 * with n_sep > 0 INVALID_ARG. */
int pcd_score_first_field_first(pcd_model* m, const pcd_cache* cache, const pcd_field* fields, int n_fields,
                                const int32_t* sep, int n_sep, pcd_field_result* out, pcd_stats* stats,
                                pcd_cache** cache_out);
/* The same from the prefix ids: one pass runs the prefix with fields[0]'s
 * rows (as pcd_prefill_score), the second runs the answer line and the
 * other fields as branch tokens on that prefix -- the four sequential passes
 * of a warm request (prefill, first field, line, the rest) in two.
 * cache_out (may be NULL) receives the prefix's cache (without the line). */
int pcd_prefill_score_first_field_first(pcd_model* m, const int32_t* ids, int n, const pcd_field* fields,
                                        int n_fields, const int32_t* sep, int n_sep, pcd_field_result* out,
                                        pcd_stats* stats, pcd_cache** cache_out);

/* Waits for the model stream; reports a device-side failure recorded since
 * the last pcd_sync (PCD_ERR_DEVICE_TIMEOUT, PCD_ERR_TOKEN_RANGE). */
int pcd_sync(pcd_model* m);

/* ---------------------------------------------------------- instrumentation */
/* Per-kernel-class timing: when enabled, every launch is bracketed by CUDA
 * events on the model stream.  A pass still runs as a CUDA graph (a separate
 * graph that holds the event records), and the call that replays it
 * synchronises the stream and adds up its events before returning, so
 * profiled calls are synchronous; the event records between launches cost
 * the overlap of one launch's start with the previous one's tail.  Classes: 0 prefill GEMMs, 1 branch GEMMs, 2 prefill attention,
 * 3 branch attention, 4 fused readout, 5 other, 6 single-pass GEMMs other
 * than the gate/up projection, 7 the single-pass gate/up projection (with
 * its SwiGLU epilogue).  pcd_profile_read synchronises, returns per class the
 * launch count and the summed milliseconds, and resets the counters. */
#define PCD_PROF_CLASSES 8
int pcd_profile_enable(pcd_model* m, int on);
int pcd_profile_read(pcd_model* m, int* launches, float* ms);

const char* pcd_strerror(int code);
const char* pcd_last_error(void);

/* The byte layout of the ABI structs as this library was compiled, for a
 * binding to check its own copy of the declarations: for pcd_model_config,
 * pcd_field, pcd_field_result and pcd_stats in that order, the struct's size
 * and then the offset of each member in declaration order.  Writes at most n
 * values to out (out may be NULL with n = 0) and returns how many the full
 * layout has.  Host only. */
int pcd_abi_layout(int32_t* out, int n);

#ifdef __cplusplus
}
#endif
#endif
