// Branch compiler: a closed schema's fields -> one packed branch batch.
//
// Each field contributes its scaffold tokens and the internal nodes of the
// trie of its label token paths (a label's last token is only predicted,
// never fed).  Readout rows are the scaffold's last token and every internal
// trie node; each readout row's children are the candidate next tokens.  A
// label's score is the sum, along its path, of (logit - log-sum-exp) at the
// readout rows ("When one token is not enough", How TypeSafe's Jev Might
// Work: follow shared prefixes and multiply the per-token probabilities).
#pragma once
#include <cstdint>
#include <string>
#include <vector>

#include "pcd.h"

namespace pcd {

struct HostPlan {
  int n_fields = 0, T = 0, R = 0, n_children = 0, n_labels = 0, n_path = 0;
  int max_rel = 0;                 // largest relative position
  std::vector<int32_t> tok;        // [T] token id of each branch token
  std::vector<int32_t> rel;        // [T] position after the prefix end: C + k for scaffold token k,
                                   //     C + S + depth - 1 for a trie node at depth >= 1, with C
                                   //     context tokens before the fields (k for context token k)
  std::vector<int32_t> anc_off;    // [T + 1] ancestors of each token (same field, itself included)
  std::vector<int32_t> anc_idx;
  std::vector<int32_t> ro_tok;     // [R] branch token whose output is read
  std::vector<int32_t> row_ch;     // [R + 1] child entries of each readout row
  std::vector<int32_t> ch_tok;     // [n_children] candidate token id of each child entry
  std::vector<int32_t> child_row;  // [n_children] its readout row
  std::vector<int32_t> lab_off;    // [n_labels + 1] path steps of each candidate path
                                   // (n_labels counts candidate paths, n_out the labels they spell)
  std::vector<int32_t> path;       // [n_path] child entry of each step
  std::vector<int32_t> fld_lab;    // [n_fields + 1] labels of each field
  std::vector<int32_t> fld_root;   // [n_fields] readout row of the field's scaffold end
  std::vector<float> temp;         // [n_fields]
  std::vector<int32_t> scoring;    // [n_fields] PCD_SCORE_* rule
  int n_out = 0;                   // labels (outputs) of all fields
  std::vector<int32_t> cand_label; // [n_labels] label (within its field) each candidate path spells
  std::vector<int32_t> fld_out;    // [n_fields + 1] outputs of each field
  std::vector<int32_t> seg_off;    // [requests + 1] branch tokens of each request (empty: one request)
};

// Appends `fields` to `p` (so several requests can share one batch).  With
// n_ctx > 0 the context tokens ctx[0..n_ctx) come first: branch tokens right
// after the prefix (each an ancestor of the ones after it, no readout), and
// every field's scaffold follows them (an answer line written before the
// fields: first field first).  On error returns a PCD_ERR_* code and sets
// *msg; `p` is then unspecified.
int compile_fields(const pcd_field* fields, int n_fields, int vocab, HostPlan* p, std::string* msg,
                   const int32_t* ctx = nullptr, int n_ctx = 0);

// The tokens that write a decided field into the prompt (first field first):
// its scaffold, the first listed path that spells `label`, then sep.  Returns
// PCD_ERR_INVALID_ARG when no path spells the label.
int answer_line(const pcd_field& f, int label, const int32_t* sep, int n_sep, std::vector<int32_t>* line);

}  // namespace pcd
