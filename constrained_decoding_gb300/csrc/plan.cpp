// Branch compiler (see plan.h).
#include "plan.h"

#include <algorithm>
#include <climits>
#include <cmath>
#include <string>
#include <utility>
#include <vector>

namespace pcd {

namespace {
struct Node {
  int token = -1;
  int parent = -1;
  int depth = 0;
  bool label_end = false;
  int branch = -1;  // branch token index (internal nodes)
  int row = -1;     // readout row (root and internal nodes)
  int entry = -1;   // child entry of the edge parent -> this node
  std::vector<std::pair<int, int>> kids;  // (token, node), ascending token
};
}  // namespace

int compile_fields(const pcd_field* fields, int n_fields, int vocab, HostPlan* p, std::string* msg,
                   const int32_t* ctx, int n_ctx) {
  if (n_fields < 0 || (n_fields > 0 && !fields)) {
    *msg = "fields is NULL or n_fields < 0";
    return PCD_ERR_INVALID_ARG;
  }
  if (n_ctx < 0 || (n_ctx > 0 && !ctx)) {
    *msg = "context tokens NULL or n_ctx < 0";
    return PCD_ERR_INVALID_ARG;
  }
  for (int k = 0; k < n_ctx; ++k)
    if (ctx[k] < 0 || ctx[k] >= vocab) {
      *msg = "context token out of range";
      return PCD_ERR_TOKEN_RANGE;
    }
  if (p->anc_off.empty()) p->anc_off.push_back(0);
  if (p->row_ch.empty()) p->row_ch.push_back(0);
  if (p->lab_off.empty()) p->lab_off.push_back(0);
  if (p->fld_lab.empty()) p->fld_lab.push_back(0);
  if (p->fld_out.empty()) p->fld_out.push_back(0);

  // ---- context tokens: a chain right after the prefix, ancestors of every field
  const int c0 = p->T;
  for (int k = 0; k < n_ctx; ++k) {
    p->tok.push_back(ctx[k]);
    p->rel.push_back(k);
    for (int a = 0; a <= k; ++a) p->anc_idx.push_back(c0 + a);
    p->anc_off.push_back(static_cast<int32_t>(p->anc_idx.size()));
    p->T++;
  }
  if (n_ctx - 1 > p->max_rel) p->max_rel = n_ctx - 1;

  // reused across fields
  std::vector<Node> nodes;
  std::vector<int> lab_node, lab_start, order, chain, paths;
  for (int f = 0; f < n_fields; ++f) {
    const pcd_field& F = fields[f];
    // the message names the field only when there is an error
    auto bad = [&](int code, const std::string& text) {
      *msg = "field " + std::to_string(p->n_fields) + ": " + text;
      return code;
    };
    if (F.n_scaffold < 1 || !F.scaffold) return bad(PCD_ERR_INVALID_ARG, "the scaffold needs at least one token");
    if (F.n_cands > 255)
      return bad(PCD_ERR_TOO_MANY_CANDIDATES, std::to_string(F.n_cands) + " candidates (at most 255)");
    if (F.n_cands < 2) return bad(PCD_ERR_TOO_FEW_CANDIDATES, "fewer than 2 candidates");
    if (!F.cand_tokens || !F.cand_offsets || F.cand_offsets[0] != 0)
      return bad(PCD_ERR_INVALID_ARG, "candidate arrays missing or cand_offsets[0] != 0");
    if (!(F.temperature >= 0.f) || std::isinf(F.temperature))
      return bad(PCD_ERR_INVALID_ARG, "temperature must be finite and >= 0");
    // spellings: the label each candidate path spells
    int n_out = F.n_cands;
    if (F.cand_label) {
      n_out = F.n_labels;
      if (n_out < 2) return bad(PCD_ERR_TOO_FEW_CANDIDATES, "fewer than 2 labels");
      if (n_out > F.n_cands) return bad(PCD_ERR_INVALID_ARG, "more labels than candidate paths");
      paths.assign(n_out, 0);
      for (int c = 0; c < F.n_cands; ++c) {
        if (F.cand_label[c] < 0 || F.cand_label[c] >= n_out) return bad(PCD_ERR_INVALID_ARG, "cand_label out of range");
        paths[F.cand_label[c]]++;
      }
      for (int l = 0; l < n_out; ++l)
        if (!paths[l]) return bad(PCD_ERR_INVALID_ARG, "label " + std::to_string(l) + " has no spelling");
    }
    if (F.scoring != PCD_SCORE_SUM && F.scoring != PCD_SCORE_MEAN && F.scoring != PCD_SCORE_LEVEL)
      return bad(PCD_ERR_INVALID_ARG, "unknown scoring rule " + std::to_string(F.scoring));
    for (int k = 0; k < F.n_scaffold; ++k)
      if (F.scaffold[k] < 0 || F.scaffold[k] >= vocab) return bad(PCD_ERR_TOKEN_RANGE, "scaffold token out of range");

    // ---- trie of the label paths; node 0 is the scaffold end
    nodes.assign(1, Node());
    lab_node.clear();
    lab_start.assign(1, 0);
    for (int c = 0; c < F.n_cands; ++c) {
      const int b = F.cand_offsets[c], e = F.cand_offsets[c + 1];
      if (e < b) return bad(PCD_ERR_INVALID_ARG, "cand_offsets not increasing");
      if (e == b) return bad(PCD_ERR_EMPTY_LABEL, "label " + std::to_string(c) + " is empty");
      int cur = 0;
      for (int j = b; j < e; ++j) {
        const int t = F.cand_tokens[j];
        if (t < 0 || t >= vocab) return bad(PCD_ERR_TOKEN_RANGE, "label token out of range");
        auto& kids = nodes[cur].kids;
        const auto it = std::lower_bound(kids.begin(), kids.end(), std::make_pair(t, INT_MIN));
        int nx;
        if (it != kids.end() && it->first == t) {
          nx = it->second;
        } else {
          const auto at = it - kids.begin();
          nx = static_cast<int>(nodes.size());
          Node n;
          n.token = t;
          n.parent = cur;
          n.depth = nodes[cur].depth + 1;
          nodes.push_back(std::move(n));  // may move nodes: index, don't hold references across it
          nodes[cur].kids.insert(nodes[cur].kids.begin() + at, std::make_pair(t, nx));
        }
        lab_node.push_back(nx);
        cur = nx;
      }
      lab_start.push_back(static_cast<int>(lab_node.size()));
      if (nodes[cur].label_end)
        return bad(PCD_ERR_DUPLICATE_LABEL, "label " + std::to_string(c) + " repeats an earlier label");
      nodes[cur].label_end = true;
    }
    for (const Node& n : nodes)
      if (n.label_end && !n.kids.empty())
        return bad(PCD_ERR_PREFIX_LABEL, "a label is a strict prefix of another (append its terminator token)");

    // ---- branch tokens: the scaffold, then internal nodes in breadth-first order
    const int S = F.n_scaffold;
    const int t0 = p->T;
    for (int k = 0; k < S; ++k) {
      p->tok.push_back(F.scaffold[k]);
      p->rel.push_back(n_ctx + k);
      for (int a = 0; a < n_ctx; ++a) p->anc_idx.push_back(c0 + a);
      for (int a = 0; a <= k; ++a) p->anc_idx.push_back(t0 + a);
      p->anc_off.push_back(static_cast<int32_t>(p->anc_idx.size()));
      p->T++;
    }
    nodes[0].branch = t0 + S - 1;
    order.assign(1, 0);
    for (size_t i = 0; i < order.size(); ++i)
      for (const auto& kv : nodes[order[i]].kids) order.push_back(kv.second);
    for (int id : order) {
      if (id == 0 || nodes[id].kids.empty()) continue;
      Node& n = nodes[id];
      n.branch = p->T;
      p->tok.push_back(n.token);
      const int rel = n_ctx + S + n.depth - 1;
      p->rel.push_back(rel);
      if (rel > p->max_rel) p->max_rel = rel;
      for (int a = 0; a < n_ctx; ++a) p->anc_idx.push_back(c0 + a);
      for (int a = 0; a < S; ++a) p->anc_idx.push_back(t0 + a);
      chain.clear();
      for (int x = id; x != 0; x = nodes[x].parent) chain.push_back(nodes[x].branch);
      p->anc_idx.insert(p->anc_idx.end(), chain.rbegin(), chain.rend());
      p->anc_off.push_back(static_cast<int32_t>(p->anc_idx.size()));
      p->T++;
    }
    if (n_ctx + S - 1 > p->max_rel) p->max_rel = n_ctx + S - 1;

    // ---- readout rows and their child entries
    p->fld_root.push_back(p->R);
    for (int id : order) {
      Node& n = nodes[id];
      if (n.kids.empty()) continue;
      n.row = p->R++;
      p->ro_tok.push_back(n.branch);
      for (const auto& kv : n.kids) {
        nodes[kv.second].entry = p->n_children++;
        p->ch_tok.push_back(kv.first);
        p->child_row.push_back(n.row);
      }
      p->row_ch.push_back(p->n_children);
    }

    // ---- label paths: the child entry of every step
    for (int c = 0; c < F.n_cands; ++c) {
      for (int j = lab_start[c]; j < lab_start[c + 1]; ++j) {
        p->path.push_back(nodes[lab_node[j]].entry);
        p->n_path++;
      }
      p->lab_off.push_back(p->n_path);
      p->n_labels++;
    }
    p->fld_lab.push_back(p->n_labels);
    p->temp.push_back(F.temperature > 0.f ? F.temperature : 1.f);
    p->scoring.push_back(F.scoring);
    for (int c = 0; c < F.n_cands; ++c) p->cand_label.push_back(F.cand_label ? F.cand_label[c] : c);
    p->n_out += n_out;
    p->fld_out.push_back(p->n_out);
    p->n_fields++;
  }
  return PCD_OK;
}

int answer_line(const pcd_field& f, int label, const int32_t* sep, int n_sep, std::vector<int32_t>* line) {
  if (label < 0 || n_sep < 0 || (n_sep > 0 && !sep) || !f.cand_offsets || !f.cand_tokens) return PCD_ERR_INVALID_ARG;
  if (f.n_scaffold < 0 || (f.n_scaffold > 0 && !f.scaffold) || f.n_cands < 0) return PCD_ERR_INVALID_ARG;
  int path = -1;
  for (int c = 0; c < f.n_cands && path < 0; ++c)
    if ((f.cand_label ? f.cand_label[c] : c) == label) path = c;
  if (path < 0) return PCD_ERR_INVALID_ARG;
  // the chosen path's token range must be well formed before it is read
  if (f.cand_offsets[0] != 0 || f.cand_offsets[path] < 0 || f.cand_offsets[path] > f.cand_offsets[path + 1] ||
      f.cand_offsets[path + 1] > f.cand_offsets[f.n_cands])
    return PCD_ERR_INVALID_ARG;
  line->assign(f.scaffold, f.scaffold + f.n_scaffold);
  line->insert(line->end(), f.cand_tokens + f.cand_offsets[path], f.cand_tokens + f.cand_offsets[path + 1]);
  line->insert(line->end(), sep, sep + n_sep);
  return PCD_OK;
}

}  // namespace pcd
