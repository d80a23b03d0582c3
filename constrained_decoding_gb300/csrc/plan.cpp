// Branch compiler (see plan.h).
#include "plan.h"

#include <cmath>
#include <map>
#include <string>
#include <vector>

namespace pcd {

namespace {
struct Node {
  int token = -1;
  int parent = -1;
  int depth = 0;
  std::map<int, int> children;  // token -> node
  bool label_end = false;
  int branch = -1;              // branch token index (internal nodes)
  int row = -1;                 // readout row (root and internal nodes)
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

  for (int f = 0; f < n_fields; ++f) {
    const pcd_field& F = fields[f];
    const std::string where = "field " + std::to_string(p->n_fields) + ": ";
    if (F.n_scaffold < 1 || !F.scaffold) {
      *msg = where + "the scaffold needs at least one token";
      return PCD_ERR_INVALID_ARG;
    }
    if (F.n_cands > 255) {
      *msg = where + std::to_string(F.n_cands) + " candidates (at most 255)";
      return PCD_ERR_TOO_MANY_CANDIDATES;
    }
    if (F.n_cands < 2) {
      *msg = where + "fewer than 2 candidates";
      return PCD_ERR_TOO_FEW_CANDIDATES;
    }
    if (!F.cand_tokens || !F.cand_offsets || F.cand_offsets[0] != 0) {
      *msg = where + "candidate arrays missing or cand_offsets[0] != 0";
      return PCD_ERR_INVALID_ARG;
    }
    if (!(F.temperature >= 0.f) || std::isinf(F.temperature)) {
      *msg = where + "temperature must be finite and >= 0";
      return PCD_ERR_INVALID_ARG;
    }
    // spellings: the label each candidate path spells
    int n_out = F.n_cands;
    if (F.cand_label) {
      n_out = F.n_labels;
      if (n_out < 2) {
        *msg = where + "fewer than 2 labels";
        return PCD_ERR_TOO_FEW_CANDIDATES;
      }
      if (n_out > F.n_cands) {
        *msg = where + "more labels than candidate paths";
        return PCD_ERR_INVALID_ARG;
      }
      std::vector<int> paths(n_out, 0);
      for (int c = 0; c < F.n_cands; ++c) {
        if (F.cand_label[c] < 0 || F.cand_label[c] >= n_out) {
          *msg = where + "cand_label out of range";
          return PCD_ERR_INVALID_ARG;
        }
        paths[F.cand_label[c]]++;
      }
      for (int l = 0; l < n_out; ++l)
        if (!paths[l]) {
          *msg = where + "label " + std::to_string(l) + " has no spelling";
          return PCD_ERR_INVALID_ARG;
        }
    }
    if (F.scoring != PCD_SCORE_SUM && F.scoring != PCD_SCORE_MEAN && F.scoring != PCD_SCORE_LEVEL) {
      *msg = where + "unknown scoring rule " + std::to_string(F.scoring);
      return PCD_ERR_INVALID_ARG;
    }
    for (int k = 0; k < F.n_scaffold; ++k)
      if (F.scaffold[k] < 0 || F.scaffold[k] >= vocab) {
        *msg = where + "scaffold token out of range";
        return PCD_ERR_TOKEN_RANGE;
      }

    // ---- trie of the label paths
    std::vector<Node> nodes(1);  // node 0: the scaffold end
    std::vector<std::vector<int>> label_nodes(F.n_cands);
    for (int c = 0; c < F.n_cands; ++c) {
      const int b = F.cand_offsets[c], e = F.cand_offsets[c + 1];
      if (e < b) {
        *msg = where + "cand_offsets not increasing";
        return PCD_ERR_INVALID_ARG;
      }
      if (e == b) {
        *msg = where + "label " + std::to_string(c) + " is empty";
        return PCD_ERR_EMPTY_LABEL;
      }
      int cur = 0;
      for (int j = b; j < e; ++j) {
        const int t = F.cand_tokens[j];
        if (t < 0 || t >= vocab) {
          *msg = where + "label token out of range";
          return PCD_ERR_TOKEN_RANGE;
        }
        auto it = nodes[cur].children.find(t);
        int nx;
        if (it == nodes[cur].children.end()) {
          nx = static_cast<int>(nodes.size());
          Node n;
          n.token = t;
          n.parent = cur;
          n.depth = nodes[cur].depth + 1;
          nodes.push_back(n);
          nodes[cur].children[t] = nx;
        } else {
          nx = it->second;
        }
        label_nodes[c].push_back(nx);
        cur = nx;
      }
      if (nodes[cur].label_end) {
        *msg = where + "label " + std::to_string(c) + " repeats an earlier label";
        return PCD_ERR_DUPLICATE_LABEL;
      }
      nodes[cur].label_end = true;
    }
    for (const Node& n : nodes)
      if (n.label_end && !n.children.empty()) {
        *msg = where + "a label is a strict prefix of another (append its terminator token)";
        return PCD_ERR_PREFIX_LABEL;
      }

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
    std::vector<int> order(1, 0);
    for (size_t i = 0; i < order.size(); ++i)
      for (auto& kv : nodes[order[i]].children) order.push_back(kv.second);
    for (int id : order) {
      if (id == 0 || nodes[id].children.empty()) continue;
      Node& n = nodes[id];
      n.branch = p->T;
      p->tok.push_back(n.token);
      const int rel = n_ctx + S + n.depth - 1;
      p->rel.push_back(rel);
      if (rel > p->max_rel) p->max_rel = rel;
      for (int a = 0; a < n_ctx; ++a) p->anc_idx.push_back(c0 + a);
      for (int a = 0; a < S; ++a) p->anc_idx.push_back(t0 + a);
      std::vector<int> chain;
      for (int x = id; x != 0; x = nodes[x].parent) chain.push_back(nodes[x].branch);
      for (auto it = chain.rbegin(); it != chain.rend(); ++it) p->anc_idx.push_back(*it);
      p->anc_off.push_back(static_cast<int32_t>(p->anc_idx.size()));
      p->T++;
    }
    if (n_ctx + S - 1 > p->max_rel) p->max_rel = n_ctx + S - 1;

    // ---- readout rows and their child entries
    std::map<std::pair<int, int>, int> entry_of;  // (node, child token) -> child entry
    p->fld_root.push_back(p->R);
    for (int id : order) {
      Node& n = nodes[id];
      if (n.children.empty()) continue;
      n.row = p->R++;
      p->ro_tok.push_back(n.branch);
      for (auto& kv : n.children) {
        entry_of[{id, kv.first}] = p->n_children++;
        p->ch_tok.push_back(kv.first);
        p->child_row.push_back(n.row);
      }
      p->row_ch.push_back(p->n_children);
    }

    // ---- label paths
    for (int c = 0; c < F.n_cands; ++c) {
      int parent = 0;
      for (int nid : label_nodes[c]) {
        p->path.push_back(entry_of.at({parent, nodes[nid].token}));
        p->n_path++;
        parent = nid;
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
