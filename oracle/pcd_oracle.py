"""Plain CPU oracle for parallel constrained decoding (PCD).

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg may import this module; the library's compute path never
does, and nothing here is shared with the CUDA path.  It is slow on purpose:
every step is written out as its definition, with numpy matmuls as the only
library primitive.

What it computes
----------------
A decoder language model M reads a prefix P (the shared prompt).  A field of
a closed schema has a scaffold s (the key text up to where its labels
diverge) and candidate labels l_c = (t_c1 .. t_cn).  The score of a label is
the sum of the full-vocabulary log-probabilities of its tokens under teacher
forcing,

    s_c = sum_j log softmax_V( M(P || s || t_c,<j)_last )[t_cj]

("When one token is not enough", How TypeSafe's Jev Might Work: add up how
likely the model finds each of the label's tokens; "Multi-token candidates",
PCD From First Principles: teacher-force the candidate's known tokens and sum
their log-probabilities).  The field's answer is

    p_c = exp(s_c / T) / sum_c' exp(s_c' / T),    label = argmax_c p_c,
    mass = sum_c exp(s_c)

(section 4 "The algorithm" and "Notes on the softmax", PCD: A Technical
Reference: candidate-only softmax with temperature T; ties go to the first
candidate in declaration order, the rule that reference's FAQ suggests;
"And you get confidence for free", How TypeSafe's Jev Might Work: the
candidate mass is the unrenormalised probability of the allowed labels).

For single-token labels s_c = z_c - lse(z), so p_c is exactly the softmax of
the gathered candidate logits: the full-vocabulary normaliser cancels ("The
subset softmax is exact", PCD From First Principles).

Readings where the pages are silent (each also listed in the design notes):
* decoder: pre-norm RMSNorm, q/k/v/o without bias, rotate-half RoPE with
  angles pos * theta^(-2i/dh) taken in fp64 and cos/sin rounded to the
  working dtype, GQA (query head h reads KV head h // (Hq/Hkv)), scale
  1/sqrt(dh), SwiGLU MLP, final RMSNorm, logits = E h (tied) or W_lm h;
* multi-token mass is the sequence-level sum_c P(l_c);
* T divides the summed log-probs; mass ignores T; T <= 0 means 1;
* under the alternative scorings (length-normalised mean, per-level
  product) T divides that score instead, and the label, probabilities and
  margin follow it, while mass, log-mass and first-token mass keep their
  full-vocabulary definitions;
* a label with several spellings (token paths) scores each path by the
  field's rule and takes the log-sum-exp of those path scores (for the
  summed rule: the probability of writing any of its spellings); the mass
  counts every allowed path;
* the label's last token is a leaf: a label that is a strict prefix of
  another is not a valid schema (the caller appends its terminator token).

Precision: the transformer runs in ``dtype`` (fp32 by default, fp64 for the
tight pins); the vocabulary log-sum-exp and all scoring run in fp64.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np


# ---------------------------------------------------------------------------
# Decoder building blocks
# ---------------------------------------------------------------------------
def rms_norm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """y = x / sqrt(mean(x^2) + eps) * gain, over the last axis."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + x.dtype.type(eps)) * gain.astype(x.dtype)


def rope_cos_sin(positions: np.ndarray, head_dim: int, theta: float, dtype=np.float32):
    """cos/sin of the rotary angles pos * theta^(-2i/dh), i < dh/2, taken in
    fp64 and rounded to ``dtype``.  Returns two [n, dh/2] arrays."""
    half = head_dim // 2
    inv_freq = np.power(np.float64(theta), -2.0 * np.arange(half, dtype=np.float64) / head_dim)
    ang = positions.astype(np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang).astype(dtype), np.sin(ang).astype(dtype)


def apply_rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE on x [n, H, dh]: the pair (i, i + dh/2) of every head
    is rotated by the angle of position ``positions[n]`` and frequency i."""
    n, H, dh = x.shape
    half = dh // 2
    cos, sin = rope_cos_sin(positions, dh, theta, x.dtype)
    cos, sin = cos[:, None, :], sin[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
              q_pos: np.ndarray, k_pos: np.ndarray) -> np.ndarray:
    """Causal grouped-query attention.

    q [n, Hq, dh], k/v [m, Hkv, dh]; a query at position p sees the keys
    whose position is <= p (the causal mask that makes a prefix's keys and
    values final, "The piece of plumbing you need: the KV cache", How
    TypeSafe's Jev Might Work).  Query head h reads KV head h // (Hq/Hkv).
    Returns [n, Hq, dh].
    """
    n, Hq, dh = q.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    scale = q.dtype.type(1.0 / np.sqrt(dh))
    masked = k_pos[None, :] > q_pos[:, None]
    out = np.empty_like(q)
    for h in range(Hq):
        kh = h // group
        s = (q[:, h, :] @ k[:, kh, :].T) * scale
        s = np.where(masked, -np.inf, s)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, kh, :]
    return out


def silu(x: np.ndarray) -> np.ndarray:
    return x / (x.dtype.type(1) + np.exp(-x))


def swiglu(h: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """down( silu(gate h) * (up h) )."""
    return (silu(h @ w_gate.T) * (h @ w_up.T)) @ w_down.T


def logsumexp64(z: np.ndarray) -> np.ndarray:
    """Row-wise log-sum-exp in fp64, max-shifted."""
    z = z.astype(np.float64)
    m = z.max(axis=-1, keepdims=True)
    return (m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True)))[..., 0]


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    """Bytes of K and V one token leaves in the cache: layers x 2 x KV heads x
    head dim x element size ("The piece of plumbing you need: the KV cache",
    How TypeSafe's Jev Might Work, which sizes a 1,154-token prompt this way)."""
    return n_layers * 2 * n_kv_heads * head_dim * elem_bytes


# ---------------------------------------------------------------------------
# Scoring
# ---------------------------------------------------------------------------
@dataclass
class FieldResult:
    scores: np.ndarray            # s_c, fp64 summed log-probs per label
    probs: np.ndarray             # p_c
    label: int
    mass: float                   # sum_c exp(s_c)
    log_mass: float
    margin: float                 # s_top1 - s_top2 (inf with one label)
    first_mass: float = float("nan")   # P(next token starts an allowed label)
    token_logprobs: List[np.ndarray] = field(default_factory=list)


def scores_to_result(scores: Sequence[float], temperature: float = 1.0) -> FieldResult:
    """Candidate-only softmax of the label scores at temperature T, argmax
    (first candidate on ties) and candidate mass (section 4 "The algorithm" and
    "Notes on the softmax", PCD: A Technical Reference; "And you get
    confidence for free", How TypeSafe's Jev Might Work)."""
    s = np.asarray(scores, dtype=np.float64)
    T = float(temperature) if temperature and temperature > 0 else 1.0
    a = s / T
    e = np.exp(a - a.max())
    p = e / e.sum()
    label = int(np.argmax(p))
    lm = float(np.max(s) + np.log(np.exp(s - np.max(s)).sum()))
    srt = np.sort(s)[::-1]
    margin = float(srt[0] - srt[1]) if len(s) > 1 else float("inf")
    return FieldResult(s, p, label, float(np.exp(lm)), lm, margin)


def length_normalised_scores(token_logprobs: Sequence[np.ndarray]) -> np.ndarray:
    """Alternative label score: the MEAN of the label's token log-probs,
    s_c = (sum_j lp_cj) / n_c, so that a label is not marked down merely for
    having more tokens to get right (PCD From First Principles, "Multi-token
    candidates": teacher-force, then sum or length-normalise; beam search's
    reason for dividing by the length)."""
    return np.array([float(np.sum(np.asarray(lp, np.float64))) / len(lp) for lp in token_logprobs])


def per_level_scores(labels: Sequence[Sequence[int]], token_logprobs: Sequence[np.ndarray]) -> np.ndarray:
    """Alternative label score: resolve shared prefixes one level at a time.
    At every node of the label trie the decision is the distribution over the
    node's allowed next tokens alone (renormalised), and a label's probability
    is the product of those per-level probabilities along its path ("Resolve
    shared prefixes level by level" and "Multi-level fields", PCD: A Technical
    Reference).  Returns log of that product per label.

    The full-vocabulary normaliser of a node cancels in the renormalisation,
    so the per-level log-probability of token t at the node reached by the
    prefix u is  lp(t | u) - log sum_{t' allowed after u} exp(lp(t' | u)),
    with lp the full-vocabulary token log-probs of the teacher-forced labels
    (a label passing through u carries lp(next token | u) at that step).
    A node with one allowed continuation contributes probability 1."""
    labs = [tuple(int(t) for t in l) for l in labels]
    lps = [np.asarray(lp, np.float64) for lp in token_logprobs]
    out = np.zeros(len(labs))
    for c, lab in enumerate(labs):
        for j in range(len(lab)):
            prefix = lab[:j]
            allowed = {}
            for d, other in enumerate(labs):
                if len(other) > j and other[:j] == prefix:
                    allowed.setdefault(other[j], lps[d][j])
            v = np.array(list(allowed.values()))
            m = v.max()
            out[c] += lps[c][j] - (m + np.log(np.exp(v - m).sum()))
    return out


SCORINGS = ("sum", "mean", "level")


def field_scores(scoring: str, labels, token_logprobs) -> np.ndarray:
    """The label scores a field's scoring rule asks for: "sum" (the summed
    log-probs s_c), "mean" (length-normalised) or "level" (per-level
    product)."""
    if scoring == "sum":
        return np.array([float(np.sum(np.asarray(lp, np.float64))) for lp in token_logprobs])
    if scoring == "mean":
        return length_normalised_scores(token_logprobs)
    if scoring == "level":
        return per_level_scores(labels, token_logprobs)
    raise ValueError(scoring)


def combine_spellings(path_scores: Sequence[float], label_of_path: Sequence[int]) -> np.ndarray:
    """A label with several spellings (token paths) gets the probability of
    all of them: s_label = log sum_paths exp(s_path) ("Small models quote
    their booleans", How TypeSafe's Jev Might Work)."""
    s = np.asarray(path_scores, dtype=np.float64)
    lab = np.asarray(label_of_path)
    out = np.empty(int(lab.max()) + 1)
    for c in range(len(out)):
        v = s[lab == c]
        m = v.max()
        out[c] = m + np.log(np.exp(v - m).sum())
    return out


def first_token_result(z_row: np.ndarray, labels: Sequence[np.ndarray], temperature: float = 1.0):
    """First-token-only scoring (the shortcut "Where the two real
    implementations disagree", PCD From First Principles, shows failing):
    softmax of the readout row's logits at each label's FIRST token.  Labels
    sharing a first token get the same logit and tie.  Also returns P1's
    candidate mass at the readout: the probability that the next token
    starts any allowed label (each distinct first token counted once)."""
    z64 = z_row.astype(np.float64)
    lse = logsumexp64(z64[None, :])[0]
    firsts = np.array([int(l[0]) for l in labels])
    res = scores_to_result(z64[firsts], temperature)
    first_mass = float(np.exp(z64[np.unique(firsts)] - lse).sum())
    return res, first_mass


# ---------------------------------------------------------------------------
# The decoder
# ---------------------------------------------------------------------------
@dataclass
class KVCache:
    """Per-layer keys/values [m, Hkv, dh] (after RoPE) and their positions."""
    k: List[np.ndarray]
    v: List[np.ndarray]
    pos: np.ndarray

    @property
    def length(self) -> int:
        return int(self.pos.shape[0])


def _to_float(a: np.ndarray, dtype) -> np.ndarray:
    if a.dtype == np.uint16:       # bf16 bit patterns -> exact fp32
        a = (a.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """fp32 (or fp64) CPU decoder plus the PCD scorer.

    ``weights`` has the fields of ``synth.Weights`` (embed, layers with wq,
    wk, wv, wo, w_gate, w_up, w_down, attn_norm, mlp_norm, final_norm,
    lm_head) and a ``cfg`` with the decoder's shape.
    """

    def __init__(self, weights, dtype=np.float32):
        self.cfg = weights.cfg
        self.dtype = np.dtype(dtype)
        self.embed = _to_float(weights.embed, dtype)
        self.layers = []
        for lw in weights.layers:
            self.layers.append({k: _to_float(v, dtype) for k, v in lw.items()})
        self.final_norm = _to_float(weights.final_norm, dtype)
        self.lm_head = self.embed if weights.lm_head is None else _to_float(weights.lm_head, dtype)

    # -- the forward pass ---------------------------------------------------
    def forward(self, ids: np.ndarray, positions: np.ndarray,
                cache: Optional[KVCache] = None, need_hidden: bool = True):
        """Run tokens ``ids`` at ``positions`` on top of ``cache`` (keys of
        earlier positions).  Returns (final-normed hidden [n, d] or None,
        this chunk's per-layer (k, v))."""
        c = self.cfg
        n = len(ids)
        Hq, Hkv, dh = c.n_q_heads, c.n_kv_heads, c.head_dim
        positions = np.asarray(positions, dtype=np.int64)
        x = self.embed[np.asarray(ids, dtype=np.int64)].copy()
        new_k, new_v = [], []
        for li, lw in enumerate(self.layers):
            h = rms_norm(x, lw["attn_norm"], c.rms_eps)
            q = (h @ lw["wq"].T).reshape(n, Hq, dh)
            k = (h @ lw["wk"].T).reshape(n, Hkv, dh)
            v = (h @ lw["wv"].T).reshape(n, Hkv, dh)
            q = apply_rope(q, positions, c.rope_theta)
            k = apply_rope(k, positions, c.rope_theta)
            new_k.append(k)
            new_v.append(v)
            if cache is not None:
                K = np.concatenate([cache.k[li], k], axis=0)
                V = np.concatenate([cache.v[li], v], axis=0)
                kp = np.concatenate([cache.pos, positions])
            else:
                K, V, kp = k, v, positions
            o = attention(q, K, V, positions, kp).reshape(n, Hq * dh)
            x = x + o @ lw["wo"].T
            h = rms_norm(x, lw["mlp_norm"], c.rms_eps)
            x = x + swiglu(h, lw["w_gate"], lw["w_up"], lw["w_down"])
        hid = rms_norm(x, self.final_norm, c.rms_eps) if need_hidden else None
        return hid, (new_k, new_v)

    def logits(self, hidden: np.ndarray) -> np.ndarray:
        """z = W_lm h (W_lm = E when the embedding is tied)."""
        return hidden @ self.lm_head.T

    # -- the prefix snapshot ------------------------------------------------
    def prefill(self, ids: np.ndarray) -> KVCache:
        """Prefill the shared prompt once; its keys/values are final because
        of the causal mask ("The idea: parallel constrained decoding", How
        TypeSafe's Jev Might Work, step 1)."""
        ids = np.asarray(ids)
        pos = np.arange(len(ids), dtype=np.int64)
        _, (k, v) = self.forward(ids, pos, None, need_hidden=False)
        return KVCache(k, v, pos)

    def extend(self, cache: KVCache, ids: np.ndarray) -> KVCache:
        """Append tokens to a cached prefix (a warm schema head plus a request)."""
        ids = np.asarray(ids)
        pos = cache.length + np.arange(len(ids), dtype=np.int64)
        _, (k, v) = self.forward(ids, pos, cache, need_hidden=False)
        return KVCache([np.concatenate([a, b]) for a, b in zip(cache.k, k)],
                       [np.concatenate([a, b]) for a, b in zip(cache.v, v)],
                       np.concatenate([cache.pos, pos]))

    # -- teacher-forced label log-probs -------------------------------------
    def _path_logprobs(self, hid_rows: np.ndarray, label: np.ndarray):
        z = self.logits(hid_rows)
        lse = logsumexp64(z)
        zt = z[np.arange(len(label)), label].astype(np.float64)
        return zt - lse, z

    def label_logprobs(self, cache: KVCache, scaffold: np.ndarray, label: np.ndarray) -> np.ndarray:
        """Incremental mode: the row scaffold || label[:-1] runs on top of the
        prefix cache; the row's position S-1+j predicts label token j
        ("Multi-token candidates", PCD From First Principles)."""
        S = len(scaffold)
        seq = np.concatenate([scaffold, label[:-1]])
        pos = cache.length + np.arange(len(seq), dtype=np.int64)
        hid, _ = self.forward(seq, pos, cache)
        lp, _ = self._path_logprobs(hid[S - 1:S - 1 + len(label)], label)
        return lp

    def label_logprobs_independent(self, prefix: np.ndarray, scaffold: np.ndarray,
                                   label: np.ndarray) -> np.ndarray:
        """Independent mode: prefix || scaffold || label[:-1] as one fresh
        sequence, no cache (what the model would see writing the line itself)."""
        S, Lp = len(scaffold), len(prefix)
        seq = np.concatenate([prefix, scaffold, label[:-1]])
        pos = np.arange(len(seq), dtype=np.int64)
        hid, _ = self.forward(seq, pos, None)
        lp, _ = self._path_logprobs(hid[Lp + S - 1:Lp + S - 1 + len(label)], label)
        return lp

    def readout_logits(self, cache: KVCache, scaffold: np.ndarray) -> np.ndarray:
        """Full-vocabulary logits at the scaffold's last token."""
        pos = cache.length + np.arange(len(scaffold), dtype=np.int64)
        hid, _ = self.forward(scaffold, pos, cache)
        return self.logits(hid[-1:])[0]

    # -- fields -------------------------------------------------------------
    def score_field(self, field, cache: Optional[KVCache] = None,
                    prefix: Optional[np.ndarray] = None, mode: str = "incremental") -> FieldResult:
        """Score every label of ``field`` (scaffold, labels, temperature)."""
        lps = []
        for lab in field.labels:
            lab = np.asarray(lab, dtype=np.int64)
            if mode == "incremental":
                lps.append(self.label_logprobs(cache, np.asarray(field.scaffold), lab))
            elif mode == "independent":
                lps.append(self.label_logprobs_independent(np.asarray(prefix), np.asarray(field.scaffold), lab))
            else:
                raise ValueError(mode)
        # the scoring rule decides label, probabilities and margin; the mass
        # stays the full-vocabulary probability of the allowed labels.  With
        # several spellings per label (``field.label_of``) every token path
        # is scored by the rule and a label gets the log-sum-exp of its
        # paths' scores.
        scoring = getattr(field, "scoring", "sum") or "sum"
        label_of = getattr(field, "label_of", None)
        sums = field_scores("sum", field.labels, lps)
        scores = field_scores(scoring, field.labels, lps)
        if label_of is not None:
            scores = combine_spellings(scores, label_of)
        res = scores_to_result(scores, getattr(field, "temperature", 1.0))
        if scoring != "sum" or label_of is not None:
            m = sums.max()
            res.log_mass = float(m + np.log(np.exp(sums - m).sum()))
            res.mass = float(np.exp(res.log_mass))
        res.token_logprobs = lps
        # candidate mass at the first decision: first-token probabilities of
        # the distinct first tokens; the first log-prob of every label is
        # log P(first token), so no extra forward pass is needed.
        firsts = {}
        for lab, lp in zip(field.labels, lps):
            firsts.setdefault(int(lab[0]), float(lp[0]))
        res.first_mass = float(np.exp(np.array(list(firsts.values()))).sum())
        return res

    def score(self, cache: KVCache, fields) -> List[FieldResult]:
        return [self.score_field(f, cache=cache) for f in fields]

    def answer_line(self, field, res: FieldResult, sep) -> np.ndarray:
        """The tokens that write a decided field into the prompt: its
        scaffold, the first listed spelling of the winning label, then the
        separator tokens (e.g. the closing quote, comma and newline)."""
        label_of = getattr(field, "label_of", None)
        if label_of is None:
            path = field.labels[res.label]
        else:
            path = field.labels[int(np.flatnonzero(np.asarray(label_of) == res.label)[0])]
        return np.concatenate([np.asarray(field.scaffold), np.asarray(path),
                               np.asarray(sep, dtype=np.int64)]).astype(np.int64)

    def score_first_field_first(self, cache: KVCache, fields, sep) -> List[FieldResult]:
        """Decide the schema's first field on its own, write its answer into
        the prompt, then decide every other field after that line ("The
        first key of a JSON object is a special position", How TypeSafe's
        Jev Might Work: asked as the first key of the object, later fields
        sit where the model rarely is; a warm request then costs four
        passes)."""
        first = self.score_field(fields[0], cache=cache)
        if len(fields) == 1:
            return [first]
        line = self.answer_line(fields[0], first, sep)
        cache2 = self.extend(cache, line)
        return [first] + [self.score_field(f, cache=cache2) for f in fields[1:]]
