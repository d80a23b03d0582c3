"""Seeded synthetic PCD requests.

A request is a prefix of token ids (the shared prompt) plus the fields of a
closed schema.  A field is a row of scaffold tokens (the key text up to the
point where the labels diverge) and its candidate labels, each a path of
token ids.  Token ids are uniform in ``[0, vocab)``.  The pages' prompts and
presets are private text; these requests copy only their shapes: 28-field
triage schemas of booleans and 4-way enums, a 255-choice router whose labels
share a first token, a long document with 218 line-ID-shaped labels, and
batched serving with prefix lengths uniform in [512, 4096].

Draw order (one ``numpy.random.default_rng(1000 + config)`` stream):
prefix ids first, then the fields in schema order; within a field the
scaffold, then the label lengths, then the label token ids.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

from .shapes import model_config, CONFIG_MODEL


@dataclass
class Field:
    scaffold: np.ndarray                 # int32 [S]
    labels: List[np.ndarray]             # one int32 token path per label
    temperature: float = 1.0
    kind: str = "enum"
    scoring: str = "sum"                 # "sum", "mean" (length-normalised) or "level" (per-level product)
    label_of: Optional[np.ndarray] = None  # label of each token path in `labels` (several spellings
                                           # of one label); None: one path per label


@dataclass
class Request:
    prefix: np.ndarray                   # int32 [Lp]
    fields: List[Field] = field(default_factory=list)
    head_len: int = 0                    # shared schema-head length (warm serving)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _bool_field(rng, V, S) -> Field:
    scaffold = rng.integers(0, V, S)
    ids = rng.choice(V, 2, replace=False)
    return Field(_i32(scaffold), [_i32([ids[0]]), _i32([ids[1]])], kind="bool")


def _enum_field(rng, V, S, n_labels=4, lo=1, hi=4) -> Field:
    """Labels of lo..hi tokens; all ids of the field distinct (no sharing)."""
    scaffold = rng.integers(0, V, S)
    lens = rng.integers(lo, hi + 1, n_labels)
    ids = rng.choice(V, int(lens.sum()), replace=False)
    labels, o = [], 0
    for n in lens:
        labels.append(_i32(ids[o:o + n]))
        o += n
    return Field(_i32(scaffold), labels, kind="enum")


def _shared_first_field(rng, V, S, n_labels=4, lo=2, hi=3) -> Field:
    """Labels of lo..hi tokens that all share their first token id."""
    scaffold = rng.integers(0, V, S)
    lens = rng.integers(lo, hi + 1, n_labels)
    ids = rng.choice(V, 1 + int((lens - 1).sum()), replace=False)
    first, rest = ids[0], ids[1:]
    labels, o = [], 0
    for n in lens:
        labels.append(_i32([first, *rest[o:o + n - 1]]))
        o += n - 1
    return Field(_i32(scaffold), labels, kind="enum_shared")


def _router_field(rng, V, S, n_labels=255) -> Field:
    """n_labels 3-token labels: one shared first id, distinct (2nd, 3rd) pairs."""
    scaffold = rng.integers(0, V, S)
    first = int(rng.integers(0, V))
    pairs, seen = [], set()
    while len(pairs) < n_labels:
        p = (int(rng.integers(0, V)), int(rng.integers(0, V)))
        if p not in seen:
            seen.add(p)
            pairs.append(p)
    return Field(_i32(scaffold), [_i32([first, a, b]) for a, b in pairs], kind="router")


def _line_id_field(rng, V, S, n_labels=218) -> Field:
    """Line-ID labels L000..: (shared id, tens-group id, digit id)."""
    scaffold = rng.integers(0, V, S)
    n_groups = (n_labels + 9) // 10
    ids = rng.choice(V, 1 + n_groups + 10, replace=False)
    shared, groups, digits = ids[0], ids[1:1 + n_groups], ids[1 + n_groups:]
    labels = [_i32([shared, groups[i // 10], digits[i % 10]]) for i in range(n_labels)]
    return Field(_i32(scaffold), labels, kind="line_id")


def _spelled_field(rng, V, S, n_labels=2, n_spell=2) -> Field:
    """Labels with several spellings: label i is written bare (its own ids,
    1-2 tokens), quoted (a quote id, the same ids, the quote id again) and,
    with n_spell = 3, as one more id of its own (another capitalisation)."""
    scaffold = rng.integers(0, V, S)
    lens = rng.integers(1, 3, n_labels)
    ids = rng.choice(V, 1 + int(lens.sum()) + n_labels, replace=False)
    quote, o = ids[0], 1
    paths, label_of = [], []
    for i, n in enumerate(lens):
        base = list(ids[o:o + n])
        o += n
        spellings = [base, [quote, *base, quote]]
        if n_spell >= 3:
            spellings.append([ids[1 + int(lens.sum()) + i]])
        for sp in spellings:
            paths.append(_i32(sp))
            label_of.append(i)
    return Field(_i32(scaffold), paths, kind="spelled", label_of=_i32(label_of))


def _triage_schema(rng, V, S=8) -> List[Field]:
    """28 fields: 10 booleans and 18 four-way enums of 1-4 token labels."""
    kinds = np.array(["bool"] * 10 + ["enum"] * 18)
    kinds = kinds[rng.permutation(len(kinds))]
    return [_bool_field(rng, V, S) if k == "bool" else _enum_field(rng, V, S) for k in kinds]


def make_request(config: int, seed: Optional[int] = None) -> Request:
    """The request of workload ``config`` (1..4); see ``make_requests`` for 5."""
    V = model_config(CONFIG_MODEL[config]).vocab
    rng = np.random.default_rng(1000 + config if seed is None else seed)
    if config == 1:
        prefix = rng.integers(0, V, 64)
        S = 6
        fields = [_bool_field(rng, V, S), _bool_field(rng, V, S),
                  _enum_field(rng, V, S, 4, 1, 3), _shared_first_field(rng, V, S, 4, 2, 3)]
    elif config == 2:
        prefix = rng.integers(0, V, 512)
        fields = _triage_schema(rng, V)
    elif config == 3:
        prefix = rng.integers(0, V, 1024)
        fields = [_router_field(rng, V, 8)] + [_bool_field(rng, V, 8) for _ in range(3)]
    elif config == 4:
        prefix = rng.integers(0, V, 8192)
        fields = _triage_schema(rng, V) + [_line_id_field(rng, V, 8)]
    else:
        raise ValueError(f"no single-request workload {config}")
    return Request(_i32(prefix), fields)


def make_requests(config: int = 5, n_requests: int = 64, head_len: int = 512,
                  lo: int = 512, hi: int = 4096, seed: Optional[int] = None) -> List[Request]:
    """Batched serving: one triage schema shared by every request; each prefix
    is a shared schema head of ``head_len`` ids plus a request-specific tail,
    total length uniform in [lo, hi]."""
    V = model_config(CONFIG_MODEL[config]).vocab
    rng = np.random.default_rng(1000 + config if seed is None else seed)
    fields = _triage_schema(rng, V)
    head = rng.integers(0, V, head_len)
    out = []
    for _ in range(n_requests):
        n = int(rng.integers(lo, hi + 1))
        tail = rng.integers(0, V, n - head_len)
        out.append(Request(_i32(np.concatenate([head, tail])), fields, head_len))
    return out


def make_custom(seed: int, vocab: int, prefix_len: int, specs, scaffold_len: int = 6) -> Request:
    """A request with an explicit list of field shapes, for edge-case tests.

    ``specs`` items: ("bool",), ("enum", n_labels, lo, hi), ("shared", n_labels,
    lo, hi), ("router", n_labels), ("line_id", n_labels) or ("spelled", n_labels,
    n_spell); an optional
    ("scaffold", S) item before a field sets that field's scaffold length.
    """
    rng = np.random.default_rng(seed)
    prefix = rng.integers(0, vocab, prefix_len)
    fields, S = [], scaffold_len
    for sp in specs:
        kind = sp[0]
        if kind == "scaffold":
            S = sp[1]
            continue
        if kind == "bool":
            fields.append(_bool_field(rng, vocab, S))
        elif kind == "enum":
            fields.append(_enum_field(rng, vocab, S, *sp[1:]))
        elif kind == "shared":
            fields.append(_shared_first_field(rng, vocab, S, *sp[1:]))
        elif kind == "router":
            fields.append(_router_field(rng, vocab, S, *sp[1:]))
        elif kind == "line_id":
            fields.append(_line_id_field(rng, vocab, S, *sp[1:]))
        elif kind == "spelled":
            fields.append(_spelled_field(rng, vocab, S, *sp[1:]))
        else:
            raise ValueError(kind)
    return Request(_i32(prefix), fields)
