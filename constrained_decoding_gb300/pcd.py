"""Python binding of the PCD C ABI (include/pcd.h), same names as the C
entry points.  Argument marshalling only: numpy arrays and torch tensors are
turned into pointers, results are copied into Python objects; every step of
the hot path runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes
import functools
import weakref
from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np

from . import _decls as D
from ._lib import load


class PCDError(RuntimeError):
    def __init__(self, code: int, where: str):
        lib = load()
        msg = lib.pcd_strerror(code).decode()
        detail = lib.pcd_last_error().decode()
        super().__init__(f"{where}: {msg} ({code}): {detail}")
        self.code = code


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise PCDError(rc, where)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr_i32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        return None
    return int(getattr(stream, "cuda_stream", stream))


@dataclass(slots=True)
class FieldResult:
    probs: np.ndarray
    logprobs: np.ndarray
    label: int
    mass: float
    log_mass: float
    margin: float
    first_mass: float


# ----------------------------------------------------------------- handles
class Model:
    def __init__(self, handle: int, cfg: D.pcd_model_config):
        self.handle = handle
        self.cfg = cfg
        self._children = weakref.WeakSet()

    def free(self) -> None:
        if self.handle:
            for ch in list(self._children):
                ch.free()
            load().pcd_model_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class Cache:
    def __init__(self, model: Model, handle: int):
        self.model = model
        self.handle = handle
        model._children.add(self)

    @property
    def length(self) -> int:
        return load().pcd_cache_length(self.handle)

    def free(self) -> None:
        if self.handle:
            load().pcd_cache_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class Plan:
    def __init__(self, model: Model, handle: int):
        self.model = model
        self.handle = handle
        model._children.add(self)

    @property
    def result_floats(self) -> int:
        return load().pcd_plan_result_floats(self.handle)

    def free(self) -> None:
        if self.handle:
            load().pcd_plan_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


# ------------------------------------------------------------------ models
def model_config(cfg, max_positions: int = 0) -> D.pcd_model_config:
    """A pcd_model_config from any object with the decoder-shape attributes."""
    return D.pcd_model_config(cfg.n_layers, cfg.d_model, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.d_ff,
                              cfg.vocab, float(cfg.rms_eps), float(cfg.rope_theta), 1 if cfg.tied_embedding else 0,
                              max_positions)


def pcd_load_weights(path: str, cfg=None, stream=None, max_positions: int = 0) -> Model:
    lib = load()
    c = model_config(cfg, max_positions) if cfg is not None else None
    out = ctypes.c_void_p()
    _check(lib.pcd_load_weights(ctypes.byref(c) if c is not None else None, path.encode(),
                                _stream_handle(stream), ctypes.byref(out)), "pcd_load_weights")
    return Model(out.value, c)


def pcd_load_weights_host(weights, stream=None, max_positions: int = 0) -> Model:
    """`weights` has cfg, embed, layers[i][attn_norm, wq, wk, wv, wo, mlp_norm,
    w_gate, w_up, w_down], final_norm, lm_head (None when tied); matrices are
    float32 or bf16 bit patterns (uint16)."""
    lib = load()
    c = model_config(weights.cfg, max_positions)
    arrays = [weights.embed]
    for lw in weights.layers:
        arrays += [np.asarray(lw["attn_norm"], np.float32), lw["wq"], lw["wk"], lw["wv"], lw["wo"],
                   np.asarray(lw["mlp_norm"], np.float32), lw["w_gate"], lw["w_up"], lw["w_down"]]
    arrays.append(np.asarray(weights.final_norm, np.float32))
    if weights.lm_head is not None:
        arrays.append(weights.lm_head)
    arrays = [np.ascontiguousarray(a) for a in arrays]
    dtype = 2 if weights.embed.dtype == np.uint16 else 1
    ptrs = (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])
    out = ctypes.c_void_p()
    _check(lib.pcd_load_weights_host(ctypes.byref(c), ptrs, dtype, _stream_handle(stream), ctypes.byref(out)),
           "pcd_load_weights_host")
    return Model(out.value, c)


def pcd_model_free(model: Model) -> None:
    model.free()


def pcd_kv_bytes_per_token(model: Model) -> int:
    return int(load().pcd_kv_bytes_per_token(model.handle))


# ----------------------------------------------------------------- prefill
def pcd_prefill(model: Model, ids) -> Cache:
    ids = _i32(ids)
    out = ctypes.c_void_p()
    _check(load().pcd_prefill(model.handle, _ptr_i32(ids), len(ids), ctypes.byref(out)), "pcd_prefill")
    return Cache(model, out.value)


def pcd_prefill_device(model: Model, ids_device) -> Cache:
    """ids_device: a CUDA int32 tensor (torch) or (pointer, length)."""
    if isinstance(ids_device, tuple):
        ptr, n = ids_device
    else:
        ptr, n = ids_device.data_ptr(), ids_device.numel()
    out = ctypes.c_void_p()
    _check(load().pcd_prefill_device(model.handle, ptr, int(n), ctypes.byref(out)), "pcd_prefill_device")
    return Cache(model, out.value)


def pcd_prefill_extend(model: Model, head: Cache, ids) -> Cache:
    ids = _i32(ids)
    out = ctypes.c_void_p()
    _check(load().pcd_prefill_extend(model.handle, head.handle, _ptr_i32(ids), len(ids), ctypes.byref(out)),
           "pcd_prefill_extend")
    return Cache(model, out.value)


def pcd_cache_free(cache: Cache) -> None:
    cache.free()


# ------------------------------------------------------------------- score
SCORING = {"sum": 0, "mean": 1, "level": 2}


def scoring_code(rule) -> int:
    """PCD_SCORE_* code of a field's scoring rule, given by name ("sum",
    "mean", "level") or code; None means "sum"."""
    if rule is None:
        return 0
    if isinstance(rule, str):
        if rule not in SCORING:
            raise ValueError(f"unknown scoring rule {rule!r}")
        return SCORING[rule]
    return int(rule)


def _struct_dtype(cstruct) -> np.dtype:
    """numpy record type with the byte layout of a ctypes structure (pointers
    as uint64), so an array of structs is filled column by column."""
    names, formats, offsets = [], [], []
    for name, ct in cstruct._fields_:
        names.append(name)
        offsets.append(getattr(cstruct, name).offset)
        if ct is ctypes.c_float:
            formats.append(np.float32)
        elif ct in (ctypes.c_int, ctypes.c_int32):
            formats.append(np.int32)
        else:  # a pointer
            formats.append(np.uint64)
    return np.dtype({"names": names, "formats": formats, "offsets": offsets, "itemsize": ctypes.sizeof(cstruct)})


_FIELD_DT = _struct_dtype(D.pcd_field)
_RESULT_DT = _struct_dtype(D.pcd_field_result)


def _ints(a) -> list:
    return a.tolist() if isinstance(a, np.ndarray) else [int(x) for x in a]


class Schema:
    """A list of fields packed once into the C layout (one int32 buffer and an
    array of pcd_field), for callers that score the same schema many times:
    every call that takes `fields` also takes a Schema.  Each field needs
    `scaffold` and `labels` (token paths), and may set `temperature`,
    `scoring` ("sum", "mean", "level" or a PCD_SCORE_* code) and `label_of`
    (the label each path spells)."""

    def __init__(self, fields: Sequence):
        fields = list(fields)
        ints: list = []
        cols = {k: [] for k in ("o_sc", "n_sc", "o_tok", "o_off", "n_c", "temp", "rule", "o_lab", "n_lab")}
        self.n_cands: List[int] = []
        for f in fields:
            sc = _ints(f.scaffold)
            labels = [_ints(l) for l in f.labels]
            cols["o_sc"].append(len(ints))
            cols["n_sc"].append(len(sc))
            ints.extend(sc)
            cols["o_tok"].append(len(ints))
            for l in labels:
                ints.extend(l)
            cols["o_off"].append(len(ints))
            acc = 0
            ints.append(0)
            for l in labels:
                acc += len(l)
                ints.append(acc)
            label_of = getattr(f, "label_of", None)
            if label_of is None:
                cols["o_lab"].append(-1)
                n_out = len(labels)
            else:
                lab = _ints(label_of)
                if len(lab) != len(labels):
                    raise ValueError("label_of needs one entry per token path")
                cols["o_lab"].append(len(ints))
                ints.extend(lab)
                n_out = max(lab) + 1 if lab else 0
            cols["n_c"].append(len(labels))
            cols["temp"].append(float(getattr(f, "temperature", 1.0) or 0.0))
            cols["rule"].append(scoring_code(getattr(f, "scoring", "sum")))
            cols["n_lab"].append(n_out)
            self.n_cands.append(n_out)
        self.data = np.array(ints if ints else [0], dtype=np.int32)
        base = np.uint64(self.data.ctypes.data)
        a = np.zeros(len(fields), _FIELD_DT)
        if fields:
            four = np.uint64(4)
            a["scaffold"] = base + four * np.array(cols["o_sc"], np.uint64)
            a["n_scaffold"] = cols["n_sc"]
            a["cand_tokens"] = base + four * np.array(cols["o_tok"], np.uint64)
            a["cand_offsets"] = base + four * np.array(cols["o_off"], np.uint64)
            a["n_cands"] = cols["n_c"]
            a["temperature"] = cols["temp"]
            a["scoring"] = cols["rule"]
            o_lab = np.array(cols["o_lab"], np.int64)
            a["cand_label"] = np.where(o_lab >= 0, base + four * np.maximum(o_lab, 0).astype(np.uint64), np.uint64(0))
            a["n_labels"] = cols["n_lab"]
        self.structs = a
        self.arr = ctypes.cast(a.ctypes.data, ctypes.POINTER(D.pcd_field))

    def __len__(self) -> int:
        return len(self.n_cands)


def _Fields(fields) -> Schema:
    """The packed form of `fields` (a Schema is used as it is)."""
    return fields if isinstance(fields, Schema) else Schema(fields)


@functools.lru_cache(maxsize=256)
def _result_layout(n_cands: tuple):
    """Per field count list: the total, each field's offset into the float
    buffer, and result structs whose probs/logprobs hold byte offsets."""
    total = int(sum(n_cands))
    offs = np.concatenate([[0], np.cumsum(n_cands, dtype=np.int64)])[:-1].astype(np.uint64)
    a = np.zeros(len(n_cands), _RESULT_DT)
    four = np.uint64(4)
    a["probs"] = four * offs
    a["logprobs"] = four * (np.uint64(total) + offs)
    return total, offs.tolist(), a


class _Results:
    """Result structs and one float buffer (probs, then logprobs) for a call."""

    def __init__(self, n_cands: List[int]):
        self.n_cands = list(n_cands)
        self.total, self.offs, tmpl = _result_layout(tuple(self.n_cands))
        self.buf = np.zeros(2 * max(self.total, 1), np.float32)
        a = tmpl.copy()
        base = np.uint64(self.buf.ctypes.data)
        a["probs"] += base
        a["logprobs"] += base
        self.structs = a
        self.arr = ctypes.cast(a.ctypes.data, ctypes.POINTER(D.pcd_field_result))

    def results(self) -> List[FieldResult]:
        a = self.structs
        t = self.total
        buf = self.buf
        return [FieldResult(buf[o:o + n], buf[t + o:t + o + n], lab, m, lm, mg, fm)
                for o, n, lab, m, lm, mg, fm in zip(self.offs, self.n_cands, a["label"].tolist(),
                                                    a["mass"].tolist(), a["log_mass"].tolist(),
                                                    a["margin"].tolist(), a["first_mass"].tolist())]


def _stats_dict(s: D.pcd_stats) -> dict:
    return {k: getattr(s, k) for k, _ in D.pcd_stats._fields_}


def pcd_score(model: Model, cache: Cache, fields: Sequence, with_stats: bool = False):
    f = _Fields(fields)
    r = _Results(f.n_cands)
    st = D.pcd_stats()
    _check(load().pcd_score(model.handle, cache.handle, f.arr, len(fields), r.arr, ctypes.byref(st)), "pcd_score")
    return (r.results(), _stats_dict(st)) if with_stats else r.results()


def pcd_score_batch(model: Model, caches: Sequence[Cache], fields: Sequence[Sequence], with_stats: bool = False):
    n = len(caches)
    fs = [_Fields(fl) for fl in fields]
    rs = [_Results(x.n_cands) for x in fs]
    c_arr = (ctypes.c_void_p * n)(*[c.handle for c in caches])
    f_arr = (ctypes.POINTER(D.pcd_field) * n)(*[ctypes.cast(x.arr, ctypes.POINTER(D.pcd_field)) for x in fs])
    r_arr = (ctypes.POINTER(D.pcd_field_result) * n)(
        *[ctypes.cast(x.arr, ctypes.POINTER(D.pcd_field_result)) for x in rs])
    nf = (ctypes.c_int * n)(*[len(fl) for fl in fields])
    st = D.pcd_stats()
    _check(load().pcd_score_batch(model.handle, c_arr, f_arr, nf, n, r_arr, ctypes.byref(st)), "pcd_score_batch")
    out = [x.results() for x in rs]
    return (out, _stats_dict(st)) if with_stats else out


def pcd_prefill_score(model: Model, ids, fields: Sequence, with_stats: bool = False, keep_cache: bool = False):
    """Single-pass request: prefix + every field in one forward pass.
    Returns results (and stats, and the prefix Cache when keep_cache)."""
    ids = _i32(ids)
    f = _Fields(fields)
    r = _Results(f.n_cands)
    st = D.pcd_stats()
    cache = ctypes.c_void_p()
    _check(load().pcd_prefill_score(model.handle, _ptr_i32(ids), len(ids), f.arr, len(fields), r.arr, ctypes.byref(st),
                                    ctypes.byref(cache) if keep_cache else None), "pcd_prefill_score")
    out = [r.results()]
    if with_stats:
        out.append(_stats_dict(st))
    if keep_cache:
        out.append(Cache(model, cache.value))
    return out[0] if len(out) == 1 else tuple(out)


def pcd_score_first_field_first(model: Model, cache: Cache, fields: Sequence, sep=(), with_stats: bool = False,
                                keep_cache: bool = False):
    """Decide fields[0] alone, then the other fields after its answer line
    (scaffold, winning label's first spelling, ``sep`` tokens).  With
    keep_cache the line is first written after a copy of the prefix and that
    extended prefix Cache is returned too.  Returns results (and stats)."""
    f = _Fields(fields)
    r = _Results(f.n_cands)
    sp = _i32(sep)
    st = D.pcd_stats()
    ext = ctypes.c_void_p()
    _check(load().pcd_score_first_field_first(model.handle, cache.handle, f.arr, len(fields),
                                              _ptr_i32(sp) if len(sp) else None, len(sp), r.arr, ctypes.byref(st),
                                              ctypes.byref(ext) if keep_cache else None),
           "pcd_score_first_field_first")
    out = [r.results()]
    if with_stats:
        out.append(_stats_dict(st))
    if keep_cache:
        out.append(Cache(model, ext.value) if ext.value else None)
    return out[0] if len(out) == 1 else tuple(out)


def pcd_prefill_score_first_field_first(model: Model, ids, fields: Sequence, sep=(), with_stats: bool = False,
                                        keep_cache: bool = False):
    """First field first from the prefix ids in two passes (prefix with
    fields[0]; answer line with the other fields).  Returns results (and
    stats, and the prefix Cache when keep_cache)."""
    ids = _i32(ids)
    f = _Fields(fields)
    r = _Results(f.n_cands)
    sp = _i32(sep)
    st = D.pcd_stats()
    cache = ctypes.c_void_p()
    _check(load().pcd_prefill_score_first_field_first(model.handle, _ptr_i32(ids), len(ids), f.arr, len(fields),
                                                      _ptr_i32(sp) if len(sp) else None, len(sp), r.arr,
                                                      ctypes.byref(st), ctypes.byref(cache) if keep_cache else None),
           "pcd_prefill_score_first_field_first")
    out = [r.results()]
    if with_stats:
        out.append(_stats_dict(st))
    if keep_cache:
        out.append(Cache(model, cache.value) if cache.value else None)
    return out[0] if len(out) == 1 else tuple(out)


def pcd_prefill_score_plan_device(model: Model, ids_device, plan: Plan, result_device, keep_cache: bool = False):
    """Single-pass request from device-resident ids (CUDA int32 tensor) and a plan; only enqueues."""
    cache = ctypes.c_void_p()
    ptr = result_device if isinstance(result_device, int) else result_device.data_ptr()
    _check(load().pcd_prefill_score_plan_device(model.handle, ids_device.data_ptr(), ids_device.numel(), plan.handle,
                                                ptr, ctypes.byref(cache) if keep_cache else None),
           "pcd_prefill_score_plan_device")
    return Cache(model, cache.value) if keep_cache else None


def pcd_plan_create(model: Model, fields: Sequence) -> Plan:
    f = _Fields(fields)
    out = ctypes.c_void_p()
    _check(load().pcd_plan_create(model.handle, f.arr, len(fields), ctypes.byref(out)), "pcd_plan_create")
    return Plan(model, out.value)


def pcd_score_plan_device(model: Model, cache: Cache, plan: Plan, result_device) -> None:
    """result_device: CUDA float32 tensor of plan.result_floats elements (or a pointer)."""
    ptr = result_device if isinstance(result_device, int) else result_device.data_ptr()
    _check(load().pcd_score_plan_device(model.handle, cache.handle, plan.handle, ptr), "pcd_score_plan_device")


def n_outputs(fields: Sequence) -> List[int]:
    """Labels of each field: its token paths, or the labels they spell."""
    return [len(f.labels) if getattr(f, "label_of", None) is None else int(np.max(f.label_of)) + 1
            for f in fields]


def unpack_plan_result(blob: np.ndarray, n_cands: Sequence[int]) -> List[FieldResult]:
    """Splits a plan's result blob (layout in include/pcd.h) into per-field
    results; n_cands[f] is field f's number of labels (``n_outputs``)."""
    nf = len(n_cands)
    nl = int(sum(n_cands))
    probs, lps = blob[nf * 8:nf * 8 + nl], blob[nf * 8 + nl:nf * 8 + 2 * nl]
    out, o = [], 0
    for f, n in enumerate(n_cands):
        h = blob[f * 8:(f + 1) * 8]
        out.append(FieldResult(probs[o:o + n].copy(), lps[o:o + n].copy(), int(h[0]), float(h[1]), float(h[2]),
                               float(h[3]), float(h[4])))
        o += n
    return out


def pcd_sync(model: Model) -> None:
    _check(load().pcd_sync(model.handle), "pcd_sync")


def pcd_profile_enable(model: Model, on: bool = True) -> None:
    _check(load().pcd_profile_enable(model.handle, 1 if on else 0), "pcd_profile_enable")


PROFILE_CLASSES = ("gemm_prefill", "gemm_branch", "attn_prefill", "attn_branch", "readout", "other", "gemm_single",
                   "gemm_gate_up")


def pcd_profile_read(model: Model) -> dict:
    n = (ctypes.c_int * len(PROFILE_CLASSES))()
    ms = (ctypes.c_float * len(PROFILE_CLASSES))()
    _check(load().pcd_profile_read(model.handle, n, ms), "pcd_profile_read")
    return {k: (int(n[i]), float(ms[i])) for i, k in enumerate(PROFILE_CLASSES)}


PLAN_ARRAYS = ("tok", "rel", "anc_off", "anc_idx", "ro_tok", "row_ch", "ch_tok", "child_row", "lab_off", "path",
               "fld_lab", "fld_root", "cand_label", "fld_out", "scoring")


def pcd_answer_line(field, label: int, sep=()) -> np.ndarray:
    """Host-only: the tokens first field first writes for `field` decided as
    `label` (scaffold, the label's first listed spelling, `sep`)."""
    lib = load()
    f = _Fields([field])
    sp = _i32(sep)
    sp_ptr = _ptr_i32(sp) if len(sp) else None
    n = lib.pcd_answer_line(ctypes.cast(f.arr, ctypes.c_void_p), int(label), sp_ptr, len(sp), None, 0)
    if n < 0:
        _check(n, "pcd_answer_line")
    out = np.zeros(max(n, 1), np.int32)
    lib.pcd_answer_line(ctypes.cast(f.arr, ctypes.c_void_p), int(label), sp_ptr, len(sp), _ptr_i32(out), n)
    return out[:n]


def pcd_plan_inspect(fields: Sequence, vocab: int, ctx=()) -> dict:
    """Host-only compile of `fields` (no GPU), after the context tokens `ctx`
    if any: the packed branch batch as numpy arrays."""
    lib = load()
    f = _Fields(fields)
    cx = _i32(ctx)
    cxp = _ptr_i32(cx) if len(cx) else None
    sizes = np.zeros(8, np.int32)
    _check(lib.pcd_plan_inspect(ctypes.cast(f.arr, ctypes.c_void_p), len(fields), vocab, _ptr_i32(sizes), None,
                                cxp, len(cx)), "pcd_plan_inspect")
    T, R, C, NL, NP, NA, NF, NO = (int(x) for x in sizes)
    lens = [T, T, T + 1, NA, R, R + 1, C, C, NL + 1, NP, NF + 1, NF, NL, NF + 1, NF]
    bufs = [np.zeros(max(n, 1), np.int32) for n in lens]
    ptrs = (ctypes.POINTER(ctypes.c_int32) * len(bufs))(*[_ptr_i32(b) for b in bufs])
    _check(lib.pcd_plan_inspect(ctypes.cast(f.arr, ctypes.c_void_p), len(fields), vocab, _ptr_i32(sizes), ptrs,
                                cxp, len(cx)), "pcd_plan_inspect")
    out = {k: b[:n] for k, b, n in zip(PLAN_ARRAYS, bufs, lens)}
    out.update(T=T, R=R, C=C, NL=NL, NP=NP, NA=NA, NF=NF, NO=NO)
    return out
