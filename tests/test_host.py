"""Host-side checks that need no GPU: the C ABI library loads and exports every
symbol include/*.h declares, the branch compiler's packed batch is a correct
trie of every field's labels, validation codes, and the replica path of the
benchmark on two gloo ranks."""
import os
import re
import subprocess
import sys

import numpy as np
import pytest

import synth
from synth.requests import make_custom

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from constrained_decoding_gb300.build import build
    build()
    import constrained_decoding_gb300 as pkg
    return pkg.load()


def declared_symbols():
    names = set()
    for h in ("pcd.h", "pcd_kernels.h"):
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(pcd_\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert {"pcd_load_weights", "pcd_prefill", "pcd_score", "pcd_prefill_extend", "pcd_score_batch"} <= names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    from constrained_decoding_gb300._decls import SIGNATURES
    assert {s[0] for s in SIGNATURES} == names


def _check_plan(plan, fields):
    T, R = plan["T"], plan["R"]
    # sizes
    internal = []
    for f in fields:
        prefixes = {tuple(l[:j]) for l in f.labels for j in range(1, len(l))}
        internal.append(len(prefixes))
    assert T == sum(len(f.scaffold) + n for f, n in zip(fields, internal))
    assert R == sum(1 + n for n in internal)
    assert plan["NL"] == sum(len(f.labels) for f in fields)
    tok, rel, ao, ai = plan["tok"], plan["rel"], plan["anc_off"], plan["anc_idx"]
    # ancestors: positions 0..rel of the token's own row, ending with itself
    for t in range(T):
        anc = ai[ao[t]:ao[t + 1]]
        assert anc[-1] == t
        np.testing.assert_array_equal(rel[anc], np.arange(rel[t] + 1))
    # every label's path spells its tokens; step j is read at the node of its first j tokens
    lab = 0
    for fi, f in enumerate(fields):
        S = len(f.scaffold)
        root = plan["fld_root"][fi]
        rt = plan["ro_tok"][root]
        assert tok[rt] == f.scaffold[-1] and rel[rt] == S - 1
        for l in f.labels:
            steps = plan["path"][plan["lab_off"][lab]:plan["lab_off"][lab + 1]]
            np.testing.assert_array_equal(plan["ch_tok"][steps], l)
            for j, e in enumerate(steps):
                row = plan["child_row"][e]
                b = plan["ro_tok"][row]
                if j == 0:
                    assert row == root
                else:
                    assert tok[b] == l[j - 1] and rel[b] == S + j - 1
                    # the node's ancestors spell the scaffold then the label prefix
                    anc = ai[ao[b]:ao[b + 1]]
                    np.testing.assert_array_equal(tok[anc], np.concatenate([f.scaffold, l[:j]]))
            lab += 1
    # the children of a readout row are distinct tokens
    rc = plan["row_ch"]
    for r in range(R):
        ch = plan["ch_tok"][rc[r]:rc[r + 1]]
        assert len(np.unique(ch)) == len(ch) >= 1


@pytest.mark.parametrize("which", [1, 2, 3, 4])
def test_branch_compiler_workloads(lib, which):
    import constrained_decoding_gb300.pcd as pcd
    req = synth.make_request(which)
    V = synth.model_config(synth.CONFIG_MODEL[which]).vocab
    plan = pcd.pcd_plan_inspect(req.fields, V)
    _check_plan(plan, req.fields)
    if which == 3:
        # one shared first token: the root has one child, 255 leaves below 2nd-level nodes
        assert plan["row_ch"][1] - plan["row_ch"][0] == 1


def test_branch_compiler_random_shapes(lib):
    import constrained_decoding_gb300.pcd as pcd
    for seed in range(20):
        rng = np.random.default_rng(seed)
        specs = []
        for _ in range(int(rng.integers(1, 6))):
            specs.append(("scaffold", int(rng.integers(1, 12))))
            k = rng.integers(0, 3)
            specs.append([("bool",), ("enum", int(rng.integers(2, 9)), 1, 5), ("shared", int(rng.integers(2, 9)), 2, 6)][k])
        req = make_custom(seed, 512, 10, specs)
        _check_plan(pcd.pcd_plan_inspect(req.fields, 512), req.fields)


def test_branch_compiler_validation(lib):
    import constrained_decoding_gb300.pcd as pcd
    F = synth.Field
    cases = {
        -3: [F(np.array([1]), [np.array([5])])],
        -4: [F(np.array([1]), [np.array([5]), np.array([], np.int32)])],
        -5: [F(np.array([1]), [np.array([5, 6]), np.array([5, 6])])],
        -6: [F(np.array([1]), [np.array([5]), np.array([5, 6])])],
        -7: [F(np.array([1]), [np.array([5]), np.array([512])])],
        -1: [F(np.array([], np.int32), [np.array([5]), np.array([6])])],
        -2: [F(np.array([1]), [np.array([i]) for i in range(256)])],
    }
    for code, fields in cases.items():
        with pytest.raises(pcd.PCDError) as ei:
            pcd.pcd_plan_inspect(fields, 512)
        assert ei.value.code == code
    bad_T = F(np.array([1]), [np.array([5]), np.array([6])], temperature=-1.0)
    with pytest.raises(pcd.PCDError):
        pcd.pcd_plan_inspect([bad_T], 512)
    # scoring rules: the three known ones compile to the same plan, others are rejected
    for rule in ("sum", "mean", "level", 0, 1, 2):
        ok = F(np.array([1]), [np.array([5, 7]), np.array([6])], scoring=rule)
        assert pcd.pcd_plan_inspect([ok], 512)["NL"] == 2
    for rule in (3, -1):
        with pytest.raises(pcd.PCDError) as ei:
            pcd.pcd_plan_inspect([F(np.array([1]), [np.array([5]), np.array([6])], scoring=rule)], 512)
        assert ei.value.code == -1
    with pytest.raises(ValueError):
        pcd.pcd_plan_inspect([F(np.array([1]), [np.array([5]), np.array([6])], scoring="max")], 512)


def test_branch_compiler_context_tokens(lib):
    """Context tokens (an answer line written before the fields) come first,
    chained; every field token has them as its first ancestors and its
    position moves past them; nothing else changes."""
    import constrained_decoding_gb300.pcd as pcd
    req = make_custom(6, 512, 10, [("bool",), ("shared", 3, 2, 3), ("spelled", 2, 2)])
    ctx = np.array([9, 8, 7, 6], np.int32)
    base = pcd.pcd_plan_inspect(req.fields, 512)
    plan = pcd.pcd_plan_inspect(req.fields, 512, ctx)
    C = len(ctx)
    assert plan["T"] == base["T"] + C and plan["NP"] == base["NP"] and plan["R"] == base["R"]
    np.testing.assert_array_equal(plan["tok"][:C], ctx)
    np.testing.assert_array_equal(plan["tok"][C:], base["tok"])
    np.testing.assert_array_equal(plan["rel"][:C], np.arange(C))
    np.testing.assert_array_equal(plan["rel"][C:], base["rel"] + C)
    for t in range(plan["T"]):
        anc = plan["anc_idx"][plan["anc_off"][t]:plan["anc_off"][t + 1]]
        if t < C:
            np.testing.assert_array_equal(anc, np.arange(t + 1))
        else:
            b = t - C
            np.testing.assert_array_equal(anc, np.concatenate(
                [np.arange(C), base["anc_idx"][base["anc_off"][b]:base["anc_off"][b + 1]] + C]))
    np.testing.assert_array_equal(plan["ro_tok"], base["ro_tok"] + C)
    for k in ("row_ch", "ch_tok", "child_row", "lab_off", "path", "fld_lab", "fld_root", "cand_label", "fld_out"):
        np.testing.assert_array_equal(plan[k], base[k])
    with pytest.raises(pcd.PCDError) as ei:
        pcd.pcd_plan_inspect(req.fields, 512, [3, 512])
    assert ei.value.code == -7


def test_struct_layout_matches_the_library(lib):
    """The binding's ctypes copies of the ABI structs have the sizes and
    member offsets the compiled library reports."""
    import ctypes
    from constrained_decoding_gb300 import _decls as D
    n = lib.pcd_abi_layout(None, 0)
    got = (ctypes.c_int32 * n)()
    assert lib.pcd_abi_layout(got, n) == n
    want = []
    for S in (D.pcd_model_config, D.pcd_field, D.pcd_field_result, D.pcd_stats):
        want.append(ctypes.sizeof(S))
        want += [getattr(S, name).offset for name, _ in S._fields_]
    assert list(got) == want


def test_answer_line_matches_the_oracle(lib):
    """The line first field first writes (scaffold, the winning label's first
    listed spelling, separator) is the oracle's, for plain, shared-prefix and
    spelled fields; a label no path spells is an error."""
    import constrained_decoding_gb300.pcd as pcd
    from oracle import Oracle, scores_to_result
    req = make_custom(12, 512, 10, [("enum", 4, 1, 3), ("shared", 3, 2, 3), ("spelled", 3, 3), ("spelled", 2, 2)])
    orc = Oracle.__new__(Oracle)  # answer_line needs no weights
    sep = np.array([4, 9, 2], np.int32)
    for f in req.fields:
        n_lab = len(f.labels) if f.label_of is None else int(f.label_of.max()) + 1
        for lab in range(n_lab):
            res = scores_to_result(np.zeros(n_lab))
            res.label = lab
            np.testing.assert_array_equal(pcd.pcd_answer_line(f, lab, sep), orc.answer_line(f, res, sep))
        np.testing.assert_array_equal(pcd.pcd_answer_line(f, 0, []), orc.answer_line(f, scores_to_result([0.0, 0.0]), []))
    with pytest.raises(pcd.PCDError) as ei:
        pcd.pcd_answer_line(req.fields[2], 3, sep)
    assert ei.value.code == -1


def test_answer_line_rejects_malformed_fields(lib):
    """A caller's malformed field is an error code, never a read out of
    bounds: a NULL scaffold with a nonzero length, and candidate offsets that
    run backwards or past the last candidate."""
    import ctypes
    from constrained_decoding_gb300 import _decls as D
    toks = (ctypes.c_int32 * 4)(5, 6, 7, 8)
    scaf = (ctypes.c_int32 * 2)(1, 2)

    def field(scaffold, n_scaffold, offsets):
        offs = (ctypes.c_int32 * len(offsets))(*offsets)
        f = D.pcd_field(scaffold=scaffold, n_scaffold=n_scaffold, cand_tokens=toks, cand_offsets=offs,
                        n_cands=len(offsets) - 1)
        return f, offs

    out = (ctypes.c_int32 * 16)()
    good, k0 = field(scaf, 2, [0, 2, 4])
    assert lib.pcd_answer_line(ctypes.byref(good), 1, None, 0, out, 16) == 4
    assert list(out[:4]) == [1, 2, 7, 8]
    for f, keep in (field(None, 2, [0, 2, 4]),        # no scaffold, two tokens claimed
                    field(scaf, -1, [0, 2, 4]),       # negative scaffold length
                    field(scaf, 2, [0, 3, 2]),        # path 1 runs backwards
                    field(scaf, 2, [1, 2, 4])):       # offsets do not start at 0
        assert lib.pcd_answer_line(ctypes.byref(f), 1, None, 0, out, 16) == -1
    bad, k1 = field(scaf, 2, [0, 2, 4])
    k1[1] = 9                                         # path 0 ends past the last candidate's end
    assert lib.pcd_answer_line(ctypes.byref(bad), 0, None, 0, out, 16) == -1


def test_weight_file_errors(lib, tmp_path):
    """The .pcdw loader refuses a missing, truncated, padded, foreign or
    differently shaped file with its error code before it touches a GPU."""
    import dataclasses
    import constrained_decoding_gb300.pcd as pcd
    w = synth.make_weights(synth.model_config("tiny"), seed=0)
    good = tmp_path / "tiny.pcdw"
    synth.write_pcdw(w, str(good))
    raw = good.read_bytes()

    def code(data=None, cfg=None, path=None):
        p = path or tmp_path / "case.pcdw"
        if data is not None:
            p.write_bytes(data)
        with pytest.raises(pcd.PCDError) as ei:
            pcd.pcd_load_weights(str(p), cfg)
        return ei.value.code

    assert code(path=tmp_path / "absent.pcdw") == -12
    assert code(raw[:-4]) == -12                       # truncated
    assert code(raw + b"\0" * 8) == -12                # trailing bytes
    assert code(raw[:40]) == -12                       # shorter than the header
    assert code(b"PCDX" + raw[4:]) == -12              # wrong magic
    assert code(raw[:4] + (2).to_bytes(4, "little") + raw[8:]) == -12   # unknown version
    assert code(raw[:8] + (3).to_bytes(4, "little") + raw[12:]) == -12  # unknown dtype
    wider = dataclasses.replace(w.cfg, d_ff=w.cfg.d_ff + 8)
    assert code(raw, cfg=wider) == -8                   # config does not match the header
    untied = dataclasses.replace(w.cfg, tied_embedding=False)
    assert code(raw, cfg=untied) == -8


def test_schema_packing(lib):
    """A Schema (fields packed once into the C layout) compiles to the same
    plan as the list of fields, scoring rules and label maps included."""
    import dataclasses
    import constrained_decoding_gb300.pcd as pcd
    req = make_custom(8, 512, 10, [("spelled", 3, 3), ("bool",), ("shared", 4, 2, 3), ("enum", 5, 1, 4)])
    fields = [dataclasses.replace(f, scoring=r, temperature=t)
              for f, r, t in zip(req.fields, ("level", "sum", "mean", 2), (1.0, 0.5, 0.0, 3.0))]
    a = pcd.pcd_plan_inspect(fields, 512)
    sch = pcd.Schema(fields)
    b = pcd.pcd_plan_inspect(sch, 512)
    for k in pcd.PLAN_ARRAYS:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    np.testing.assert_array_equal(b["scoring"], [2, 0, 1, 2])
    assert len(sch) == 4 and sch.n_cands == [3, 2, 4, 5]
    np.testing.assert_allclose(sch.structs["temperature"], [1.0, 0.5, 0.0, 3.0])
    assert sch.structs["cand_label"][1] == 0 and sch.structs["cand_label"][0] != 0


def test_branch_compiler_spellings(lib):
    """Candidate paths that spell one label: the plan records each path's
    label and each field's label count; bad label maps are rejected."""
    import constrained_decoding_gb300.pcd as pcd
    F = synth.Field
    req = make_custom(5, 512, 10, [("spelled", 2, 2), ("bool",), ("spelled", 3, 3)])
    plan = pcd.pcd_plan_inspect(req.fields, 512)
    want = np.concatenate([req.fields[0].label_of, [0, 1], req.fields[2].label_of])
    np.testing.assert_array_equal(plan["cand_label"], want)
    np.testing.assert_array_equal(plan["fld_out"], [0, 2, 4, 7])
    assert plan["NO"] == 7 and plan["NL"] == 4 + 2 + 9
    np.testing.assert_array_equal(pcd.n_outputs(req.fields), [2, 2, 3])
    paths = [np.array([5]), np.array([6]), np.array([7, 8])]
    for code, label_of in ((-1, [0, 0, 2]),       # label 1 has no spelling
                           (-1, [0, 3, 1]),       # out of range
                           (-3, [0, 0, 0])):      # one label
        with pytest.raises(pcd.PCDError) as ei:
            pcd.pcd_plan_inspect([F(np.array([1]), paths, label_of=np.array(label_of))], 512)
        assert ei.value.code == code, label_of
    with pytest.raises(ValueError):
        pcd.pcd_plan_inspect([F(np.array([1]), paths, label_of=np.array([0, 1]))], 512)


def _replica_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ws, r, _ = bench.dist_info()
    dist = bench.dist_init(ws)
    bench.barrier(dist)
    mx = bench.max_over_ranks(dist, 1.0 + r)
    sm = bench.sum_over_ranks(dist, 10.0)
    out.put((r, mx, sm))
    dist.destroy_process_group()


def test_replica_timing_helpers_two_gloo_ranks():
    """The N>1 benchmark path: every rank times its own replica; rank 0 reports
    the max time over ranks and the sum of the units all ranks processed."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    ps = [ctx.Process(target=_replica_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2.0, 20.0), (1, 2.0, 20.0)]


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_result_buffers_are_per_call():
    """Result structs point into their own call's float buffer (probs, then
    logprobs, field by field), and a second call gets a fresh buffer even
    though the layout is shared."""
    from constrained_decoding_gb300 import pcd
    n = [4, 2, 3]
    r1, r2 = pcd._Results(n), pcd._Results(n)
    for r in (r1, r2):
        base = r.buf.ctypes.data
        assert r.total == 9 and r.buf.size == 18
        assert r.structs["probs"].tolist() == [base, base + 16, base + 24]
        assert r.structs["logprobs"].tolist() == [base + 36, base + 52, base + 60]
    assert r1.buf.ctypes.data != r2.buf.ctypes.data
    r1.buf[:] = np.arange(18)
    r1.structs["label"] = [3, 1, 0]
    out = r1.results()
    assert [x.label for x in out] == [3, 1, 0]
    assert out[1].probs.tolist() == [4.0, 5.0] and out[2].logprobs.tolist() == [15.0, 16.0, 17.0]
    assert r2.results()[0].probs.tolist() == [0.0] * 4
