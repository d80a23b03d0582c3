"""First-field-first scoring on the CUDA path against the oracle: field 1
decided alone, its answer line written after the prefix by one extension
pass, the other fields decided after that line ("The first key of a JSON
object is a special position", How TypeSafe's Jev Might Work).  Tiny decoder
(with spellings and scoring rules) and the 28-field triage request at the
Qwen2.5-1.5B shape."""
import time

import numpy as np
import pytest

import synth
from synth.requests import make_custom
from parity import compare_request, with_rule

pytestmark = pytest.mark.gpu

SEP = np.array([7, 11, 3], np.int32)


@pytest.fixture(scope="module")
def pcd():
    import constrained_decoding_gb300.pcd as pcd
    return pcd


@pytest.fixture(scope="module")
def model(pcd, tiny_weights):
    m = pcd.pcd_load_weights_host(tiny_weights)
    yield m
    m.free()


def test_tiny(pcd, model, tiny_oracle, request1):
    cache = pcd.pcd_prefill(model, request1.prefix)
    before = pcd.pcd_score(model, cache, request1.fields)
    oc = tiny_oracle.prefill(request1.prefix)
    ref = tiny_oracle.score_first_field_first(oc, request1.fields, SEP)
    # the answer line as branch tokens ahead of the other fields: two passes
    two, st2 = pcd.pcd_score_first_field_first(model, cache, request1.fields, SEP, with_stats=True)
    compare_request(two, ref, "first field first, line in the branch pass")
    assert st2["forward_passes"] == 2
    # from the ids: prefix with field 1, then line and the rest
    pf, st3 = pcd.pcd_prefill_score_first_field_first(model, request1.prefix, request1.fields, SEP, with_stats=True)
    compare_request(pf, ref, "first field first from the ids")
    assert st3["forward_passes"] == 2
    # the line written into an extended prefix first: three passes
    got, st, ext = pcd.pcd_score_first_field_first(model, cache, request1.fields, SEP, with_stats=True,
                                                   keep_cache=True)
    compare_request(got, ref, "first field first")
    assert st["forward_passes"] == 3
    for a, b in zip(got, two):
        np.testing.assert_allclose(a.logprobs, b.logprobs, atol=2e-3)
    line = tiny_oracle.answer_line(request1.fields[0], ref[0], SEP)
    assert ext.length == len(request1.prefix) + len(line)
    # the extended prefix is the prefix followed by the line: scoring the
    # other fields on it again gives the same numbers
    again = pcd.pcd_score(model, ext, request1.fields[1:])
    for a, b in zip(got[1:], again):
        np.testing.assert_allclose(a.logprobs, b.logprobs, atol=2e-3)
    # the caller's cache is untouched
    for a, b in zip(before, pcd.pcd_score(model, cache, request1.fields)):
        np.testing.assert_array_equal(a.logprobs, b.logprobs)


@pytest.mark.parametrize("rules", [["sum"], ["level", "mean", "sum"]])
def test_spellings_and_rules(pcd, model, tiny_oracle, rules):
    req = make_custom(61, 512, 70, [("spelled", 3, 3), ("bool",), ("shared", 4, 2, 3), ("spelled", 2, 2)])
    fields = with_rule(req.fields, rules)
    cache = pcd.pcd_prefill(model, req.prefix)
    oc = tiny_oracle.prefill(req.prefix)
    ref = tiny_oracle.score_first_field_first(oc, fields, SEP)
    # the written line follows field 1's decision, so the comparison of the
    # later fields covers it too
    compare_request(pcd.pcd_score_first_field_first(model, cache, fields, SEP), ref, f"first field first {rules}")
    compare_request(pcd.pcd_score_first_field_first(model, cache, fields, SEP, keep_cache=True)[0], ref,
                    f"first field first {rules}, extended prefix")
    compare_request(pcd.pcd_prefill_score_first_field_first(model, req.prefix, fields, SEP), ref,
                    f"first field first {rules}, from the ids")


def test_single_field_and_errors(pcd, model, request1):
    cache = pcd.pcd_prefill(model, request1.prefix)
    got, st, ext = pcd.pcd_score_first_field_first(model, cache, request1.fields[:1], SEP, with_stats=True,
                                                   keep_cache=True)
    assert st["forward_passes"] == 1 and ext is None
    np.testing.assert_array_equal(got[0].logprobs, pcd.pcd_score(model, cache, request1.fields[:1])[0].logprobs)
    with pytest.raises(pcd.PCDError) as ei:
        pcd.pcd_score_first_field_first(model, cache, request1.fields, [5, 512])
    assert ei.value.code == -7
    bad = list(request1.fields) + [synth.Field(np.array([1]), [np.array([5])])]
    with pytest.raises(pcd.PCDError) as ei:
        pcd.pcd_score_first_field_first(model, cache, bad, SEP)
    assert ei.value.code == -3
    # no separator is allowed
    pcd.pcd_score_first_field_first(model, cache, request1.fields, [])


def test_config2_triage(pcd):
    from oracle import Oracle
    cfg = synth.model_config("1.5b")
    w = synth.make_weights(cfg, seed=0)
    model = pcd.pcd_load_weights_host(w)
    try:
        req = synth.make_request(2)
        sep = np.array([1, 2], np.int32)
        cache = pcd.pcd_prefill(model, req.prefix)
        got, st = pcd.pcd_score_first_field_first(model, cache, req.fields, sep, with_stats=True)
        assert st["forward_passes"] == 2
        pf, st2 = pcd.pcd_prefill_score_first_field_first(model, req.prefix, req.fields, sep, with_stats=True)
        assert st2["forward_passes"] == 2
        ext = pcd.pcd_score_first_field_first(model, cache, req.fields, sep, keep_cache=True)[0]
        orc = Oracle(w, np.float32)
        t = time.time()
        ref = orc.score_first_field_first(orc.prefill(req.prefix), req.fields, sep)
        print(f"oracle: {time.time() - t:.1f} s")
        print("config 2 first field first worst errors", compare_request(got, ref, "config 2 first field first"))
        print("config 2 first field first from the ids",
              compare_request(pf, ref, "config 2 first field first from the ids"))
        compare_request(ext, ref, "config 2 first field first, extended prefix")
    finally:
        model.free()
