"""The alternative scoring rules and spelling sets on the CUDA path against
the oracle: the length-normalised mean of a label's token log-probs, the
per-level product of renormalised trie decisions, and labels written several
ways (bare, quoted, another capitalisation) whose paths add up; field by
field and mixed within one call, on every execution path (two-pass, batched
requests, single pass, device-resident plan), with the deep, wide and
one-level tries of the edge workloads."""
import numpy as np
import pytest

from synth.requests import make_custom
from parity import compare_request, rescore, with_rule

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pcd():
    import constrained_decoding_gb300.pcd as pcd
    return pcd


@pytest.fixture(scope="module")
def model(pcd, tiny_weights):
    m = pcd.pcd_load_weights_host(tiny_weights)
    yield m
    m.free()


def _ref(orc, req, fields):
    cache = orc.prefill(req.prefix)
    return [rescore(orc.score_field(f, cache=cache), f) for f in fields]


@pytest.mark.parametrize("rule", ["mean", "level", ["level", "mean", "sum"]])
def test_rules_two_pass(pcd, model, tiny_oracle, request1, rule):
    fields = with_rule(request1.fields, rule)
    for f, T in zip(fields, (0.5, 1.0, 3.0, 1.0)):
        f.temperature = T
    got = pcd.pcd_score(model, pcd.pcd_prefill(model, request1.prefix), fields)
    compare_request(got, _ref(tiny_oracle, request1, fields), f"rule {rule}")


@pytest.mark.parametrize("seed,prefix_len,specs", [
    (12, 200, [("enum", 7, 1, 5), ("shared", 9, 2, 6), ("bool",)]),          # ragged multi-token
    (13, 77, [("router", 255)]),                                             # 255 labels, shared first token
    (14, 130, [("line_id", 218), ("scaffold", 13), ("enum", 3, 1, 1)]),       # deep line-ID trie
])
@pytest.mark.parametrize("rule", ["mean", "level"])
def test_rules_edge_shapes(pcd, model, tiny_oracle, seed, prefix_len, specs, rule):
    req = make_custom(seed, 512, prefix_len, specs)
    fields = with_rule(req.fields, rule)
    got = pcd.pcd_score(model, pcd.pcd_prefill(model, req.prefix), fields)
    ref = _ref(tiny_oracle, req, fields)
    compare_request(got, ref, f"seed {seed} rule {rule}")
    if rule == "level":
        # per-level probabilities are already normalised over the labels
        for g in got:
            assert abs(float(np.exp(g.logprobs.astype(np.float64)).sum()) - 1.0) < 1e-3


def test_rules_batch_and_single_pass(pcd, model, tiny_oracle):
    reqs = [make_custom(40 + i, 512, 25 + 19 * i, [("bool",), ("enum", 5, 1, 3), ("shared", 4, 2, 4)])
            for i in range(4)]
    fields = [with_rule(r.fields, ["level", "mean", "level"]) for r in reqs]
    caches = [pcd.pcd_prefill(model, r.prefix) for r in reqs]
    batch = pcd.pcd_score_batch(model, caches, fields)
    for r, fs, b in zip(reqs, fields, batch):
        ref = _ref(tiny_oracle, r, fs)
        compare_request(b, ref, "batch")
        compare_request(pcd.pcd_prefill_score(model, r.prefix, fs), ref, "single pass")


def test_rule_does_not_change_the_mass(pcd, model, request1):
    cache = pcd.pcd_prefill(model, request1.prefix)
    base = pcd.pcd_score(model, cache, request1.fields)
    for rule in ("mean", "level"):
        got = pcd.pcd_score(model, cache, with_rule(request1.fields, rule))
        for a, b in zip(base, got):
            assert abs(a.log_mass - b.log_mass) < 1e-5 and abs(a.first_mass - b.first_mass) < 1e-6


SPELLED = [("spelled", 2, 2), ("bool",), ("spelled", 3, 3), ("scaffold", 9), ("spelled", 4, 2), ("enum", 3, 1, 2)]


@pytest.mark.parametrize("rule", ["sum", "mean", "level"])
def test_spellings(pcd, model, tiny_oracle, rule):
    req = make_custom(31, 512, 90, SPELLED)
    fields = with_rule(req.fields, rule)
    ref = _ref(tiny_oracle, req, fields)
    cache = pcd.pcd_prefill(model, req.prefix)
    got = pcd.pcd_score(model, cache, fields)
    assert [len(g.probs) for g in got] == pcd.n_outputs(fields) == [2, 2, 3, 4, 3]
    compare_request(got, ref, f"spellings, rule {rule}")
    compare_request(pcd.pcd_prefill_score(model, req.prefix, fields), ref, f"spellings single pass, rule {rule}")


def test_spellings_batch_and_device_plan(pcd, model, tiny_oracle):
    import torch
    reqs = [make_custom(50 + i, 512, 40 + 23 * i, SPELLED) for i in range(3)]
    fields = [with_rule(r.fields, ["sum", "level", "mean"]) for r in reqs]
    caches = [pcd.pcd_prefill(model, r.prefix) for r in reqs]
    refs = [_ref(tiny_oracle, r, fs) for r, fs in zip(reqs, fields)]
    for b, ref in zip(pcd.pcd_score_batch(model, caches, fields), refs):
        compare_request(b, ref, "spellings batch")
    plan = pcd.pcd_plan_create(model, fields[0])
    assert plan.result_floats == 8 * len(fields[0]) + 2 * sum(pcd.n_outputs(fields[0]))
    out = torch.zeros(plan.result_floats, dtype=torch.float32, device="cuda")
    pcd.pcd_score_plan_device(model, caches[0], plan, out)
    pcd.pcd_sync(model)
    compare_request(pcd.unpack_plan_result(out.cpu().numpy(), pcd.n_outputs(fields[0])), refs[0],
                    "spellings device plan")


def test_one_spelling_per_label_is_unchanged(pcd, model, request1):
    """An explicit identity label map gives bit-identical results."""
    import dataclasses
    cache = pcd.pcd_prefill(model, request1.prefix)
    base = pcd.pcd_score(model, cache, request1.fields)
    ident = [dataclasses.replace(f, label_of=np.arange(len(f.labels), dtype=np.int32)) for f in request1.fields]
    for a, b in zip(base, pcd.pcd_score(model, cache, ident)):
        np.testing.assert_array_equal(a.probs, b.probs)
        np.testing.assert_array_equal(a.logprobs, b.logprobs)
        assert a.label == b.label and a.mass == b.mass


def test_schema_gives_the_same_results(pcd, model, request1):
    """A Schema packed once gives bit-identical results to the field list, on
    every path that takes fields."""
    sch = pcd.Schema(request1.fields)
    cache = pcd.pcd_prefill(model, request1.prefix)
    pairs = [(pcd.pcd_score(model, cache, request1.fields), pcd.pcd_score(model, cache, sch)),
             (pcd.pcd_prefill_score(model, request1.prefix, request1.fields),
              pcd.pcd_prefill_score(model, request1.prefix, sch)),
             (pcd.pcd_score_batch(model, [cache, cache], [request1.fields, request1.fields])[1],
              pcd.pcd_score_batch(model, [cache, cache], [sch, sch])[1]),
             (pcd.pcd_prefill_score_first_field_first(model, request1.prefix, request1.fields, [3]),
              pcd.pcd_prefill_score_first_field_first(model, request1.prefix, sch, [3]))]
    for a, b in pairs:
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x.probs, y.probs)
            np.testing.assert_array_equal(x.logprobs, y.logprobs)
            assert x.label == y.label and x.mass == y.mass and x.first_mass == y.first_mass
