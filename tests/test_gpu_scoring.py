"""The alternative scoring rules on the CUDA path against the oracle: the
length-normalised mean of a label's token log-probs and the per-level product
of renormalised trie decisions, field by field and mixed within one call, on
every execution path (two-pass, batched requests, single pass), with the
deep, wide and one-level tries of the edge workloads."""
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
