"""CUDA path vs the oracle on the tiny decoder (2 layers, d=64, V=512), through
the C ABI: the reference workload, ragged and degenerate shapes, warm
prefixes, batched requests, the device-resident plan path, and the first-
token tie that trie scoring resolves."""
import numpy as np
import pytest

import synth
from synth.requests import make_custom
from parity import compare_request, compare_field

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


def _oracle_results(orc, req):
    cache = orc.prefill(req.prefix)
    return [orc.score_field(f, cache=cache) for f in req.fields]


def test_reference_workload(pcd, model, tiny_oracle, request1):
    cache = pcd.pcd_prefill(model, request1.prefix)
    got, stats = pcd.pcd_score(model, cache, request1.fields, with_stats=True)
    ref = _oracle_results(tiny_oracle, request1)
    worst = compare_request(got, ref, "tiny")
    assert stats["forward_passes"] == 1
    # 4 fields x 6 scaffold tokens + internal trie nodes
    n_internal = sum(len(l) - 1 for l in request1.fields[2].labels) + \
        1 + sum(len(l) - 2 for l in request1.fields[3].labels)
    assert stats["branch_tokens"] == 24 + n_internal
    print("worst errors", worst)


def test_first_token_tie_resolved_by_trie(pcd, model, tiny_oracle, request1):
    """The shared-first-token enum: trie scores differ, so the label is the
    model's choice, not the lowest index a first-token gather would return."""
    cache = pcd.pcd_prefill(model, request1.prefix)
    got = pcd.pcd_score(model, cache, request1.fields)[3]
    assert len(np.unique(np.round(got.logprobs, 4))) == len(request1.fields[3].labels)
    ref = _oracle_results(tiny_oracle, request1)[3]
    compare_field(got, ref)


@pytest.mark.parametrize("seed,prefix_len,specs", [
    (11, 1, [("scaffold", 1), ("bool",)]),                                  # minimal everything
    (12, 200, [("enum", 7, 1, 5), ("shared", 9, 2, 6), ("bool",)]),         # ragged multi-token
    (13, 77, [("router", 255)]),                                            # max candidates
    (14, 130, [("line_id", 218), ("scaffold", 13), ("enum", 3, 1, 1)]),      # line-ID trie, long scaffold
    (15, 64, [("scaffold", 3)] + [("bool",)] * 40),                          # many fields
])
def test_edge_shapes(pcd, model, tiny_oracle, seed, prefix_len, specs):
    req = make_custom(seed, 512, prefix_len, specs)
    cache = pcd.pcd_prefill(model, req.prefix)
    got = pcd.pcd_score(model, cache, req.fields)
    compare_request(got, _oracle_results(tiny_oracle, req), f"seed {seed}")


def test_temperature(pcd, model, tiny_oracle, request1):
    import copy
    fields = copy.deepcopy(request1.fields)
    for f, T in zip(fields, (0.5, 2.0, 7.0, 1.0)):
        f.temperature = T
    cache = pcd.pcd_prefill(model, request1.prefix)
    got = pcd.pcd_score(model, cache, fields)
    oc = tiny_oracle.prefill(request1.prefix)
    ref = [tiny_oracle.score_field(f, cache=oc) for f in fields]
    compare_request(got, ref, "temperature")


def test_warm_extend_equals_cold(pcd, model, request1):
    P = request1.prefix
    cold = pcd.pcd_score(model, pcd.pcd_prefill(model, P), request1.fields)
    head = pcd.pcd_prefill(model, P[:40])
    warm_cache = pcd.pcd_prefill_extend(model, head, P[40:])
    assert warm_cache.length == len(P) and head.length == 40
    warm = pcd.pcd_score(model, warm_cache, request1.fields)
    for a, b in zip(cold, warm):
        np.testing.assert_allclose(a.logprobs, b.logprobs, atol=2e-3)
        np.testing.assert_allclose(a.probs, b.probs, atol=2e-4)


def test_batch_equals_single(pcd, model, tiny_oracle):
    reqs = [make_custom(20 + i, 512, 30 + 17 * i, [("bool",), ("enum", 4, 1, 3), ("shared", 3, 2, 3)])
            for i in range(5)]
    caches = [pcd.pcd_prefill(model, r.prefix) for r in reqs]
    batch = pcd.pcd_score_batch(model, caches, [r.fields for r in reqs])
    for r, c, b in zip(reqs, caches, batch):
        single = pcd.pcd_score(model, c, r.fields)
        # a single request runs one tree-attention launch, a batch of several
        # requests the split attention + merge launches: the key blocks, and
        # so the fp16 rounding of the softmax weights, differ
        for x, y in zip(single, b):
            np.testing.assert_allclose(x.logprobs, y.logprobs, atol=2e-3)
        compare_request(b, _oracle_results(tiny_oracle, r), "batch")


def test_plan_device_path(pcd, model, request1):
    import torch
    plan = pcd.pcd_plan_create(model, request1.fields)
    ids = torch.tensor(request1.prefix, dtype=torch.int32, device="cuda")
    cache = pcd.pcd_prefill_device(model, ids)
    out = torch.zeros(plan.result_floats, dtype=torch.float32, device="cuda")
    pcd.pcd_score_plan_device(model, cache, plan, out)
    pcd.pcd_sync(model)
    got = pcd.unpack_plan_result(out.cpu().numpy(), [len(f.labels) for f in request1.fields])
    host = pcd.pcd_score(model, pcd.pcd_prefill(model, request1.prefix), request1.fields)
    for a, b in zip(got, host):
        assert a.label == b.label
        np.testing.assert_allclose(a.logprobs, b.logprobs, atol=1e-5)


def test_validation_errors(pcd, model, request1):
    cache = pcd.pcd_prefill(model, request1.prefix)
    F = synth.Field
    bad = {
        -3: [F(np.array([1]), [np.array([5])])],                               # one candidate
        -4: [F(np.array([1]), [np.array([5]), np.array([], np.int32)])],        # empty label
        -5: [F(np.array([1]), [np.array([5, 6]), np.array([5, 6])])],           # duplicate
        -6: [F(np.array([1]), [np.array([5]), np.array([5, 6])])],              # prefix label
        -7: [F(np.array([1]), [np.array([5]), np.array([512])])],               # token range
        -1: [F(np.array([], np.int32), [np.array([5]), np.array([6])])],        # empty scaffold
        -2: [F(np.array([1]), [np.array([i]) for i in range(256)])],            # 256 candidates
    }
    for code, fields in bad.items():
        with pytest.raises(pcd.PCDError) as ei:
            pcd.pcd_score(model, cache, fields)
        assert ei.value.code == code
    with pytest.raises(pcd.PCDError) as ei:
        pcd.pcd_prefill(model, np.array([0, 1, 600]))
    assert ei.value.code == -7
    # a valid call still works afterwards
    pcd.pcd_score(model, cache, request1.fields)


def test_kv_bytes(pcd, model, tiny_weights):
    c = tiny_weights.cfg
    assert pcd.pcd_kv_bytes_per_token(model) == c.n_layers * 2 * c.n_kv_heads * c.head_dim * 2


@pytest.mark.parametrize("prefix_len", [300, 700, 1500])
def test_long_prefix_split_attention(pcd, model, tiny_oracle, prefix_len):
    """Prefixes long enough that the prefill attention cuts its keys into
    several ranges (and the branch pass does too) still match the oracle."""
    req = make_custom(40 + prefix_len, 512, prefix_len, [("bool",), ("enum", 4, 1, 3), ("shared", 5, 2, 3)])
    cache = pcd.pcd_prefill(model, req.prefix)
    got = pcd.pcd_score(model, cache, req.fields)
    compare_request(got, _oracle_results(tiny_oracle, req), f"prefix {prefix_len}")


@pytest.mark.parametrize("seed,prefix_len,specs", [
    (1, None, None),                                                         # the reference workload
    (12, 200, [("enum", 7, 1, 5), ("shared", 9, 2, 6), ("bool",)]),
    (13, 77, [("router", 255)]),
    (16, 700, [("bool",), ("line_id", 30), ("scaffold", 2), ("enum", 4, 1, 4)]),   # split prefix attention
    (17, 1, [("scaffold", 1), ("bool",)]),
])
def test_single_pass_matches_oracle(pcd, model, tiny_oracle, request1, seed, prefix_len, specs):
    """Prefix and branches in one forward pass (README single-pass mode)."""
    req = request1 if specs is None else make_custom(seed, 512, prefix_len, specs)
    got, cache = pcd.pcd_prefill_score(model, req.prefix, req.fields, keep_cache=True)
    compare_request(got, _oracle_results(tiny_oracle, req), f"single pass {seed}")
    # the prefix cache it leaves behind is the prefill's
    again = pcd.pcd_score(model, cache, req.fields)
    for a, b in zip(got, again):
        assert a.label == b.label
        np.testing.assert_allclose(a.logprobs, b.logprobs, atol=2e-3)

