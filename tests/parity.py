"""Shared parity check of the CUDA path against the oracle.

Tolerances of the PCD hot path (bf16 weights and activations, fp32
accumulation, against the fp32 oracle):
  * label: bit-exact wherever the oracle's top-2 log-prob margin > 0.05
    (a closer call may flip under bf16, as batch-shape drift does);
  * probabilities within 2e-3 absolute;
  * label log-probs (summed), log mass within 3e-2 absolute;
  * first-decision mass within 2e-3 absolute (a probability).

The library's precision policy makes these bounds hold at every workload
shape: at the Qwen2.5-7B width every fp16 operand carries its rounding
remainder (the random 28-layer decoder amplifies a 2^-11 perturbation about a
hundredfold there).
"""
import numpy as np

PROB_TOL = 2e-3
LOGP_TOL = 3e-2
MARGIN_EXACT = 0.05


def compare_field(gpu, ref, where="", prob_tol=PROB_TOL):
    """gpu: constrained_decoding_gb300.pcd.FieldResult; ref: oracle FieldResult."""
    n = len(ref.scores)
    assert len(gpu.probs) == n, where
    errs = {
        "probs": float(np.max(np.abs(gpu.probs - ref.probs))),
        "logprobs": float(np.max(np.abs(gpu.logprobs - ref.scores))),
        "log_mass": abs(gpu.log_mass - ref.log_mass),
        "first_mass": abs(gpu.first_mass - ref.first_mass),
    }
    assert errs["probs"] <= prob_tol, (where, errs)
    assert errs["logprobs"] <= LOGP_TOL, (where, errs)
    assert errs["log_mass"] <= LOGP_TOL, (where, errs)
    assert errs["first_mass"] <= PROB_TOL, (where, errs)
    assert abs(gpu.mass - ref.mass) <= max(PROB_TOL, 3e-2 * ref.mass), (where, gpu.mass, ref.mass)
    if ref.margin > MARGIN_EXACT:
        assert gpu.label == ref.label, (where, gpu.label, ref.label, ref.margin)
    else:
        # a near tie: the GPU's label must be one of the near-best
        assert ref.scores[gpu.label] >= ref.scores.max() - MARGIN_EXACT - LOGP_TOL, where
    assert abs(float(np.sum(gpu.probs)) - 1.0) < 1e-4, where
    return errs


def compare_request(gpu_results, ref_results, where="", prob_tol=PROB_TOL):
    worst = {}
    for i, (g, r) in enumerate(zip(gpu_results, ref_results)):
        e = compare_field(g, r, f"{where} field {i}", prob_tol)
        for k, v in e.items():
            worst[k] = max(worst.get(k, 0.0), v)
    return worst


def with_rule(fields, rule):
    """Copies of `fields` scored under `rule` ("sum", "mean", "level"); a list
    of rules is applied field by field, cycling."""
    import dataclasses
    rules = [rule] if isinstance(rule, str) else list(rule)
    return [dataclasses.replace(f, scoring=rules[i % len(rules)]) for i, f in enumerate(fields)]


def rescore(ref, field):
    """The oracle's result for `field` under its scoring rule, from an oracle
    result `ref` of the same labels (its token log-probs; the decoder does
    not run again)."""
    from oracle import combine_spellings, field_scores, scores_to_result
    rule = getattr(field, "scoring", "sum") or "sum"
    scores = field_scores(rule, field.labels, ref.token_logprobs)
    if getattr(field, "label_of", None) is not None:
        scores = combine_spellings(scores, field.label_of)
    out = scores_to_result(scores, field.temperature)
    out.mass, out.log_mass, out.first_mass = ref.mass, ref.log_mass, ref.first_mass
    out.token_logprobs = ref.token_logprobs
    return out
