"""Tree attention variants against the oracle: every cluster size, the
tensor-core kernel (head dim 128) and the warp-MMA one, and the split
attention + merge launches, on requests whose ancestor sets span several
64-key chunks, in both the single pass and the prefill + branch passes."""
import os
import subprocess
import sys
from types import SimpleNamespace

import numpy as np
import pytest

import synth
from parity import compare_field

pytestmark = pytest.mark.gpu

VARIANTS = {
    "tiny": [{"PCD_TREE_CSK": "1"}, {"PCD_TREE_CSK": "2"}, {"PCD_TREE_CSK": "3"}, {"PCD_TREE_CSK": "8"},
             {"PCD_TREE_ATTN": "0"}],
    "tiny-h128": [{}, {"PCD_TREE_CSK": "2"}, {"PCD_TREE_CSK": "3"}, {"PCD_TREE_CSK": "5"}, {"PCD_TREE_CSK": "8"},
                  {"PCD_ATTN_TC": "0"}, {"PCD_TREE_ATTN": "0"},
                  # every remainder term of the attention (the 7B width's default), and none in P.V
                  {"PCD_ATTN_LO_TERMS": "3"}, {"PCD_ATTN_LO_TERMS": "1"}, {"PCD_ATTN_LO_TERMS": "3", "PCD_TREE_CSK": "3"}],
}
CASES = [(shape, env) for shape, envs in VARIANTS.items() for env in envs]


@pytest.fixture(scope="module")
def oracles():
    from oracle import Oracle
    return {shape: Oracle(synth.make_weights(synth.model_config(shape), seed=0), np.float32) for shape in VARIANTS}


@pytest.mark.parametrize("shape,env", CASES, ids=[f"{s}-{'-'.join(f'{k}={v}' for k, v in e.items()) or 'default'}"
                                                 for s, e in CASES])
def test_attention_variants(oracles, tmp_path, shape, env):
    import attn_variant_worker as wk
    out = tmp_path / "res.npz"
    subprocess.run([sys.executable, wk.__file__, str(out), shape], env={**os.environ, **env}, check=True,
                   timeout=600)
    got = np.load(out)
    orc = oracles[shape]
    for i, req in enumerate(wk.requests()):
        cache = orc.prefill(req.prefix)
        ref = [orc.score_field(f, cache=cache) for f in req.fields]
        for mode in ("single", "two"):
            for f, r in enumerate(ref):
                sc = got[f"{mode}_{i}_{f}_scalars"]
                g = SimpleNamespace(logprobs=got[f"{mode}_{i}_{f}_logprobs"], probs=got[f"{mode}_{i}_{f}_probs"],
                                    label=int(sc[0]), mass=float(sc[1]), log_mass=float(sc[2]),
                                    first_mass=float(sc[3]))
                compare_field(g, r, f"{shape} {env} {mode} request {i} field {f}")


def test_batch_and_extend_head_dim_128(oracles):
    """A batch of requests with different prefix lengths in one branch pass
    (each tile reads its own request's cache), and prefixes extended from a
    cached head (prefill queries at positions past the head), against the
    oracle on the head-dim-128 decoder."""
    import constrained_decoding_gb300.pcd as pcd
    from synth.requests import make_custom
    orc = oracles["tiny-h128"]
    w = synth.make_weights(synth.model_config("tiny-h128"), seed=0)
    m = pcd.pcd_load_weights_host(w)
    try:
        specs = [("bool",), ("enum", 4, 1, 3), ("shared", 5, 2, 3), ("scaffold", 70), ("enum", 3, 2, 4)]
        reqs = [make_custom(60 + i, 512, n, specs) for i, n in enumerate((40, 130, 257, 7, 333))]
        caches = [pcd.pcd_prefill(m, r.prefix) for r in reqs]
        batch = pcd.pcd_score_batch(m, caches, [r.fields for r in reqs])
        head = pcd.pcd_prefill(m, reqs[4].prefix[:100])
        ext = pcd.pcd_prefill_extend(m, head, reqs[4].prefix[100:])
        warm = pcd.pcd_score(m, ext, reqs[4].fields)
        for i, (r, got) in enumerate(zip(reqs, batch)):
            oc = orc.prefill(r.prefix)
            ref = [orc.score_field(f, cache=oc) for f in r.fields]
            for f, (g, rf) in enumerate(zip(got, ref)):
                compare_field(g, rf, f"batch request {i} field {f}")
            if i == 4:
                for f, (g, rf) in enumerate(zip(warm, ref)):
                    compare_field(g, rf, f"extended prefix field {f}")
        for c in caches + [head, ext]:
            c.free()
    finally:
        m.free()
