"""Child process of test_attention_variants: runs the CUDA path on a small
decoder (argv: output .npz, shape name) under the attention settings its
environment selects (tree attention on the tensor cores or on warp MMA, a
forced cluster size, or the split attention + merge launches) and saves
every field's results.  The settings are read once per process, hence a
process per variant."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import synth  # noqa: E402
from synth.requests import make_custom  # noqa: E402

# (seed, prefix length, field specs): a 70-token scaffold makes a tile whose
# ancestor union spans two 64-key chunks; the others mix tries and shapes
VARIANT_REQUESTS = [
    (50, 100, [("scaffold", 70), ("enum", 5, 2, 4), ("bool",)]),
    (51, 300, [("line_id", 60), ("shared", 9, 2, 6), ("scaffold", 1), ("bool",)]),
    (52, 1, [("scaffold", 2), ("router", 40)]),
    (53, 130, [("bool",)] * 30),
]


def requests():
    return [synth.make_request(1)] + [make_custom(s, 512, n, sp) for s, n, sp in VARIANT_REQUESTS]


def main(out_path, shape="tiny"):
    import constrained_decoding_gb300.pcd as pcd
    w = synth.make_weights(synth.model_config(shape), seed=0)
    m = pcd.pcd_load_weights_host(w)
    arrays = {}
    for i, req in enumerate(requests()):
        single = pcd.pcd_prefill_score(m, req.prefix, req.fields)
        two = pcd.pcd_score(m, pcd.pcd_prefill(m, req.prefix), req.fields)
        for mode, res in (("single", single), ("two", two)):
            for f, r in enumerate(res):
                arrays[f"{mode}_{i}_{f}_logprobs"] = r.logprobs
                arrays[f"{mode}_{i}_{f}_probs"] = r.probs
                arrays[f"{mode}_{i}_{f}_scalars"] = np.array([r.label, r.mass, r.log_mass, r.first_mass])
    m.free()
    np.savez(out_path, **arrays)


if __name__ == "__main__":
    main(*sys.argv[1:])
