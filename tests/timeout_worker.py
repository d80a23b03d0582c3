"""Child process of test_device_wait_timeout.

With PCD_WAIT_LIMIT_MS set far below a copy's latency (read once, when a
model is loaded), the pipeline waits of a prefill at the Qwen2.5-1.5B shape
give up (a GEMM's epilogue waits for a whole K loop of 24 to 140 blocks,
longer than one hardware try-wait window; the tiny decoder's one-block loops
finish inside it): the kernels record an error word, drain the copies and
MMAs they already issued and return, so pcd_sync reports
PCD_ERR_DEVICE_TIMEOUT.  The same process then loads the tiny decoder under
the default limit and scores its request correctly, which shows the CUDA
context survived.  Prints one line per step; exits 0 only if every step went
as stated.
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import synth  # noqa: E402


def main():
    import constrained_decoding_gb300.pcd as pcd
    from oracle import Oracle
    import torch
    assert float(os.environ["PCD_WAIT_LIMIT_MS"]) < 1e-3
    big = synth.make_weights(synth.model_config("1.5b"), seed=0)
    m = pcd.pcd_load_weights_host(big)
    del big
    prefix = np.arange(64, dtype=np.int32) * 37 % 151936
    codes = []
    for _ in range(3):
        ids = torch.tensor(prefix, dtype=torch.int32, device="cuda")
        c = pcd.pcd_prefill_device(m, ids)       # enqueued, not synchronised
        try:
            pcd.pcd_sync(m)
            codes.append(0)
        except pcd.PCDError as e:
            codes.append(e.code)
        c.free()
    print("timeout codes", codes, flush=True)
    m.free()
    assert -11 in codes, codes
    assert all(c in (0, -11) for c in codes), codes

    del os.environ["PCD_WAIT_LIMIT_MS"]
    w = synth.make_weights(synth.model_config("tiny"), seed=0)
    req = synth.make_request(1)
    m = pcd.pcd_load_weights_host(w)
    got = pcd.pcd_score(m, pcd.pcd_prefill(m, req.prefix), req.fields)
    pcd.pcd_sync(m)
    orc = Oracle(w, np.float32)
    oc = orc.prefill(req.prefix)
    for g, f in zip(got, req.fields):
        r = orc.score_field(f, cache=oc)
        assert np.max(np.abs(g.probs - r.probs)) <= 2e-3
    m.free()
    print("recovered ok", flush=True)


if __name__ == "__main__":
    main()
