"""Child process of test_device_wait_timeout.

With PCD_WAIT_LIMIT_MS set far below a copy's latency (read once, when a
model is loaded), the GEMM pipeline waits of the tiny decoder give up: the
kernels record an error word, drain the copies and MMAs they already issued
and return, so pcd_sync reports PCD_ERR_DEVICE_TIMEOUT.  The same process then
loads the model again under the default limit and scores the request
correctly, which shows the CUDA context survived.  Prints one line per step;
exits 0 only if every step went as stated.
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import synth  # noqa: E402


def main():
    import constrained_decoding_gb300.pcd as pcd
    from oracle import Oracle
    w = synth.make_weights(synth.model_config("tiny"), seed=0)
    req = synth.make_request(1)
    assert float(os.environ["PCD_WAIT_LIMIT_MS"]) < 1e-3
    m = pcd.pcd_load_weights_host(w)
    codes = []
    for _ in range(3):
        import torch
        ids = torch.tensor(req.prefix, dtype=torch.int32, device="cuda")
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
