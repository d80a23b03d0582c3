"""Failure paths that run without faulting the GPU: the weight file loader,
a cache scored on a model it does not belong to, and a device pipeline wait
that runs out (in a child process, under a shrunken wait limit)."""
import os
import subprocess
import sys

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", ["tiny", "tiny-h128"])
def test_weight_file_loads_like_host_arrays(tmp_path, shape):
    """A model loaded from a .pcdw file gives bit-identical results to the
    same weights passed as host arrays."""
    import constrained_decoding_gb300.pcd as pcd
    w = synth.make_weights(synth.model_config(shape), seed=0)
    path = tmp_path / f"{shape}.pcdw"
    synth.write_pcdw(w, str(path))
    req = synth.make_request(1)
    results = []
    for m in (pcd.pcd_load_weights(str(path)), pcd.pcd_load_weights_host(w)):
        c = pcd.pcd_prefill(m, req.prefix)
        results.append(pcd.pcd_score(m, c, req.fields))
        c.free()
        m.free()
    for a, b in zip(*results):
        np.testing.assert_array_equal(a.probs, b.probs)
        np.testing.assert_array_equal(a.logprobs, b.logprobs)
        assert a.label == b.label and a.mass == b.mass


def test_cache_of_another_model_is_refused(tiny_weights):
    import constrained_decoding_gb300.pcd as pcd
    req = synth.make_request(1)
    a = pcd.pcd_load_weights_host(tiny_weights)
    b = pcd.pcd_load_weights_host(tiny_weights)
    ca = pcd.pcd_prefill(a, req.prefix)
    with pytest.raises(pcd.PCDError) as ei:
        pcd.pcd_score(b, ca, req.fields)
    assert ei.value.code == -8
    with pytest.raises(pcd.PCDError) as ei:
        pcd.pcd_prefill_extend(b, ca, req.prefix[:4])
    assert ei.value.code == -8
    ca.free()
    a.free()
    b.free()


def test_device_wait_timeout():
    """Under a 1 ns wait limit the pipelines' bounded waits expire; pcd_sync
    reports PCD_ERR_DEVICE_TIMEOUT, and a model loaded afterwards in the same
    process scores correctly."""
    import timeout_worker as wk
    env = {**os.environ, "PCD_WAIT_LIMIT_MS": "0.000001"}
    r = subprocess.run([sys.executable, wk.__file__], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "timeout codes" in r.stdout and "recovered ok" in r.stdout, r.stdout
