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
    """A model loaded from a .pcdw file scores like the same weights passed
    as host arrays.  At head dim 128 the projections run split-K with fp32
    atomic adds, whose order varies from run to run; a different order can
    tip an fp16 rounding of an activation, so the two agree to that
    run-to-run spread (seen up to 3e-5 in a probability), not bit for bit.
    The bounds sit well above that spread and far below what a misread or
    misconverted tensor gives (differences of order 0.1)."""
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
        np.testing.assert_allclose(a.probs, b.probs, rtol=0, atol=2e-4)
        np.testing.assert_allclose(a.logprobs, b.logprobs, rtol=1e-3, atol=1e-3)
        assert a.label == b.label
        assert abs(a.mass - b.mass) <= 1e-3 * max(1.0, abs(b.mass))


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


def test_handles_outliving_their_model():
    """Freeing a model releases the device memory of its caches and plans and
    detaches them: freeing them afterwards only deletes the handles, and a
    detached cache or plan is refused by another model."""
    import constrained_decoding_gb300.pcd as pcd
    from constrained_decoding_gb300 import load
    lib = load()
    w = synth.make_weights(synth.model_config("tiny"), seed=0)
    req = synth.make_request(1)
    a = pcd.pcd_load_weights_host(w)
    cache = pcd.pcd_prefill(a, req.prefix)
    plan = pcd.pcd_plan_create(a, req.fields)
    handles = (cache.handle, plan.handle)
    lib.pcd_model_free(a.handle)        # through the C ABI: the binding's handles stay live
    a.handle = None
    b = pcd.pcd_load_weights_host(w)
    with pytest.raises(pcd.PCDError) as ei:
        pcd.pcd_score(b, cache, req.fields)
    assert ei.value.code == -8
    lib.pcd_cache_free(handles[0])
    lib.pcd_plan_free(handles[1])
    cache.handle = plan.handle = None
    # the process is intact: the second model scores as usual
    c2 = pcd.pcd_prefill(b, req.prefix)
    got = pcd.pcd_score(b, c2, req.fields)
    assert all(abs(float(np.sum(g.probs)) - 1.0) < 1e-4 for g in got)
    c2.free()
    b.free()


def test_bounded_wait_gives_up():
    """A wait on an mbarrier that nothing arrives on ends after its limit with
    an error code in the device error word, and the stream stays usable."""
    import torch
    from constrained_decoding_gb300 import load
    lib = load()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    el = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    for limit in (1_000, 2_000_000):
        err.zero_()
        assert lib.pcd_k_wait_probe(limit, err.data_ptr(), el.data_ptr(), st) == 0
        torch.cuda.synchronize()
        assert int(err.item()) == 6
        assert limit <= int(el.item()) < limit + 50_000_000, (limit, int(el.item()))
    assert lib.pcd_k_wait_probe(-1, err.data_ptr(), el.data_ptr(), st) == -1
    assert lib.pcd_k_wait_probe(10, 0, 0, st) == -1
    # the context still runs work after the abandoned waits
    a = torch.randn(256, 128, device="cuda").half()
    b = torch.randn(256, 128, device="cuda").half()
    out = torch.zeros(256, 256, device="cuda")
    assert lib.pcd_k_gemm(a.data_ptr(), 256, 128, b.data_ptr(), 256, 128, 128, 1, out.data_ptr(), 256, 0, 0, 1,
                          None, st) == 0
    torch.testing.assert_close(out, a.float() @ b.float().T, atol=1e-2, rtol=1e-3)


def test_device_wait_timeout():
    """Under a 1 ns wait limit the pipelines' bounded waits expire; pcd_sync
    reports PCD_ERR_DEVICE_TIMEOUT, and a model loaded afterwards in the same
    process scores correctly."""
    import timeout_worker as wk
    env = {**os.environ, "PCD_WAIT_LIMIT_MS": "0.000001"}
    r = subprocess.run([sys.executable, wk.__file__], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "timeout codes" in r.stdout and "recovered ok" in r.stdout, r.stdout
