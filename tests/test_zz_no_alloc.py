"""The allocation-free readout entry point (pcd_k_readout_noalloc).

It serves callers that cannot allocate device memory mid-call: a serving
loop whose GPU memory is already held by its own pool, or a latency-critical
stream on which cudaMalloc/cudaFree would synchronise the whole device.  It
keeps its scratch in a fixed array in device memory instead of taking one from
the caller.  Here it is checked through the C ABI against pcd_k_readout (the
same readout with caller-provided scratch) on two calls in a row, with
different problem sizes, so the second call runs on top of whatever the first
left in the shared array.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

TOL = 1e-3  # the readout tests' tolerance on log-sum-exp and gathered logits


def _lib():
    import constrained_decoding_gb300 as pkg
    return pkg.load()


def _case(R, V, d, n_cand, seed):
    rng = np.random.default_rng(seed)
    h = torch.from_numpy(rng.normal(0, 1, (R, d)).astype(np.float16)).cuda()
    w = torch.from_numpy(rng.normal(0, 0.02, (V, d)).astype(np.float16)).cuda()
    rows = np.ascontiguousarray(rng.integers(0, R, n_cand), np.int32)
    toks = np.ascontiguousarray(rng.integers(0, V, n_cand), np.int32)
    return h, w, rows, toks


def _call(noalloc, h, w, rows, toks):
    lib = _lib()
    R, d = h.shape
    V = w.shape[0]
    P = ctypes.POINTER(ctypes.c_int32)
    lse = torch.full((R,), float("nan"), dtype=torch.float32, device="cuda")
    z = torch.full((len(rows),), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    if noalloc:
        rc = lib.pcd_k_readout_noalloc(h.data_ptr(), R, w.data_ptr(), V, d, rows.ctypes.data_as(P),
                                       toks.ctypes.data_as(P), len(rows), lse.data_ptr(), z.data_ptr(),
                                       err.data_ptr(), s)
    else:
        nbytes = lib.pcd_k_readout_scratch_bytes(R, V, len(rows))
        scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        rc = lib.pcd_k_readout(h.data_ptr(), R, w.data_ptr(), V, d, rows.ctypes.data_as(P),
                               toks.ctypes.data_as(P), len(rows), lse.data_ptr(), z.data_ptr(),
                               scratch.data_ptr(), nbytes, err.data_ptr(), s)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return lse.cpu().numpy(), z.cpu().numpy()


def test_noalloc_readout_matches_caller_scratch_twice():
    for R, V, d, seed in ((117, 151936, 1536, 1), (300, 4096, 256, 2)):
        h, w, rows, toks = _case(R, V, d, 3 * R, seed)
        lse_a, z_a = _call(True, h, w, rows, toks)
        lse_b, z_b = _call(False, h, w, rows, toks)
        assert np.all(np.isfinite(lse_a)) and np.all(np.isfinite(z_a))
        np.testing.assert_allclose(lse_a, lse_b, atol=TOL, rtol=0)
        np.testing.assert_allclose(z_a, z_b, atol=TOL, rtol=0)


def test_noalloc_rejects_problems_beyond_the_array():
    lib = _lib()
    from constrained_decoding_gb300._decls import c_int
    limit = 8 * 1024 * 1024
    R, V = 4096, 151936
    assert lib.pcd_k_readout_scratch_bytes(R, V, 0) > limit
    h = torch.zeros(1, dtype=torch.float16, device="cuda")
    lse = torch.zeros(1, dtype=torch.float32, device="cuda")
    rc = lib.pcd_k_readout_noalloc(h.data_ptr(), R, h.data_ptr(), V, 1536, None, None, 0, lse.data_ptr(), None,
                                   None, torch.cuda.current_stream().cuda_stream)
    assert rc == -9  # PCD_ERR_OOM, before anything is launched
