"""The fused vocabulary readout (tensor-core LM-head tiles with an online
log-sum-exp and a candidate gather) against the log-sum-exp and logits
written out in fp64 on the host from the same fp16 operands."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import logsumexp64

pytestmark = pytest.mark.gpu


def _lib():
    import constrained_decoding_gb300 as pkg
    return pkg.load()


def run_readout(h, w, rows, toks, entry="pcd_k_readout"):
    lib = _lib()
    R, d = h.shape
    V = w.shape[0]
    hd, wd = torch.from_numpy(h).cuda(), torch.from_numpy(w).cuda()
    lse = torch.zeros(R, dtype=torch.float32, device="cuda")
    z = torch.zeros(max(len(rows), 1), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows_c = np.ascontiguousarray(rows, np.int32)
    toks_c = np.ascontiguousarray(toks, np.int32)
    P = ctypes.POINTER(ctypes.c_int32)
    s = torch.cuda.current_stream().cuda_stream
    nbytes = lib.pcd_k_readout_scratch_bytes(R, V, len(rows))
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    rc = lib.pcd_k_readout(hd.data_ptr(), R, wd.data_ptr(), V, d, rows_c.ctypes.data_as(P),
                           toks_c.ctypes.data_as(P), len(rows), lse.data_ptr(), z.data_ptr(),
                           scratch.data_ptr(), nbytes, err.data_ptr(), s)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return lse.cpu().numpy(), z.cpu().numpy()[:len(rows)]


def make_case(R, V, d, n_cand, seed):
    rng = np.random.default_rng(seed)
    h = rng.normal(0, 1, (R, d)).astype(np.float16)
    w = (rng.normal(0, 0.02, (V, d))).astype(np.float16)
    rows = rng.integers(0, R, n_cand)
    toks = rng.integers(0, V, n_cand)
    toks[:min(3, n_cand)] = [0, V - 1, V // 2][:min(3, n_cand)]   # first, last and a middle tile
    return h, w, rows, toks


@pytest.mark.parametrize("R,V,d", [(1, 512, 64), (117, 151936, 1536), (260, 151936, 1536), (600, 4096, 256)])
def test_readout_lse_and_gather(R, V, d):
    h, w, rows, toks = make_case(R, V, d, 3 * R, seed=R)
    lse, z = run_readout(h, w, rows, toks)
    logits = h.astype(np.float64) @ w.astype(np.float64).T
    ref_lse = logsumexp64(logits)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-3, rtol=0)
    np.testing.assert_allclose(z, logits[rows, toks], atol=1e-3, rtol=0)
