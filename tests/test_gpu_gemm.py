"""The tcgen05 GEMM against a plain fp32 matmul of the same bf16 operands."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _lib():
    import constrained_decoding_gb300 as pcd
    return pcd.load()


def _ref(a, b):
    return a.float().cpu() @ b.float().cpu().T


def _run(M, N, K, epi, mt, bn, splits, seed=0):
    lib = _lib()
    g = torch.Generator().manual_seed(seed)
    a = (torch.randn(M, K, generator=g) * 0.5).to(torch.float16).cuda()
    b = (torch.randn(N, K, generator=g) * 0.05).to(torch.float16).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    if epi == 0:
        out = torch.zeros(M, N, dtype=torch.float16, device="cuda")
    elif epi == 3:
        out = torch.zeros(M, N // 2, dtype=torch.float16, device="cuda")
    else:
        out = torch.full((M, N), 0.25, dtype=torch.float32, device="cuda")
    rc = lib.pcd_k_gemm(a.data_ptr(), M, K, b.data_ptr(), N, K, K, epi, out.data_ptr(), out.shape[1],
                        mt, bn, splits, err.data_ptr(), s)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = _ref(a, b)
    if epi == 0:
        return out.float().cpu(), ref, 1e-2
    if epi == 3:
        g_, u_ = ref[:, 0::2], ref[:, 1::2]
        return out.float().cpu(), torch.nn.functional.silu(g_) * u_, 2e-2
    return out.cpu(), ref + 0.25, 1e-3


@pytest.mark.parametrize("M,N,K,mt,bn", [
    (128, 128, 64, 1, 128),      # one tile, one k-block
    (128, 256, 128, 1, 256),
    (200, 384, 320, 1, 128),     # ragged M, several tiles
    (333, 512, 1536, 2, 256),    # the branch-pass shape class
    (512, 640, 256, 4, 128),
    (77, 256, 192, 2, 128),      # M smaller than one group
])
def test_gemm_bf16_store(M, N, K, mt, bn):
    out, ref, tol = _run(M, N, K, 0, mt, bn, 1)
    err = (out - ref).abs().max().item()
    assert err < tol * max(1.0, ref.abs().max().item()), err


@pytest.mark.parametrize("splits", [1, 3, 8])
def test_gemm_f32_accumulate(splits):
    epi = 1 if splits == 1 else 2
    out, ref, tol = _run(300, 256, 1024, epi, 1, 128, splits, seed=1)
    assert (out - ref).abs().max().item() < tol


def test_gemm_swiglu():
    out, ref, tol = _run(150, 512, 256, 3, 2, 256, 1, seed=2)
    assert (out - ref).abs().max().item() < tol


@pytest.mark.parametrize("M,N,K,bn", [
    (825, 17920, 1536, 256),     # the gate/up projection: 490 units, the last 5 N tiles as 140 narrow units
    (640, 8192, 256, 256),       # 160 units: 2 N tiles become 40 narrow units
    (512, 5120, 192, 128),       # 128-wide tiles: 2 N tiles become 16 narrow units
])
def test_gemm_swiglu_narrow_tail(M, N, K, bn):
    """More units than SMs with a part-filled last wave: the last N tiles run
    as 64-column units (another B box, MMA width and epilogue width)."""
    out, ref, tol = _run(M, N, K, 3, 1, bn, 1, seed=9)
    assert (out - ref).abs().max().item() < tol


def test_gemm_auto_tiling_large():
    out, ref, tol = _run(332, 2048, 1536, 2, 0, 0, 0, seed=3)
    assert (out - ref).abs().max().item() < 1e-3


@pytest.mark.parametrize("epi,bn,splits", [(1, 128, 1), (2, 256, 4), (3, 256, 1), (3, 128, 1)])
def test_gemm_split_activation(epi, bn, splits):
    """A carried as fp16 hi + lo: the product matches the fp32 activation's
    product far more closely than the hi half alone."""
    lib = _lib()
    M, N, K = 313, 1024, 1536
    g = torch.Generator().manual_seed(7)
    a32 = torch.randn(M, K, generator=g)
    hi = a32.half()
    lo = (a32 - hi.float()).half()
    b = (torch.randn(N, K, generator=g) * 0.05).half()
    ref = a32.double() @ b.double().T
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    if epi == 3:
        out = torch.zeros(M, N // 2, dtype=torch.float16, device="cuda")
        ref = (torch.nn.functional.silu(ref[:, 0::2]) * ref[:, 1::2])
    else:
        out = torch.zeros(M, N, dtype=torch.float32, device="cuda")
    hi_d, lo_d, b_d = hi.cuda(), lo.cuda(), b.cuda()   # keep the device copies alive for the call
    rc = lib.pcd_k_gemm_split(hi_d.data_ptr(), lo_d.data_ptr(), M, K, b_d.data_ptr(), N, K, K, epi,
                              out.data_ptr(), out.shape[1], bn, splits, err.data_ptr(), s)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.double().cpu()
    hi_only = hi.double() @ b.double().T
    if epi == 3:
        hi_only = torch.nn.functional.silu(hi_only[:, 0::2]) * hi_only[:, 1::2]
        # fp16 output rounding dominates: within one fp16 ulp of the exact value
        assert ((got - ref).abs() <= ref.abs() * 2.0 ** -10 + 1e-3).all()
    else:
        e_split = (got - ref).abs().max().item()
        e_hi = (hi_only - ref).abs().max().item()
        assert e_split < 2e-4 and e_split < e_hi / 4, (e_split, e_hi)


@pytest.mark.parametrize("M,N,K,epi,bn,splits", [
    (128, 256, 256, 0, 128, 1),     # one pair tile, the peer's rows all past M
    (300, 512, 512, 0, 128, 1),     # ragged M: the last pair tile half empty
    (825, 2048, 1536, 0, 256, 1),
    (825, 1536, 8960, 2, 256, 3),   # split-K with atomics
    (825, 4096, 1536, 3, 128, 1),   # SwiGLU epilogue
    (57, 512, 512, 1, 256, 1),      # fp32 add, fewer rows than one CTA
])
def test_gemm_cta_pair(M, N, K, epi, bn, splits):
    """CTA pairs sharing one 256-row tcgen05 MMA (each CTA: its 128 rows of
    A, half of the B tile, half of the accumulator rows)."""
    out, ref, tol = _run(M, N, K, epi, 3, bn, splits)
    err = (out - ref).abs().max().item()
    assert err < tol * max(1.0, ref.abs().max().item()), err
