"""The weight-streaming GEMM (weights as the 256-row side of a CTA-pair MMA,
tokens as its N side) against a plain fp32 matmul of the same fp16 operands."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _lib():
    import constrained_decoding_gb300 as pcd
    return pcd.load()


def _run(M, N, K, epi, splits, lo, seed=0):
    lib = _lib()
    g = torch.Generator().manual_seed(seed)
    a32 = torch.randn(M, K, generator=g) * 0.5
    a = a32.to(torch.float16)
    a_lo = (a32 - a.float()).to(torch.float16) if lo else None
    b = (torch.randn(N, K, generator=g) * 0.05).to(torch.float16)
    ad, bd = a.cuda(), b.cuda()
    ald = a_lo.cuda() if lo else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    if epi == 3:
        out = torch.zeros(M, N // 2, dtype=torch.float16, device="cuda")
    else:
        out = torch.full((M, N), 0.25, dtype=torch.float32, device="cuda")
    rc = lib.pcd_k_gemm_swap(ad.data_ptr(), ald.data_ptr() if lo else None, M, K, bd.data_ptr(), N, K, K, epi,
                             out.data_ptr(), out.shape[1], splits, err.data_ptr(), s)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    af = a.double() + (a_lo.double() if lo else 0.0)
    ref = af @ b.double().T
    if epi == 3:
        g_, u_ = ref[:, 0::2], ref[:, 1::2]
        return out.double().cpu(), torch.nn.functional.silu(g_) * u_
    return out.double().cpu(), ref + 0.25


SHAPES = [
    (1, 256, 64),        # one token, one k block
    (20, 512, 128),      # tokens past the padded piece are zero-filled
    (64, 768, 192),      # one piece, N of three pair tiles
    (255, 256, 256),     # one piece of 256 columns
    (257, 512, 320),     # two pieces (288 = 2 x 144)
    (313, 2048, 1536),   # the 28-field branch pass: QKV / O shapes
    (363, 1280, 704),    # the long-document branch count, ragged weight tiles
    (512, 512, 128),     # the largest token count
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("lo", [False, True])
def test_swap_f32_add(M, N, K, lo):
    out, ref = _run(M, N, K, 1, 1, lo)
    assert (out - ref).abs().max().item() < 2e-3 * max(1.0, ref.abs().max().item())


@pytest.mark.parametrize("M,N,K,splits", [(313, 1536, 1536, 6), (313, 1536, 8960, 12), (100, 512, 512, 0),
                                          (400, 1024, 2048, 3)])
@pytest.mark.parametrize("lo", [False, True])
def test_swap_f32_atomic_split(M, N, K, splits, lo):
    out, ref = _run(M, N, K, 2, splits, lo)
    assert (out - ref).abs().max().item() < 2e-3 * max(1.0, ref.abs().max().item())


@pytest.mark.parametrize("M,N,K", [(1, 256, 64), (33, 512, 128), (313, 17920 // 4, 1536), (300, 1024, 256),
                                   (512, 512, 192)])
@pytest.mark.parametrize("lo", [False, True])
def test_swap_swiglu(M, N, K, lo):
    out, ref = _run(M, N, K, 3, 1, lo)
    assert (out - ref).abs().max().item() < 2e-2 * max(1.0, ref.abs().max().item())


def test_swap_rejects_bad_shapes():
    lib = _lib()
    x = torch.zeros(16, dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    # too many token rows, K not a multiple of 64, a split with the SwiGLU epilogue
    assert lib.pcd_k_gemm_swap(x.data_ptr(), None, 513, 64, x.data_ptr(), 256, 64, 64, 1, x.data_ptr(), 256, 1,
                               None, s) == -1
    assert lib.pcd_k_gemm_swap(x.data_ptr(), None, 16, 96, x.data_ptr(), 256, 96, 96, 1, x.data_ptr(), 256, 1,
                               None, s) == -1
    assert lib.pcd_k_gemm_swap(x.data_ptr(), None, 16, 64, x.data_ptr(), 256, 64, 64, 3, x.data_ptr(), 128, 2,
                               None, s) == -1
