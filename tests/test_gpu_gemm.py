"""Projection kernels through the C ABI against the plain definition of the
contraction, C[m, n] = sum_k A[m, k] W[n, k], evaluated in float64 on the same
bf16 values (the decoder-layer projections of Eq. 3 / §4.1)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHAPES = [  # (M, N, K): ragged tails, single rows, the gathered-row sizes of the
    # LLaDA-8B / Dream-7B layer loop, and a block-entry row count
    (1, 128, 64), (7, 200, 448), (33, 384, 1376), (80, 4096, 4096), (136, 4096, 4096),
    (136, 1024, 3584), (257, 512, 1184), (96, 18944, 3584), (768, 4096, 4096),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from drift_aware_kv_gb300.build import build
    build()


def _ref(A, W, rows):
    a = A[rows].double().cpu().numpy()
    w = W.double().cpu().numpy()
    return a @ w.T


@pytest.mark.parametrize("path", [1, 0])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_matches_definition(path, M, N, K):
    from drift_aware_kv_gb300 import polestar as P
    g = torch.Generator(device="cpu").manual_seed(M * 7919 + N * 31 + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    W = (0.02 * torch.randn(N, K, generator=g)).to(torch.bfloat16).cuda()
    C = torch.full((M, N), float("nan"), device="cuda")
    P.debug_gemm(A, W, C, path)
    torch.cuda.synchronize()
    rows = np.arange(M) if M * N * K <= 2**31 else np.unique(np.linspace(0, M - 1, 64).astype(int))
    ref = _ref(A, W, rows)
    got = C[rows].double().cpu().numpy()
    scale = np.sqrt((A[rows].double().cpu().numpy() ** 2).sum(1))[:, None] * \
        np.sqrt((W.double().cpu().numpy() ** 2).sum(1))[None, :]
    err = np.abs(got - ref) / scale
    assert np.all(np.isfinite(got))
    assert err.max() < 2e-6, err.max()


def test_gemm_device_row_count_leaves_tail_untouched():
    from drift_aware_kv_gb300 import polestar as P
    g = torch.Generator(device="cpu").manual_seed(5)
    M, N, K = 200, 256, 512
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    W = (0.02 * torch.randn(N, K, generator=g)).to(torch.bfloat16).cuda()
    C = torch.full((M, N), -7.0, device="cuda")
    m = torch.tensor([77], dtype=torch.int32, device="cuda")
    P.debug_gemm(A, W, C, 1, m_dev=m)
    torch.cuda.synchronize()
    ref = _ref(A, W, np.arange(77))
    assert np.allclose(C[:77].double().cpu().numpy(), ref, atol=1e-3)
    assert torch.all(C[77:] == -7.0)
