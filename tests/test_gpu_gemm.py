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


# path: 0 CUDA cores, 1 tcgen05 (library's choice), 2 row-tiled, 3 weight-stationary,
# 7 persistent pair tiles on the pair's joint MMA
@pytest.mark.parametrize("path", [1, 0, 2, 3, 7])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_matches_definition(path, M, N, K):
    if path == 3 and M > 256:
        pytest.skip("weight-stationary kernels hold at most 256 rows")
    _check_gemm(path, M, N, K)


# column widths, K splits and ring depths of the row-tiled kernel, forced; one
# and two 128-row sub-tiles, ragged columns and K
@pytest.mark.parametrize("bn,splits,stages", [(16, 1, 0), (48, 3, 0), (176, 1, 0), (256, 2, 3), (144, 8, 4),
                                              (80, 1, 2)])
@pytest.mark.parametrize("M,N,K", [(100, 1000, 1376), (200, 4608, 2048), (33, 384, 4096)])
def test_row_tiled_configs(bn, splits, stages, M, N, K):
    from drift_aware_kv_gb300 import polestar as P
    _check_gemm(P.gemm_path(2, stages, splits, bn), M, N, K)


# ring depths and cluster K splits of the weight-stationary kernel, forced
@pytest.mark.parametrize("stages,splits", [(2, 1), (3, 2), (4, 4), (8, 1), (5, 8), (6, 3)])
@pytest.mark.parametrize("M,N,K", [(136, 4096, 4096), (16, 640, 1024), (256, 384, 3584)])
def test_weight_stationary_configs(stages, splits, M, N, K):
    from drift_aware_kv_gb300 import polestar as P
    np_rows = max(16, (M + 15) // 16 * 16)
    stage = 128 * 64 * 2 + np_rows * 64 * 2
    if stages * stage + 2048 > 232448 or (splits > 1 and stages * stage < np_rows * 132 * 4):
        with pytest.raises(P.PolestarError):  # does not fit in shared memory
            _check_gemm(P.gemm_path(3, stages, splits), M, N, K)
        return
    _check_gemm(P.gemm_path(3, stages, splits), M, N, K)


# column widths and ring depths of the persistent pair kernel, forced: tiles cut
# at ragged rows, columns and K, one pair tile and many waves of them
@pytest.mark.parametrize("bn,stages", [(256, 0), (256, 7), (192, 2), (240, 3), (128, 0), (32, 8), (16, 4)])
@pytest.mark.parametrize("M,N,K", [(700, 1000, 1376), (2560, 4096, 4096), (300, 4608, 2048), (1, 96, 64),
                                   (513, 12288, 4096)])
def test_two_sm_pair_configs(bn, stages, M, N, K):
    from drift_aware_kv_gb300 import polestar as P
    _check_gemm(P.gemm_path(7, stages, 0, bn), M, N, K)


def _check_gemm(path, M, N, K):
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


@pytest.mark.parametrize("path,m_live", [(1, 77), (2, 77), (3, 77), (3, 0), (3, 1), ((2 << 16) | 3, 17),
                                         ((4 << 16) | 3, 200), (7, 77), (7, 0), (7, 129), (7, 200)])
def test_gemm_device_row_count_leaves_tail_untouched(path, m_live):
    from drift_aware_kv_gb300 import polestar as P
    g = torch.Generator(device="cpu").manual_seed(5)
    M, N, K = 200, 256, 1024
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    W = (0.02 * torch.randn(N, K, generator=g)).to(torch.bfloat16).cuda()
    C = torch.full((M, N), -7.0, device="cuda")
    m = torch.tensor([m_live], dtype=torch.int32, device="cuda")
    P.debug_gemm(A, W, C, path, m_dev=m)
    torch.cuda.synchronize()
    ref = _ref(A, W, np.arange(m_live))
    assert np.allclose(C[:m_live].double().cpu().numpy(), ref, atol=1e-3)
    assert torch.all(C[m_live:] == -7.0)


def test_gemm_rejects_unrunnable_choice():
    from drift_aware_kv_gb300 import polestar as P
    A = torch.zeros(300, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(300, 128, device="cuda")
    with pytest.raises(P.PolestarError):
        P.debug_gemm(A, W, C, P.gemm_path(3))          # more than 256 rows
    with pytest.raises(P.PolestarError):
        P.debug_gemm(A[:64], W, C[:64], P.gemm_path(3, 9))   # ring deeper than the kernel's barriers
    with pytest.raises(P.PolestarError):
        P.debug_gemm(A[:64], W, C[:64], P.gemm_path(3, 2, 9))  # cluster larger than 8
    for kernel in (4, 5, 6, 8, 15):                  # kernel numbers the library does not have
        with pytest.raises(P.PolestarError):
            P.debug_gemm(A[:64], W, C[:64], P.gemm_path(kernel))
    with pytest.raises(P.PolestarError):
        P.debug_gemm(A, W, C, P.gemm_path(7, 8, 0, 256))  # eight 32 KB stages do not fit


@pytest.mark.parametrize("M,Ns,K", [(136, [4096, 1024, 1024], 4096), (32, [12288, 12288], 4096), (128, [4096], 12288),
                                    (80, [3584], 3584), (200, [512, 512], 1184), (2560, [12288], 4096),
                                    (768, [4096, 1024, 1024], 4096)])
def test_library_choice_is_valid_and_reproducible(M, Ns, K):
    """The launch the library picks is a runnable configuration, and forcing
    exactly that configuration reproduces the automatic launch bit for bit."""
    from drift_aware_kv_gb300 import polestar as P
    ch = P.gemm_choice(M, Ns, K)
    assert ch["kernel"] in (1, 2, 5) and ch["splits"] >= 1 and ch["stages"] >= 2
    assert ch["bn"] % 16 == 0 and 16 <= ch["bn"] <= 256
    N = Ns[0]
    g = torch.Generator(device="cpu").manual_seed(M + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    W = (0.02 * torch.randn(N, K, generator=g)).to(torch.bfloat16).cuda()
    c1 = torch.empty(M, N, device="cuda")
    c2 = torch.empty(M, N, device="cuda")
    P.debug_gemm(A, W, c1, P.gemm_path(1))
    ch1 = P.gemm_choice(M, [N], K)
    kern = {1: 2, 2: 3, 5: 7}[ch1["kernel"]]
    path = P.gemm_path(kern, ch1["stages"], ch1["splits"], ch1["bn"] if ch1["kernel"] in (1, 5) else 0)
    P.debug_gemm(A, W, c2, path)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


def _swiglu_ref(A, Wg, Wu, rows):
    a = A[rows].double().cpu().numpy()
    g = a @ Wg.double().cpu().numpy().T
    u = a @ Wu.double().cpu().numpy().T
    return g / (1.0 + np.exp(-g)) * u


# gate/up projections with the activation fused into the epilogue: library
# choice and forced row-tiled configurations (direct epilogue, K split over a
# cluster, ragged widths and rows)
@pytest.mark.parametrize("path", [1, (176 // 16) << 24 | 2, (48 // 16) << 24 | (3 << 16) | 2,
                                  (128 // 16) << 24 | (6 << 16) | 2, (256 // 16) << 24 | 2])
@pytest.mark.parametrize("M,F,K", [(128, 12288, 4096), (136, 1376, 512), (7, 200, 448), (300, 1000, 1184)])
def test_gate_up_swiglu_fused(path, M, F, K):
    from drift_aware_kv_gb300 import polestar as P
    g = torch.Generator(device="cpu").manual_seed(M * 31 + F + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    Wg = (0.05 * torch.randn(F, K, generator=g)).to(torch.bfloat16).cuda()
    Wu = (0.05 * torch.randn(F, K, generator=g)).to(torch.bfloat16).cuda()
    act = torch.full((M, F + 8), float("nan"), dtype=torch.bfloat16, device="cuda")
    try:
        P.debug_gemm_swiglu(A, Wg, Wu, act, path)
    except P.PolestarError:
        if path == 1:
            pytest.skip("library picks a kernel without the fused epilogue for this shape")
        raise
    torch.cuda.synchronize()
    rows = np.arange(M) if M * F * K <= 2**31 else np.unique(np.linspace(0, M - 1, 48).astype(int))
    ref = _swiglu_ref(A, Wg, Wu, rows)
    got = act[rows, :F].double().cpu().numpy()
    assert np.all(np.isfinite(got))
    # bf16 output: half an ulp of bf16 plus the fp32 accumulation
    assert np.all(np.abs(got - ref) <= 4e-3 * np.abs(ref) + 1e-4 * np.abs(ref).max()), np.abs(got - ref).max()
    assert torch.isnan(act[:, F:].float()).all()  # nothing written past F


# the same through the two-SM pair kernel (path 7: bn / 2 gate and bn / 2 up
# columns per pair tile; one or two k-blocks per stage; ragged F and rows)
@pytest.mark.parametrize("path", [(256 // 16) << 24 | (2 << 16) | 7, (192 // 16) << 24 | (1 << 16) | 7,
                                  (128 // 16) << 24 | (2 << 16) | (3 << 8) | 7])
@pytest.mark.parametrize("M,F,K", [(513, 1000, 1408), (300, 1376, 512), (2560, 4096, 4096)])
def test_gate_up_swiglu_pair_kernel(path, M, F, K):
    test_gate_up_swiglu_fused(path, M, F, K)


# the pair kernel's tile walk in groups of row pairs (about 48 MB of A rows per
# group): K = 12288 gives groups of 8 row pairs, so 2560 rows walk two groups
# (8 + 2 pairs) and 4352 rows three (8 + 8 + 1); every output element once
@pytest.mark.parametrize("M,N,K", [(2560, 1000, 12288), (4352, 512, 12288)])
def test_two_sm_pair_grouped_walk(M, N, K):
    from drift_aware_kv_gb300 import polestar as P
    _check_gemm(P.gemm_path(7, 0, 2, 256), M, N, K)
    _check_gemm(P.gemm_path(7, 0, 1, 192), M, N, K)


# the pair kernel's split tail: with a device row count, the tiles of the last,
# partly filled wave are split along K over the idle clusters (each split sums
# one column slice over all splits' partial tiles, in split order) when at
# least four splits fit and a tile is at least 32 stages deep (K = 12288 at two
# k-blocks per stage: 96).  With 76 clusters: 2560 rows leave 8 tail tiles (eight
# splits each), 256 rows 16 tiles in all (four splits each), 300 and 4096 rows
# too many for a split.  Live rows must match the definition, rows past the
# count stay untouched, and repeated launches (the split counters cleared by
# each launch for the next) give identical bits.
@pytest.mark.parametrize("m_live", [2560, 256, 300, 4096, 0])
def test_two_sm_pair_split_tail(m_live):
    from drift_aware_kv_gb300 import polestar as P
    g = torch.Generator(device="cpu").manual_seed(11)
    M, N, K = 4096, 4096, 12288
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    W = (0.02 * torch.randn(N, K, generator=g)).to(torch.bfloat16).cuda()
    m = torch.tensor([m_live], dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(3):
        C = torch.full((M, N), -7.0, device="cuda")
        P.debug_gemm(A, W, C, P.gemm_path(7, 0, 2, 256), m_dev=m)
        torch.cuda.synchronize()
        outs.append(C)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    C = outs[0]
    assert torch.all(C[m_live:] == -7.0)
    if m_live:
        rows = np.unique(np.linspace(0, m_live - 1, 48).astype(int))
        ref = _ref(A, W, rows)
        got = C[rows].double().cpu().numpy()
        scale = np.sqrt((A[rows].double().cpu().numpy() ** 2).sum(1))[:, None] * \
            np.sqrt((W.double().cpu().numpy() ** 2).sum(1))[None, :]
        assert (np.abs(got - ref) / scale).max() < 2e-6


def test_gate_up_swiglu_matches_unfused():
    """The fused epilogue computes silu(g) * u from the same fp32 accumulators as
    the unfused projections (same kernel, same tile width), so the results agree
    to the bf16 rounding of the activation."""
    from drift_aware_kv_gb300 import polestar as P
    g = torch.Generator(device="cpu").manual_seed(3)
    M, F, K = 128, 4096, 4096
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    Wg = (0.02 * torch.randn(F, K, generator=g)).to(torch.bfloat16).cuda()
    Wu = (0.02 * torch.randn(F, K, generator=g)).to(torch.bfloat16).cuda()
    act = torch.empty(M, F, dtype=torch.bfloat16, device="cuda")
    path = (128 // 16) << 24 | 2  # row-tiled, 64 gate + 64 up columns per tile, no K split
    P.debug_gemm_swiglu(A, Wg, Wu, act, path)
    C = torch.empty(M, 2 * F, device="cuda")
    P.debug_gemm(A, torch.cat([Wg, Wu]), C, P.gemm_path(2, 0, 1, 128))
    torch.cuda.synchronize()
    gg, uu = C[:, :F], C[:, F:]
    ref = (gg / (1.0 + torch.exp(-gg)) * uu).to(torch.bfloat16)
    assert (act.float() - ref.float()).abs().max().item() <= 2 ** -7 * ref.float().abs().max().item()


# two-SM pair kernel with two k-blocks per stage (one 3D TMA box per operand)
@pytest.mark.parametrize("bn,stages", [(256, 0), (192, 2), (128, 3)])
@pytest.mark.parametrize("M,N,K", [(2560, 4096, 4096), (700, 1000, 1408), (513, 12288, 4096), (1, 96, 128)])
def test_two_sm_pair_two_kblocks(bn, stages, M, N, K):
    from drift_aware_kv_gb300 import polestar as P
    _check_gemm(P.gemm_path(7, stages, 2, bn), M, N, K)


def test_two_kblock_stages_need_whole_kblocks():
    from drift_aware_kv_gb300 import polestar as P
    A = torch.zeros(300, 100, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(256, 100, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(300, 256, device="cuda")
    with pytest.raises(P.PolestarError):
        P.debug_gemm(A, W, C, P.gemm_path(7, 0, 2, 256))  # K = 100 is not a multiple of 64


# row-tiled kernel with two k-blocks per stage: K splits whose ranges end inside
# a stage (odd k-block counts), one and two row sub-tiles
@pytest.mark.parametrize("bn,splits,stages", [(176, 1, 0), (128, 3, 0), (208, 6, 2), (256, 2, 0), (48, 8, 0)])
@pytest.mark.parametrize("M,N,K", [(100, 1000, 1344), (200, 4608, 2048), (33, 384, 4096), (128, 24576, 4096)])
def test_row_tiled_two_kblocks(bn, splits, stages, M, N, K):
    from drift_aware_kv_gb300 import polestar as P
    mt = 2 if M > 128 else 1
    stage = 2 * (mt * 128 * 64 * 2 + bn * 64 * 2)  # two k-blocks of the A sub-tiles and the W tile
    max_stages = min(8, (232448 - 2048) // stage)
    st = stages or max_stages
    if st < 2 or st > max_stages or (splits > 1 and st * stage < 128 * (bn + 4) * 4):
        with pytest.raises(P.PolestarError):  # does not fit in shared memory
            _check_gemm(P.gemm_path(2, stages, splits, bn, kpack=2), M, N, K)
        return
    _check_gemm(P.gemm_path(2, stages, splits, bn, kpack=2), M, N, K)
