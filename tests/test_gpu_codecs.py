"""The storage formats of the quantization ablation (paper: "Polestar: Drift-Aware
Cache Calibration and Token Commitment for Efficient Inference of Diffusion
LLMs", Table 11; NVFP4 of App. C.3) on the GPU through the C ABI, against the
CPU oracle (oracle/residual_codecs.py) on the same fp32 values: codes and
scales bit for bit, decoded states exactly, plain and residual, at LLaDA-8B
and Dream-7B widths, a ragged row count and edge rows (zero rows, zero blocks,
ties on the rounding grids, values far apart in magnitude)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FORMATS = ["fp16", "fp8", "int8", "mxfp4", "int2", "nvfp4"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from drift_aware_kv_gb300.build import build
    build()


def _states(rows, d, K, seed):
    """Clustered window-like states: K anchors + per-row spread, plus edge rows."""
    from oracle import polestar_oracle as O
    g = np.random.default_rng(seed)
    cent = g.standard_normal((K, d)) * 2.0
    labels = g.integers(0, K, rows).astype(np.uint8)
    h = cent[labels] + 0.3 * g.standard_normal((rows, d))
    h[1] = 0.0                                            # zero row
    h[2, :64] = 0.0                                       # zero blocks / groups
    h[3] = g.standard_normal(d) * np.where(np.arange(d) % 2, 1e-6, 1e3)  # magnitudes far apart
    h[4] = np.resize([0.25, -0.75, 1.25, -2.5, 3.5, 5.0, 0.5, -6.0], d)  # E2M1 midpoints and grid values
    h = O.to_f32(h)
    anchors = O.to_f32(np.stack([h[labels == c].mean(0) if np.any(labels == c) else np.zeros(d) for c in range(K)]))
    return h, anchors, labels


def _oracle_codes(fmt, r):
    """Oracle codes/scales in the library's storage layout."""
    from oracle import polestar_oracle as O
    from oracle import residual_codecs as R
    rows, d = r.shape
    if fmt == "fp16":
        return np.asarray(r, dtype=np.float64).astype(np.float16).view(np.uint8).reshape(-1), np.zeros(0, np.uint8)
    if fmt == "fp8":
        c, s = R.fp8_encode(r)
        return c.reshape(-1), s.astype(np.float32).view(np.uint8)
    if fmt == "int8":
        c, s = R.int8_encode(r)
        return c.view(np.uint8).reshape(-1), s.astype(np.float32).view(np.uint8)
    if fmt == "int2":
        c, s = R.int2_encode(r)
        t = (c.astype(np.int64) & 3).reshape(rows, d // 4, 4)
        packed = (t[..., 0] | t[..., 1] << 2 | t[..., 2] << 4 | t[..., 3] << 6).astype(np.uint8)
        return packed.reshape(-1), s.astype(np.float32).view(np.uint8)
    if fmt == "mxfp4":
        c, e = R.mxfp4_encode(r)
        packed = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
        return packed.reshape(-1), (e + 127).astype(np.uint8).reshape(-1)
    c, sb, _ = O.nvfp4_encode(r)
    packed = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    return packed.reshape(-1), sb.reshape(-1)


def _oracle_decode(fmt, r):
    from oracle import residual_codecs as R
    if fmt == "fp16":
        return R.fp16_roundtrip(r)
    return R.FORMATS[fmt][0](r)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("rows,d", [(96, 4096), (64, 3584), (37, 512)])
def test_codec_matches_oracle_bit_for_bit(fmt, residual, rows, d):
    from drift_aware_kv_gb300 import polestar as P
    from oracle import polestar_oracle as O
    h, anchors, labels = _states(rows, d, 8, rows + d)
    hg = torch.tensor(h, dtype=torch.float32, device="cuda")
    ag = torch.tensor(anchors, dtype=torch.float32, device="cuda") if residual else None
    lg = torch.tensor(labels, dtype=torch.uint8, device="cuda") if residual else None
    codes, scales = P.codec_encode(fmt, hg, ag, lg)
    dec = P.codec_decode(fmt, codes, scales, rows, d, ag, lg)
    torch.cuda.synchronize()
    r = O.to_f32(h - anchors[labels]) if residual else h
    oc, os_ = _oracle_codes(fmt, r)
    assert np.array_equal(codes.cpu().numpy(), oc), f"{fmt} codes"
    assert np.array_equal(scales.cpu().numpy(), os_), f"{fmt} scales"
    ref = _oracle_decode(fmt, r)
    if residual:
        ref = O.to_f32(anchors[labels] + ref)
    got = dec.cpu().numpy().astype(np.float64)
    assert np.array_equal(got, ref), f"{fmt} decoded values, max diff {np.max(np.abs(got - ref))}"


def test_codec_sizes_and_argument_errors():
    from drift_aware_kv_gb300 import polestar as P
    assert P.codec_bytes("nvfp4", 96, 4096) == (96 * 2048, 96 * 256)
    assert P.codec_bytes("mxfp4", 96, 4096) == (96 * 2048, 96 * 128)
    assert P.codec_bytes("int2", 10, 64) == (160, 40)
    assert P.codec_bytes("fp16", 3, 32) == (192, 0)
    lib = P.load()
    assert lib.polestar_codec_bytes(9, 1, 32, None, None) == -1
    assert lib.polestar_codec_bytes(0, 1, 48, None, None) == -1
    h = torch.zeros(4, 64, device="cuda")
    c = torch.zeros(4 * 64, dtype=torch.uint8, device="cuda")
    s = torch.zeros(64, dtype=torch.uint8, device="cuda")
    a = torch.zeros(2, 64, device="cuda")
    assert lib.polestar_codec_encode(1, P._ptr(h), 4, 64, P._ptr(a), None, P._ptr(c), P._ptr(s), None) == \
        P.ERR_INVALID_ARG  # anchors without labels
    assert lib.polestar_codec_encode(1, P._ptr(h), 4, 64, None, None, P._ptr(c), None, None) == P.ERR_INVALID_ARG
    assert lib.polestar_codec_decode(3, P._ptr(c), P._ptr(s), 4, 40, None, None, P._ptr(h), None) == \
        P.ERR_INVALID_ARG
