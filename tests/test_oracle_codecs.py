"""Pins of the oracle's hidden-state storage formats (the quantization ablation of
"Polestar: Drift-Aware Cache Calibration and Token Commitment for Efficient
Inference of Diffusion LLMs", Table 11; NVFP4 of App. C.3 is pinned in
test_oracle_pins.py)."""
import math

import numpy as np
import pytest

from oracle import polestar_oracle as O
from oracle import residual_codecs as R


def test_fp16_constants():
    """binary16 nearest-even: 1/3 -> 0.333251953125 (10-bit mantissa 0x155), the
    largest finite value 65504, the smallest subnormal 2^-24 and ties to even."""
    v = R.fp16_roundtrip(np.array([1 / 3, 65504.0, 2.0 ** -24, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11]))
    assert v[0] == 0.333251953125 and v[1] == 65504.0 and v[2] == 2.0 ** -24
    assert v[3] == 1.0 and v[4] == 1 + 2.0 ** -9


def test_fp8_rows_scale_grid_and_error():
    g = np.random.default_rng(0)
    r = O.to_f32(g.standard_normal((5, 64)) * np.array([1e-3, 0.1, 1.0, 10.0, 300.0])[:, None])
    r[2] = 0.0
    codes, s = R.fp8_encode(r)
    dec = R.fp8_decode(codes, s)
    amax = np.max(np.abs(r), axis=1)
    assert s[2] == 0 and np.all(dec[2] == 0)
    for i in (0, 1, 3, 4):
        assert s[i] == np.float32(amax[i] / np.float32(448.0))
        q = O.e4m3_value(codes[i])
        # the decoded row is the code's E4M3 value times the row scale (fp32)
        assert np.array_equal(dec[i], O.to_f32(q * s[i]))
        assert np.all(np.signbit(q) == np.signbit(r[i].astype(np.float32)))
        # the row maximum maps to the top of the grid
        assert np.max(np.abs(q)) == 448.0
        # nearest rounding: within half a quantum (2^-4 relative in the normal range)
        x = np.abs(r[i] / s[i])
        normal = x >= 2.0 ** -6
        assert np.all(np.abs(np.abs(q) - x)[normal] <= x[normal] * 2.0 ** -4 + 1e-6)
        assert np.all(np.abs(np.abs(q) - x)[~normal] <= 2.0 ** -10 + 1e-9)


def test_int8_rows_exact_scale_and_half_step_error():
    g = np.random.default_rng(1)
    r = O.to_f32(g.standard_normal((4, 32)))
    r[1] = 0.0
    codes, s = R.int8_encode(r)
    dec = R.int8_decode(codes, s)
    assert np.all(dec[1] == 0) and np.all(np.abs(codes.astype(int)) <= 127)
    for i in (0, 2, 3):
        j = np.argmax(np.abs(r[i]))
        assert abs(int(codes[i, j])) == 127
        assert np.all(np.abs(dec[i] - r[i]) <= s[i] / 2 * (1 + 1e-6) + 1e-12)
    # ties at half a step go to the even integer: 2.5 s -> 2, 3.5 s -> 4
    row = np.zeros((1, 4))
    row[0] = [127.0, 2.5, 3.5, -2.5]
    c, s1 = R.int8_encode(row)
    assert s1[0] == 1.0 and list(c[0]) == [127, 2, 4, -2]


def test_mxfp4_power_of_two_scale_on_worked_blocks():
    """OCP rule X = 2^(floor(log2 amax) - 2): a block whose largest element is 6
    keeps X = 1 and 6 exactly; largest 1.0 gives X = 1/4 and code 4 (value 1.0);
    largest 7 gives X = 1 and saturates at 6; an all-zero block stays zero."""
    b = np.zeros((4, 32))
    b[0, 0], b[0, 1] = 6.0, 1.5
    b[1, 0], b[1, 1] = 1.0, 0.25
    b[2, 0] = 7.0
    codes, e = R.mxfp4_encode(b)
    dec = R.mxfp4_decode(codes, e)
    assert list(e[:, 0]) == [0, -2, 0, 0]
    assert dec[0, 0] == 6.0 and dec[0, 1] == 1.5
    assert dec[1, 0] == 1.0 and dec[1, 1] == 0.25
    assert dec[2, 0] == 6.0
    assert np.all(dec[3] == 0) and np.all(codes[3] == 0)


def test_mxfp4_grid_and_range():
    g = np.random.default_rng(2)
    r = O.to_f32(g.standard_normal((3, 128)) * 3.0)
    codes, e = R.mxfp4_encode(r)
    dec = R.mxfp4_decode(codes, e).reshape(3, 4, 32)
    X = np.power(2.0, e)[..., None]
    q = dec / X
    assert np.all(np.isin(np.abs(q), O.E2M1_VALUES))
    amax = np.max(np.abs(r.reshape(3, 4, 32)), axis=-1)
    ratio = amax / np.power(2.0, e)
    assert np.all((ratio >= 4) & (ratio < 8))


def test_int2_ternary():
    r = np.array([[1.0, 0.6, 0.5, -0.51, 0.2, -1.0, 0.0, 0.49]])
    codes, s = R.int2_encode(r)
    assert s[0] == 1.0 and list(codes[0]) == [1, 1, 0, -1, 0, -1, 0, 0]
    assert np.array_equal(R.int2_decode(codes, s)[0], [1.0, 1.0, 0, -1.0, 0, -1.0, 0, 0])


def _window_states(seed, d, scale):
    g = np.random.default_rng(seed)
    centers = g.standard_normal((8, d)) * scale
    H = O.to_f32(centers[g.integers(0, 8, 96)] + g.standard_normal((96, d)))
    labels, z, s, A, gap = O.spherical_kmeans(H, 8, 10, O.kmeans_init(0, 0, 0, 0, 96, 8))
    return H, A, labels


@pytest.mark.parametrize("seed,d,scale", [(0, 512, 2.0), (1, 1024, 0.5), (2, 4096, 5.0)])
def test_table11_ordering_on_clustered_window_states(seed, d, scale):
    """Reconstruction error of the window states under each format (Table 11):
    binary16 best; the 8-bit residual formats below NVFP4 residuals; NVFP4
    residuals below MXFP4 residuals (16-element groups with an E4M3 scale against
    32-element blocks with a power-of-two scale) and below NVFP4 of the raw
    states (the paper's point for residuals); ternary last.
    Storage per element follows the format (NVFP4 0.5625 B)."""
    H, A, lab = _window_states(seed, d, scale)
    err, size = {}, {}
    for f in ("fp16", "fp8", "int8", "mxfp4", "int2", "nvfp4"):
        hp, size[f] = R.reconstruct(H, A, lab, f)
        err[f] = np.linalg.norm(hp - H) / np.linalg.norm(H)
    hp, _ = R.reconstruct(H, A, lab, "nvfp4", residual=False)
    err["nvfp4_plain"] = np.linalg.norm(hp - H) / np.linalg.norm(H)
    assert err["fp16"] < min(err["fp8"], err["int8"])
    assert max(err["fp8"], err["int8"]) < err["nvfp4"] < err["mxfp4"] < err["int2"]
    assert err["nvfp4"] < err["nvfp4_plain"] < err["int2"]
    assert math.isclose(size["nvfp4"], 0.5625) and math.isclose(size["mxfp4"], 0.53125)
    assert size["fp16"] == 2.0 and size["fp8"] == size["int8"] == 1.0 + 4.0 / d


def test_mxfp4_scale_exponent_stays_in_the_e8m0_range():
    """OCP MX scales are E8M0 bytes, 2^-127 .. 2^127: a block whose maximum is
    below 2^-125 keeps the smallest scale 2^-127 (its elements then round to 0
    or small codes), and the stored exponent never leaves the range."""
    r = np.zeros((1, 64))
    r[0, :32] = 2.0 ** -140 * np.arange(1, 33)      # block 0: amax = 2^-135
    r[0, 32:] = 2.0 ** 100 * np.linspace(-1, 1, 32)  # block 1: amax = 2^100
    codes, e = R.mxfp4_encode(O.to_f32(r))
    assert e[0, 0] == -127 and e[0, 1] == 98
    assert np.all(codes[0, :32] == 0)  # 2^-135..2^-130 over 2^-127 is below 0.25
    dec = R.mxfp4_decode(codes, e)
    assert np.all(np.isfinite(dec)) and np.all(dec[0, :32] == 0)
