"""Pins of the CPU oracle against things other than itself: library routines,
published test vectors, closed forms, invariants and brute force.

Citations name the paper "Polestar: Drift-Aware Cache Calibration and Token
Commitment for Efficient Inference of Diffusion LLMs" by section / equation."""
import math

import numpy as np
import pytest
import scipy.special
import torch

from oracle import polestar_oracle as O


def rng(seed=0):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- number formats
def test_bf16_rounding_matches_torch():
    x = rng(1).standard_normal(20000) * np.exp(rng(2).uniform(-20, 20, 20000))
    ref = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    assert np.array_equal(O.to_bf16(x), ref)


def test_e4m3_decode_matches_torch_table():
    """Every FP8 E4M3 byte decodes like torch.float8_e4m3fn (OCP FP8 format)."""
    codes = np.arange(256)
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = O.e4m3_value(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_e4m3_round_matches_torch_rne():
    """Scale rounding (App. C.3: FP8 E4M3 group scale) equals torch's RNE cast,
    including exact midpoints and the subnormal range; bytes round-trip."""
    table = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mids = (table[:-1] + table[1:]) / 2
    v = np.concatenate([table, mids, rng(3).uniform(0, 460, 5000),
                        np.exp(rng(4).uniform(-14, 6, 5000))])
    v = v[v < 464].astype(np.float32).astype(np.float64)
    ref = torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn)
    val, byte, _ = O.e4m3_round(v)
    assert np.array_equal(val, ref.double().numpy())
    assert np.array_equal(byte, ref.view(torch.uint8).numpy())
    assert np.array_equal(O.e4m3_value(byte), val)


def test_e4m3_saturates():
    val, byte, _ = O.e4m3_round(np.array([448.0, 463.0, 1e6]))
    assert np.all(val == 448.0) and np.all(byte == 0x7E)


def _e2m1_from_bits(code):
    """E2M1 decode from its bit fields (1 sign, 2 exponent bits with bias 1,
    1 mantissa bit; exponent 0 is subnormal)."""
    s = -1.0 if code & 8 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    return s * (m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1))


def test_e2m1_values_match_bitfield_definition():
    for c in range(16):
        assert O.e2m1_value(c) == _e2m1_from_bits(c)


def test_e2m1_rounding_nearest_even_and_saturating():
    grid = np.array([_e2m1_from_bits(c) for c in range(8)])
    x = np.concatenate([rng(5).uniform(-7, 7, 20000), (grid[:-1] + grid[1:]) / 2,
                        -(grid[:-1] + grid[1:]) / 2])
    codes, _ = O.e2m1_round(x)
    dec = O.e2m1_value(codes)
    xs = np.clip(x, -6, 6)
    # brute force: the decoded value is a nearest grid point
    best = np.min(np.abs(np.abs(xs)[:, None] - grid[None, :]), axis=1)
    assert np.allclose(np.abs(np.abs(xs) - np.abs(dec)), best, atol=0, rtol=0)
    # ties go to the even code (round-half-even on the code index)
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for t, want in ties.items():
        c, m = O.e2m1_round(np.array([t, -t]))
        assert list(O.e2m1_value(c)) == [want, -want]
        assert np.all(m == 0)


def test_nvfp4_grid_membership_and_error_bound():
    """Decoded residuals lie on {0,.5,1,1.5,2,3,4,6} x scale; per-element error is at
    most half the local grid step x scale (App. C.3 NVFP4)."""
    r = rng(6).standard_normal((64, 256)) * rng(7).uniform(0.01, 3, (64, 1))
    r = O.to_f32(r)
    codes, sb, _ = O.nvfp4_encode(r)
    s = O.e4m3_value(sb).reshape(64, 16, 1)
    dec = O.nvfp4_decode(codes, sb).reshape(64, 16, 16)
    ratio = dec / s
    grid = np.concatenate([O.E2M1_VALUES, -O.E2M1_VALUES])
    assert np.all(np.min(np.abs(ratio[..., None] - grid), axis=-1) == 0)
    steps = np.array([0.5, 0.5, 0.5, 0.5, 1.0, 1.0, 2.0, 2.0])
    x = (r.reshape(64, 16, 16) / s)
    idx = np.searchsorted(O.E2M1_VALUES, np.minimum(np.abs(x), 6.0))
    bound = steps[np.minimum(idx, 7)] / 2 * s
    err = np.abs(r.reshape(64, 16, 16) - dec)
    amax_over = np.abs(x) > 6.0
    assert np.all((err <= bound * (1 + 1e-6)) | amax_over)


def test_nvfp4_encode_of_decoded_is_identity():
    """App. C.3: a group's scale is E4M3(amax / 6), so its largest element always
    encodes to 6 (amax / s lies within E4M3's relative step of 6); re-encoding the
    decoded group therefore finds the same scale and the same codes."""
    r = O.to_f32(rng(10).standard_normal((32, 128)) * rng(11).uniform(1e-3, 50, (32, 1)))
    codes, sb, _ = O.nvfp4_encode(r)
    assert np.all(np.max(codes.reshape(32, 8, 16) & 7, axis=-1) == 7)  # index 7 is magnitude 6
    c2, s2, _ = O.nvfp4_encode(O.nvfp4_decode(codes, sb))
    assert np.array_equal(c2, codes) and np.array_equal(s2, sb)


def test_nvfp4_zero_group_and_sign():
    r = np.zeros((1, 32))
    r[0, 16:] = rng(8).standard_normal(16)
    codes, sb, _ = O.nvfp4_encode(r)
    assert np.all(codes[0, :16] == 0) and sb[0, 0] == 0
    assert np.all((codes[0, 16:] >= 8) == (r[0, 16:] < 0) | (codes[0, 16:] == 8))


def test_residual_nvfp4_beats_plain_nvfp4():
    """Table 11's ordering: residual NVFP4 reconstructs clustered hidden states with a
    lower error than plain NVFP4 of the same rows."""
    g = rng(9)
    centers = g.standard_normal((8, 512)) * 3
    lab = g.integers(0, 8, 96)
    H = O.to_f32(centers[lab] + 0.3 * g.standard_normal((96, 512)))
    A = O.to_f32(np.stack([H[lab == c].mean(0) for c in range(8)]))
    c1, s1, _ = O.nvfp4_encode(O.to_f32(H - A[lab]))
    rec_res = O.nvfp4_decode(c1, s1) + A[lab]
    c2, s2, _ = O.nvfp4_encode(H)
    rec_plain = O.nvfp4_decode(c2, s2)
    e_res = np.sqrt(np.mean((rec_res - H) ** 2))
    e_plain = np.sqrt(np.mean((rec_plain - H) ** 2))
    assert e_res < 0.5 * e_plain


# ---------------------------------------------------------------- seeded init
def test_splitmix64_published_vector():
    """splitmix64 reference implementation, state 0: first three outputs."""
    g = O.splitmix64_stream(0)
    assert [next(g) for _ in range(3)] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                           0x06C45D188009454F]


def test_kmeans_init_is_a_distinct_subset():
    for seq in range(3):
        for layer in range(4):
            idx = O.kmeans_init(7, seq, 2, layer, 96, 8)
            assert len(set(idx)) == 8 and all(0 <= i < 96 for i in idx)
    assert O.kmeans_init(7, 0, 2, 0, 96, 8) != O.kmeans_init(7, 0, 2, 1, 96, 8)


# ---------------------------------------------------------------- model pieces
def test_rmsnorm_matches_torch():
    x = rng(10).standard_normal((5, 64))
    g = rng(11).uniform(0.5, 1.5, 64)
    ref = torch.nn.functional.rms_norm(torch.tensor(x), (64,), torch.tensor(g), eps=1e-6)
    assert np.allclose(O.rmsnorm(x, g, 1e-6), ref.numpy(), rtol=1e-13, atol=1e-13)


def test_rope_equals_complex_rotation():
    """Rotate-half rotary embedding = multiplying z_i = x_i + i x_{i+dh/2} by
    exp(i p base^(-2i/dh))."""
    x = rng(12).standard_normal((7, 3, 16))
    pos = np.array([0, 1, 5, 17, 100, 511, 2047])
    got = O.rope(x, pos, 10000.0)
    z = x[..., :8] + 1j * x[..., 8:]
    theta = 10000.0 ** (-np.arange(8) / 8.0)
    zr = z * np.exp(1j * pos[:, None, None] * theta[None, None, :])
    assert np.allclose(got, np.concatenate([zr.real, zr.imag], -1), atol=1e-12)


def _tiny_cfg(**kw):
    from drift_aware_kv_gb300.synth import WORKLOADS
    return WORKLOADS["tiny_l1_d256_fp32"].replace(**kw)


def test_attention_matches_torch_sdpa_gqa():
    cfg = _tiny_cfg(n_heads=4, n_kv_heads=2, head_dim=16, d_model=64)
    orc = O.PolestarOracle.__new__(O.PolestarOracle)
    orc.cfg, orc.bf16 = cfg, False
    q = rng(13).standard_normal((5, 4, 16))
    kv = rng(14).standard_normal((9, 2, 2, 16))
    out, s, lse = orc.attend(q, kv)
    qt = torch.tensor(q).transpose(0, 1)  # [H, R, dh]
    kt = torch.tensor(kv[:, 0]).transpose(0, 1).repeat_interleave(2, 0)
    vt = torch.tensor(kv[:, 1]).transpose(0, 1).repeat_interleave(2, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)
    assert np.allclose(out, ref.transpose(0, 1).reshape(5, -1).numpy(), atol=1e-12)
    p = np.exp(s - lse[..., None])
    assert np.allclose(p.sum(-1), 1.0, atol=1e-12)


def test_attention_first_order_drift_of_proposition_1():
    """App. B, Proposition 1: when position s's layer input moves from x_s to
    x_s + eta (every other input fixed), the attention output of a position i
    that attends to s changes by a_is W_V eta + a_is (q_i^T W_K eta / sqrt(dh))
    (v_s - o_i) to first order.  The oracle's attention, fed keys W_K x and values
    W_V x, must follow that derivative: the finite-difference remainder shrinks
    like eps^2 (halving eps quarters it)."""
    dh, d, N = 8, 12, 7
    cfg = _tiny_cfg(n_heads=1, n_kv_heads=1, head_dim=dh, d_model=d)
    orc = O.PolestarOracle.__new__(O.PolestarOracle)
    orc.cfg, orc.bf16 = cfg, False
    g = rng(21)
    x = g.standard_normal((N, d))
    WK, WV = g.standard_normal((dh, d)) * 0.4, g.standard_normal((dh, d))
    q = g.standard_normal((N, 1, dh))
    eta = g.standard_normal(d)
    s_pos = 3

    def outputs(xx):
        kv = np.stack([xx @ WK.T, xx @ WV.T], axis=1)[:, :, None, :]  # [N, 2, 1, dh]
        o, sc, lse = orc.attend(q, kv)
        return o, np.exp(sc - lse[..., None])[:, 0, :]  # o [N, dh], a [N, N]

    o0, a = outputs(x)
    v_s = WV @ x[s_pos]
    rem = []
    for eps in (1e-3, 5e-4):
        xe = x.copy()
        xe[s_pos] += eps * eta
        o1, _ = outputs(xe)
        for i in range(N):
            if i == s_pos:
                continue
            lin = a[i, s_pos] * (WV @ eta) + a[i, s_pos] * (q[i, 0] @ (WK @ eta)) / math.sqrt(dh) * (v_s - o0[i])
            err = np.linalg.norm((o1[i] - o0[i]) - eps * lin)
            # a dropped or mis-scaled first-order term would leave an O(eps) residue
            assert err < 5.0 * eps * eps
            rem.append(err)
    half = len(rem) // 2
    ratio = np.array(rem[half:]) / np.maximum(np.array(rem[:half]), 1e-300)
    assert np.all((ratio > 0.2) & (ratio < 0.3))  # second-order remainder: about 1/4


def test_kl_closed_forms_and_scipy():
    """KL of Eq. 4: zero for identical scores, non-negative, equal to
    scipy.special.rel_entr, and Pinsker's bound ||p-q||_1 <= sqrt(2 KL) (App. B,
    Proposition 2)."""
    s = rng(15).standard_normal((6, 50)) * 2
    sp = s + rng(16).standard_normal((6, 50)) * 0.3
    lse, lsp = O.logsumexp(s), O.logsumexp(sp)
    assert np.all(O.kl_div(s, lse, s, lse) == 0.0)
    kl = O.kl_div(s, lse, sp, lsp)
    p = scipy.special.softmax(s, axis=-1)
    q = scipy.special.softmax(sp, axis=-1)
    ref = scipy.special.rel_entr(p, q).sum(-1)
    assert np.allclose(kl, ref, rtol=1e-12, atol=1e-15)
    assert np.all(kl >= 0)
    assert np.all(np.abs(p - q).sum(-1) <= np.sqrt(2 * kl) + 1e-12)


def test_topk_equals_full_sort():
    g = rng(17)
    for _ in range(200):
        D = g.integers(0, 4, 8).astype(float) * 0.1  # many ties
        ids, _ = O.topk_clusters(D, 4)
        ref = list(np.argsort(-D, kind="stable")[:4])
        assert ids == ref


def test_spherical_kmeans_recovers_planted_clusters():
    g = rng(18)
    dirs = np.linalg.qr(g.standard_normal((64, 8)))[0].T  # 8 orthonormal directions
    lab = np.repeat(np.arange(8), 12)
    H = dirs[lab] * g.uniform(1, 5, (96, 1)) + 0.02 * g.standard_normal((96, 64))
    init = [int(np.nonzero(lab == c)[0][0]) for c in range(8)]
    labels, z, s, A, gap = O.spherical_kmeans(H, 8, 10, init)
    assert np.array_equal(labels, lab)
    assert np.allclose(np.linalg.norm(z, axis=1), 1.0, atol=1e-12)
    for c in range(8):
        assert np.allclose(A[c], H[lab == c].mean(0), rtol=1e-6)
    assert gap > 0.5


def test_spherical_kmeans_fixed_point_and_monotone():
    """Labels are the brute-force argmax cosine against the previous update's
    centroids, and the objective sum <x, z_label> never decreases."""
    g = rng(19)
    H = g.standard_normal((40, 12))
    init = O.kmeans_init(3, 0, 0, 0, 40, 4)
    X = H / np.linalg.norm(H, axis=1, keepdims=True)
    objs = []
    for it in range(1, 11):
        labels, z, _, _, _ = O.spherical_kmeans(H, 4, it, init)
        objs.append(sum(float(X[i] @ z[labels[i]]) for i in range(40)))
        if it > 1:
            best = [max(range(4), key=lambda c: (float(X[i] @ zprev[c]), -c))
                    for i in range(40)]
            assert list(labels) == best
        zprev = z
    assert all(b >= a - 1e-12 for a, b in zip(objs, objs[1:]))


def test_kmeans_brute_force_tiny():
    """6 points, K = 2: exhaustive search over all 2^6 labellings finds every Lloyd
    fixed point (each point's best centroid, among the normalised member sums of
    that labelling, is its own cluster); the oracle's converged labels are one."""
    g = rng(20)
    H = g.standard_normal((6, 5))
    X = H / np.linalg.norm(H, axis=1, keepdims=True)
    labels, z, _, _, _ = O.spherical_kmeans(H, 2, 10, [0, 1])

    def is_fixed_point(lab):
        if len(set(lab.tolist())) < 2:
            return False
        cents = [X[lab == c].sum(0) for c in range(2)]
        cents = [c / np.linalg.norm(c) for c in cents]
        for i in range(6):
            cos = [float(X[i] @ cents[c]) for c in range(2)]
            want = 0 if cos[0] >= cos[1] else 1
            if want != lab[i]:
                return False
        return True

    fixed = [m for m in range(64)
             if is_fixed_point(np.array([(m >> i) & 1 for i in range(6)]))]
    got = sum(int(labels[i]) << i for i in range(6))
    assert fixed and got in fixed


# ---------------------------------------------------------------- commit gate
def test_gate_worked_values():
    """tau_d = alpha (tau_s - c)^2: c = 0.8 gives 0.1 at alpha = 10, tau_s = 0.9, and
    tau_d -> 0 as c -> tau_s (§4.2)."""
    assert abs(O.drift_threshold(0.8, 0.9, 10.0) - 0.1) < 1e-12
    assert O.drift_threshold(0.9, 0.9, 10.0) == 0.0
    assert O.drift_threshold(0.9 - 1e-4, 0.9, 10.0) < 1e-6


def test_confidence_matches_generator_target():
    from drift_aware_kv_gb300.synth import Trajectory
    tr = Trajectory(_tiny_cfg())
    step = tr.next_step()
    conf = O.confidence(step["logits"][0].numpy())
    assert np.allclose(conf, step["conf_target"][0].numpy(), rtol=1e-5)
