"""Pins of the oracle's decoder layer (paper: "Polestar: Drift-Aware Cache
Calibration and Token Commitment for Efficient Inference of Diffusion LLMs",
§2 Eq. 3 -- the masked-diffusion transformer whose K/V cache Polestar
calibrates; the LLaDA / Dream layer: RMSNorm, Q/K/V, rotary embedding,
bidirectional attention, output projection + residual, RMSNorm, SwiGLU FFN +
residual).

The reference here is a per-element loop over plain Python floats, written from
the definitions of each operation and sharing nothing with the oracle's
vectorised code.  The two RMSNorm gains are distinct and non-unit and the
gate/up matrices differ, so swapping the norms, applying a gain twice or not at
all, or exchanging gate and up inside the SiLU cannot pass."""
import math

import numpy as np
import pytest

from drift_aware_kv_gb300 import synth
from oracle import polestar_oracle as O

torch = pytest.importorskip("torch")


def _naive_layer(h, W, pos, H, Hkv, dh, eps, base):
    """One decoder layer by explicit loops (float64 Python arithmetic)."""
    n, d = len(h), len(h[0])
    half = dh // 2

    def rms(x, g):
        ms = sum(v * v for v in x) / len(x)
        r = 1.0 / math.sqrt(ms + eps)
        return [x[i] * r * g[i] for i in range(len(x))]

    def matvec(M, x):  # M [out][in]
        return [sum(M[o][i] * x[i] for i in range(len(x))) for o in range(len(M))]

    def rotate(vec, p):  # rotate-half rotary: pairs (i, i + dh/2) of every head
        out = list(vec)
        for hh in range(len(vec) // dh):
            for i in range(half):
                theta = p * base ** (-2.0 * i / dh)
                a, b = vec[hh * dh + i], vec[hh * dh + i + half]
                out[hh * dh + i] = a * math.cos(theta) - b * math.sin(theta)
                out[hh * dh + i + half] = b * math.cos(theta) + a * math.sin(theta)
        return out

    xs = [rms(h[r], W["attn_norm"]) for r in range(n)]
    Q = [rotate(matvec(W["wq"], xs[r]), pos[r]) for r in range(n)]
    Kk = [rotate(matvec(W["wk"], xs[r]), pos[r]) for r in range(n)]
    V = [matvec(W["wv"], xs[r]) for r in range(n)]
    out = []
    for r in range(n):
        attn = []
        for hh in range(H):
            g = hh // (H // Hkv)
            sc = [sum(Q[r][hh * dh + i] * Kk[j][g * dh + i] for i in range(dh)) / math.sqrt(dh) for j in range(n)]
            m = max(sc)
            e = [math.exp(s - m) for s in sc]
            z = sum(e)
            for i in range(dh):
                attn.append(sum(e[j] / z * V[j][g * dh + i] for j in range(n)))
        h1 = [h[r][i] + v for i, v in enumerate(matvec(W["wo"], attn))]
        y = rms(h1, W["ffn_norm"])
        gt, up = matvec(W["w_gate"], y), matvec(W["w_up"], y)
        act = [gt[f] / (1.0 + math.exp(-gt[f])) * up[f] for f in range(len(gt))]
        out.append([h1[i] + v for i, v in enumerate(matvec(W["w_down"], act))])
    return out


def _tiny():
    cfg = synth.WORKLOADS["tiny_l1_d256_fp32"].replace(d_model=16, n_heads=4, n_kv_heads=2, head_dim=4,
                                                       ffn_dim=24, prompt_len=4, gen_len=2, norm_gain_std=0.4)
    W = O.weights_to_numpy(synth.make_weights(cfg))[0]
    # weights at a scale where every term of the layer matters
    g = np.random.default_rng(3)
    for k in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"):
        W[k] = W[k] * 15.0 + 0.05 * g.standard_normal(W[k].shape)
    return cfg, W


def test_synth_norm_gains_are_distinct_and_non_unit():
    cfg, W = _tiny()
    a, f = W["attn_norm"], W["ffn_norm"]
    assert np.all(a != 1.0) and np.all(f != 1.0) and not np.allclose(a, f)


def test_oracle_decoder_layer_equals_per_element_loops():
    """qkv -> attend -> post of the oracle over a 6-position sequence (grouped
    query heads 4:2, rotary at absolute positions) equals the loop reference."""
    cfg, W = _tiny()
    orc = O.PolestarOracle(cfg, [W])
    g = np.random.default_rng(7)
    h = g.standard_normal((6, cfg.d_model)) * 1.5
    pos = np.array([0, 1, 2, 3, 9, 17])
    q, k, v = orc.qkv(0, h, pos)
    kv = np.stack([k, v], axis=1)
    o, _, _ = orc.attend(q, kv)
    got = orc.post(0, h, o)
    ref = np.array(_naive_layer(h.tolist(), {k_: W[k_].tolist() for k_ in W}, pos.tolist(), cfg.n_heads,
                                cfg.n_kv_heads, cfg.head_dim, cfg.rms_eps, cfg.rope_base))
    assert np.allclose(got, ref, rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("mutation", ["swap_norms", "swap_gate_up", "unit_ffn_norm"])
def test_layer_pin_catches_plausible_mistakes(mutation):
    """The loop reference distinguishes the mistakes it is meant to catch: each
    mutated weight set changes the layer's output well beyond the tolerance."""
    cfg, W = _tiny()
    M = dict(W)
    if mutation == "swap_norms":
        M["attn_norm"], M["ffn_norm"] = W["ffn_norm"], W["attn_norm"]
    elif mutation == "swap_gate_up":
        M["w_gate"], M["w_up"] = W["w_up"], W["w_gate"]
    else:
        M["ffn_norm"] = np.ones_like(W["ffn_norm"])
    g = np.random.default_rng(7)
    h = g.standard_normal((6, cfg.d_model)) * 1.5
    pos = [0, 1, 2, 3, 9, 17]
    a = np.array(_naive_layer(h.tolist(), {k: W[k].tolist() for k in W}, pos, cfg.n_heads, cfg.n_kv_heads,
                              cfg.head_dim, cfg.rms_eps, cfg.rope_base))
    b = np.array(_naive_layer(h.tolist(), {k: M[k].tolist() for k in M}, pos, cfg.n_heads, cfg.n_kv_heads,
                              cfg.head_dim, cfg.rms_eps, cfg.rope_base))
    assert np.max(np.abs(a - b)) > 1e-3 * np.max(np.abs(a))


def test_oracle_silu_equals_torch():
    x = np.linspace(-30.0, 30.0, 2001)
    ref = torch.nn.functional.silu(torch.tensor(x, dtype=torch.float64)).numpy()
    assert np.allclose(O.silu(x), ref, rtol=1e-14, atol=1e-300)
