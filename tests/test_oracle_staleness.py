"""Pins of the oracle's KV-cache staleness (App. C.2 "KV-Cache Staleness Metric" of
"Polestar: Drift-Aware Cache Calibration and Token Commitment for Efficient
Inference of Diffusion LLMs") and of its full-sequence forward, plus the staleness
study on the oracle: Polestar's sparse refresh against no refresh within a block."""
import math

import numpy as np
import pytest

from drift_aware_kv_gb300 import synth
from oracle import polestar_oracle as O


def _rows(g, n, Hkv, dh):
    return g.standard_normal((n, 2, Hkv * dh))


def test_zero_on_itself_and_scale_invariant():
    g = np.random.default_rng(1)
    a = _rows(g, 7, 3, 16)
    assert np.all(np.abs(O.kv_staleness(a, a, 3, 16)) < 1e-15)
    assert np.all(np.abs(O.kv_staleness(a, 2.5 * a, 3, 16)) < 1e-15)


def test_two_on_the_negation_and_bounds():
    g = np.random.default_rng(2)
    a = _rows(g, 9, 2, 8)
    assert np.allclose(O.kv_staleness(a, -a, 2, 8), 2.0, atol=1e-15)
    E = O.kv_staleness(a, _rows(g, 9, 2, 8), 2, 8)
    assert np.all((E >= 0) & (E <= 2))


@pytest.mark.parametrize("which", [0, 1])
def test_rotation_in_one_head_closed_form(which):
    """One head of K (or of V) turned by theta, every other vector unchanged:
    the head average of that tensor is (cos(theta) + Hkv - 1) / Hkv and the other
    tensor's is 1, so E = (1 - cos(theta)) / (2 Hkv)."""
    Hkv, dh, theta = 3, 4, math.pi / 3
    a = np.zeros((1, 2, Hkv, dh))
    a[0, :, :, 2] = 1.0
    a[0, which, 1] = [1.0, 0.0, 0.0, 0.0]
    b = a.copy()
    b[0, which, 1] = [math.cos(theta), math.sin(theta), 0.0, 0.0]
    E = O.kv_staleness(a, b, Hkv, dh)
    assert E.shape == (1,)
    assert abs(E[0] - (1 - math.cos(theta)) / (2 * Hkv)) < 1e-15
    assert abs(E[0] - 1.0 / 12.0) < 1e-15


def test_orthogonal_and_zero_vectors():
    a = np.zeros((3, 2, 1, 8))
    b = np.zeros((3, 2, 1, 8))
    a[0, :, 0, 0] = 1.0
    b[0, :, 0, 1] = 1.0          # orthogonal K and V: E = 1
    a[1, :, 0, 3] = 2.0          # non-zero against zero: cos 0, E = 1
    # row 2: zero against zero everywhere: identical, E = 0
    E = O.kv_staleness(a, b, 1, 8)
    assert np.array_equal(E, [1.0, 1.0, 0.0])


def test_matches_scipy_cosine_distance_per_head():
    from scipy.spatial.distance import cosine
    g = np.random.default_rng(3)
    Hkv, dh = 4, 8
    a = _rows(g, 5, Hkv, dh)
    b = a + 0.3 * _rows(g, 5, Hkv, dh)
    E = O.kv_staleness(a, b, Hkv, dh)
    for r in range(5):
        d = [cosine(a[r, t, h * dh:(h + 1) * dh], b[r, t, h * dh:(h + 1) * dh])
             for t in range(2) for h in range(Hkv)]
        assert abs(E[r] - np.mean(d)) < 1e-12


def _oracle(cfg, **kw):
    W = O.weights_to_numpy(synth.make_weights(cfg))
    return O.PolestarOracle(cfg.replace(**kw) if kw else cfg, W)


def test_full_forward_equals_even_block_entry_and_has_zero_staleness():
    cfg = synth.WORKLOADS["tiny_l1_d256_fp32"].replace(n_layers=2)
    orc = _oracle(cfg)
    tr = synth.Trajectory(cfg)
    st = tr.next_step()
    x0 = st["x0"].double().numpy()
    orc.calibrate_step(x0, st["n_unmasked"], 0, True)
    ref = orc.full_forward_kv(x0[0])
    for l in range(cfg.n_layers):
        assert np.allclose(orc.seqs[0].kv[l], ref[l], rtol=1e-12, atol=1e-13)
        E = O.kv_staleness(orc.seqs[0].kv[l], ref[l], cfg.n_kv_heads, cfg.head_dim)
        assert np.all(np.abs(E) < 1e-12)


def _study(cfg, policy, steps):
    """Mean window staleness (per layer) over the within-block steps of a
    trajectory, for one cache policy: "polestar" (the method), "none" (no refresh
    between block entries) or "full" (full recompute every step: zero)."""
    kw = dict(tau_upd=10 ** 6) if policy == "none" else {}
    run_cfg = cfg.replace(**kw)
    W = O.weights_to_numpy(synth.make_weights(cfg))
    orc = O.PolestarOracle(run_cfg, W)
    ref = O.PolestarOracle(cfg, W)
    tr = synth.Trajectory(cfg)
    res = []
    outside0 = []
    for _ in range(steps):
        st = tr.next_step()
        if st is None:
            break
        x0 = st["x0"].to(synth.torch_dtype(cfg)).double().numpy()
        orc.calibrate_step(x0, st["n_unmasked"], st["block_index"], st["block_entry"])
        if policy == "full":
            orc.full_forward(x0)
        if st["block_entry"]:
            continue
        ref_kv = ref.full_forward_kv(x0[0])
        win = orc.window(st["block_index"])
        E = np.stack([O.kv_staleness(orc.seqs[0].kv[l], ref_kv[l], cfg.n_kv_heads, cfg.head_dim)
                      for l in range(cfg.n_layers)])
        res.append(E[:, win].mean(axis=1))
        if st["block_index"] % 2 == 0:  # after a full-sequence entry forward
            out = np.setdiff1d(np.arange(orc.N), win + list(range(*orc._span(st["block_index"]))))
            outside0.append(float(np.max(np.abs(E[0, out]))))
    return np.array(res), outside0


def test_study_polestar_is_fresher_than_no_refresh():
    """App. C.2 / Fig. 3: within a block the window K/V drift away from the full
    recompute.  Polestar's sparse refresh keeps them closer than reusing the
    block-entry cache; recomputing everything gives zero.  In a block entered
    with a full-sequence forward (even index), layer-0 K/V of positions outside
    the window and the block do not go stale: their inputs do not change."""
    cfg = synth.WORKLOADS["tiny_l1_d256_fp32"].replace(n_layers=2)
    pol, out_p = _study(cfg, "polestar", 12)
    none, out_n = _study(cfg, "none", 12)
    full, _ = _study(cfg, "full", 12)
    assert len(pol) >= 8 and pol.shape == none.shape
    assert np.all(np.abs(full) < 1e-12)
    assert max(out_p + out_n) < 1e-12
    assert np.all(none[-1] > 0)
    # over the whole run and at every layer, the refreshed cache is fresher
    assert np.all(pol.mean(axis=0) < none.mean(axis=0))


def test_study_refresh_budget_and_trigger_move_staleness_monotonically():
    """The two knobs of Polestar-Cache (Table 5): refreshing more clusters per layer
    (k) keeps the window fresher, and a higher refresh trigger tau_upd (fewer
    refreshes) lets it go staler; tau_upd out of reach is block-wise reuse."""
    base = synth.WORKLOADS["tiny_l1_d256_fp32"].replace(n_layers=2)
    by_k = [float(_study(base.replace(topk=k), "polestar", 12)[0].mean()) for k in (1, 4, 8)]
    by_tau = [float(_study(base.replace(tau_upd=t), "polestar", 12)[0].mean()) for t in (3, 4, 10 ** 6)]
    assert by_k[0] > by_k[1] > by_k[2] > 0
    assert by_tau[0] < by_tau[1] < by_tau[2]
