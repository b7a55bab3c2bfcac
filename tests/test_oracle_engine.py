"""Engine-level pins of the CPU oracle (paper: "Polestar: Drift-Aware Cache
Calibration and Token Commitment for Efficient Inference of Diffusion LLMs")."""
import numpy as np
import pytest

from drift_aware_kv_gb300 import synth
from oracle import polestar_oracle as O


def _run(cfg, exact_cache=False, steps=None):
    W = O.weights_to_numpy(synth.make_weights(cfg))
    orc = O.PolestarOracle(cfg, W, exact_cache=exact_cache)
    tr = synth.Trajectory(cfg)
    out = []
    while True:
        st = tr.next_step()
        if st is None or (steps is not None and len(out) >= steps):
            break
        x0 = st["x0"].to(synth.torch_dtype(cfg)).double().numpy()
        rec = orc.calibrate_step(x0, st["n_unmasked"], st["block_index"], st["block_entry"])
        com = orc.commit(st["logits"].numpy(), st["masked"].numpy())
        out.append((st, rec, com))
    return orc, out


def test_sparse_refresh_with_all_clusters_equals_block_entry_forward():
    """Closed-form special case of §4.1: when the refresh fires, every cluster is
    selected (k = K) and the cached hidden states are exact, the sparse layer-wise
    update of the window equals a forward of window + active block over the cached
    context, i.e. the block-entry forward at an odd block (Algorithm 1, block-entry context)."""
    cfg = synth.WORKLOADS["tiny_l1_d256_fp32"].replace(n_layers=3, topk=8, tau_upd=0)
    W = O.weights_to_numpy(synth.make_weights(cfg))
    tr = synth.Trajectory(cfg)
    s0 = tr.next_step()
    # move to block 1 (odd) directly: fresh state for both engines
    x0 = s0["x0"].double().numpy()
    a = O.PolestarOracle(cfg, W, exact_cache=True)
    b = O.PolestarOracle(cfg, W, exact_cache=True)
    a.calibrate_step(x0, [0], 0, True)  # full forward fills every position
    a.calibrate_step(x0, [0], 1, True)
    b.calibrate_step(x0, [0], 0, True)
    x1 = x0.copy()
    g = np.random.default_rng(0)
    win = a.window(1)
    x1[0, win] += 0.3 * g.standard_normal((len(win), cfg.d_model))
    x1[0, 96:100] = g.standard_normal((4, cfg.d_model))
    rec = a.calibrate_step(x1, [5], 1, False)[0]
    assert rec["fire"] and all(len(t) == 8 for t in rec["topk"])
    b.calibrate_step(x1, [0], 1, True)
    pos = sorted(set(win) | set(range(96, 128)))
    for l in range(cfg.n_layers):
        assert np.allclose(a.seqs[0].kv[l][pos], b.seqs[0].kv[l][pos], rtol=1e-10, atol=1e-12)
        assert np.allclose(a.exact_H[0][l], b.exact_H[0][l], rtol=1e-10, atol=1e-12)


def test_tiny_trajectory_invariants():
    """Whole-trajectory sanity on the fp32 single-layer workload: drift is
    non-negative, selected rows are exactly the members of the top-k clusters,
    committed rows were masked, and tau_d = alpha (tau_s - c)^2."""
    cfg = synth.WORKLOADS["tiny_l1_d256_fp32"]
    orc, out = _run(cfg)
    assert len(out) == 16
    fired = 0
    for st, recs, coms in out:
        for si in range(cfg.batch):
            rec, com = recs[si], coms[si]
            if not st["block_entry"]:
                assert np.all(rec["delta"] >= -1e-15)
                if rec["fire"]:
                    fired += 1
                    for D, ids, sel in zip(rec["D"], rec["topk"], rec["sel"]):
                        assert np.all(D >= -1e-15)
                        assert len(set(ids)) == cfg.topk
                assert np.allclose(com["tau_d"][:32], 10 * (0.9 - com["conf"][:32]) ** 2)
            start = cfg.prompt_len + st["block_index"] * cfg.block
            m = st["masked"][si].numpy()
            for j in np.nonzero(com["commit"])[0]:
                assert m[start + j]
    assert fired >= 2


@pytest.mark.parametrize("name", ["mini_l2_d512_bf16", "mini_gqa_l2_d448_bf16"])
def test_mini_bf16_runs(name):
    cfg = synth.WORKLOADS[name].replace(n_steps=6)
    orc, out = _run(cfg)
    assert len(out) == 6
    for st, recs, coms in out:
        for rec in recs:
            if "act_out" in rec:
                assert np.all(np.isfinite(rec["act_out"]))


def test_incremental_centroid_update_closed_form_at_layer_0():
    """§4.1 "Compute Update Packets" with the readings R5/R6: at layer 0 the update
    packet of every window row is the caller's current input, and a refreshing
    step patches all of them, so with an exact cache the member sums become
    s_c = sum over members of x_i / |x_i| of this step's inputs (the K-means sums
    at block entry minus the old directions plus the new), and z_c = s_c / |s_c|."""
    cfg = synth.WORKLOADS["tiny_l1_d256_fp32"].replace(n_layers=2)
    W = O.weights_to_numpy(synth.make_weights(cfg))
    orc = O.PolestarOracle(cfg, W, exact_cache=True)
    tr = synth.Trajectory(cfg)
    checked = 0
    for _ in range(10):
        st = tr.next_step()
        x0 = st["x0"].double().numpy()
        rec = orc.calibrate_step(x0, st["n_unmasked"], st["block_index"], st["block_entry"])[0]
        if st["block_entry"] or not rec["fire"]:
            continue
        s0 = orc.seqs[0]
        X = x0[0][orc.window(st["block_index"])]
        Xh = X / np.linalg.norm(X, axis=1, keepdims=True)
        for c in range(cfg.K):
            mem = s0.labels[0] == c
            if not mem.any():
                continue
            assert np.allclose(s0.s[0][c], Xh[mem].sum(0), rtol=1e-10, atol=1e-10)
            zc = Xh[mem].sum(0)
            assert np.allclose(s0.z[0][c], zc / np.linalg.norm(zc), rtol=1e-10, atol=1e-12)
        checked += 1
    assert checked >= 3


def test_proxy_query_of_a_token_at_position_0_equals_its_query():
    """§4.1 "Measuring Drift" with reading R2: a proxy query is W_q RMSNorm(z_c)
    with no rotary (a centroid has no position).  The rotary of position 0 is the
    identity, so a proxy built from the input of the token at position 0 scores
    every key exactly as that token's own query does."""
    cfg = synth.WORKLOADS["tiny_l1_d256_fp32"]
    W = O.weights_to_numpy(synth.make_weights(cfg))
    orc = O.PolestarOracle(cfg, W)
    tr = synth.Trajectory(cfg)
    st = tr.next_step()
    x0 = st["x0"].double().numpy()
    orc.calibrate_step(x0, st["n_unmasked"], 0, True)
    kv = orc.seqs[0].kv[0]
    h0 = x0[0, :1]
    s_proxy, lse_proxy = orc.proxy_scores(0, h0, kv)
    q, _, _ = orc.qkv(0, h0, np.array([0]))
    s_tok = orc.scores(q, kv)
    assert np.allclose(s_proxy, s_tok, rtol=1e-12, atol=1e-12)
    # any other position rotates the query: scores differ
    q7, _, _ = orc.qkv(0, h0, np.array([7]))
    assert not np.allclose(orc.scores(q7, kv), s_tok, atol=1e-6)


def _oracle_fires(tau_upd, counts_per_block):
    """Refresh decisions of the oracle engine itself over hand-chosen unmasked
    counts: each entry of counts_per_block is one block (a block entry, then one
    within-block step per count).  The inputs do not change between steps; only
    the counts drive the trigger."""
    cfg = synth.WORKLOADS["tiny_l1_d256_fp32"].replace(tau_upd=tau_upd)
    W = O.weights_to_numpy(synth.make_weights(cfg))
    orc = O.PolestarOracle(cfg, W)
    x0 = synth.Trajectory(cfg).next_step()["x0"].double().numpy()
    out = []
    for b, counts in enumerate(counts_per_block):
        orc.calibrate_step(x0, [0], b, True)
        out.append([bool(orc.calibrate_step(x0, [n], b, False)[0]["fire"]) for n in counts])
    return out


@pytest.mark.parametrize("tau,counts,expected", [
    # §4.1 "Update Schedule": refresh once the tokens unmasked since the last
    # refresh exceed tau_upd (R10: this step's count included), then restart
    (3, [1, 1, 1, 1, 1, 1, 1, 1], [0, 0, 0, 1, 0, 0, 0, 1]),
    (3, [4, 0, 0, 5], [1, 0, 0, 1]),          # more than tau_upd in one step
    (3, [3, 0, 0, 0, 1], [0, 0, 0, 0, 1]),    # exactly tau_upd is not enough ("exceeds")
    (3, [2, 2, 2, 2], [0, 1, 0, 1]),
    (3, [0, 0, 0], [0, 0, 0]),                # nothing unmasked: never
    (0, [1, 0, 2, 0], [1, 0, 1, 0]),          # tau_upd = 0: every step that unmasks
    (5, [6, 3, 3, 5, 1], [1, 0, 1, 0, 1]),
])
def test_oracle_trigger_closed_form(tau, counts, expected):
    assert _oracle_fires(tau, [counts]) == [[bool(e) for e in expected]]


def test_oracle_trigger_restarts_at_block_entry():
    """A block entry rebuilds every cluster and proxy baseline, so the count
    since the last refresh restarts there: 3 tokens left over from block 0 do
    not add to block 1's first count of 1."""
    assert _oracle_fires(3, [[1, 1, 1], [1, 3]]) == [[False, False, False], [False, True]]
