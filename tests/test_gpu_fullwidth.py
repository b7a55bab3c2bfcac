"""Step-level lockstep parity at the real model widths (paper: "Polestar:
Drift-Aware Cache Calibration and Token Commitment for Efficient Inference of
Diffusion LLMs", Algorithm 1 layer loop and Polestar-Commit): the benchmark
workloads' shapes -- LLaDA-8B (d 4096, 32 heads, N 768), Dream-7B (d 3584, 28
query / 4 KV heads), and the batch-32 stress shape (N 2048) -- truncated in
depth and batch so that the CPU oracle keeps up (the N = 2048 and Dream cases
join their trajectory at block 1 from a seeded cache imported on both sides, so
the CPU runs no full-sequence forward), compared with the oracle at every step: K-means labels, NVFP4 codes, centroids and anchors at the block
entry; trigger, drift D, top-k sets, member rows, the incremental centroid
update, token drift, K/V of every layer, active outputs and update packets
within the block; confidences, Delta, tau_d and commit masks (tests/parity.py
states the bar)."""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from drift_aware_kv_gb300.build import build
    build()


CASES = [
    # workload, truncation, steps (one block entry + within-block steps), perturbed oracle copies, start block
    ("llada8b_p512_g256_b1", dict(n_layers=2), 6, 2, 0),
    ("dream7b_p512_g256_b4", dict(n_layers=2, batch=2), 5, 1, 1),
    ("llada8b_p1024_g1024_b32", dict(n_layers=2, batch=4), 5, 1, 1),
]


@pytest.mark.parametrize("name,trunc,steps,npert,start", CASES, ids=[c[0] for c in CASES])
def test_full_width_lockstep(name, trunc, steps, npert, start):
    from drift_aware_kv_gb300 import synth
    from parity import Lockstep
    w = synth.WORKLOADS[name].replace(**trunc)
    ls = Lockstep(w, kv_tol=1e-2, act_tol=1e-2, n_perturbed=npert, start_block=start)
    rep = ls.run(max_steps=steps)
    ls.lib.close()
    print(name, trunc, f"near ties {rep.near_ties}, sensitivity ties {rep.sensitivity_ties}", rep)
    assert rep.steps == steps
    # every step is compared in full, or ends in a counted tie after which the
    # library takes over the oracle's state and comparison goes on
    assert rep.compared + rep.resyncs == steps and rep.compared >= steps - 2 and rep.fires >= 2, rep
    assert rep.near_ties + rep.sensitivity_ties == rep.resyncs, rep


def test_state_import_round_trip():
    """polestar_debug_write of every calibration-state buffer reads back
    unchanged through polestar_debug_read (the export), and enter_block sets
    the block so that a within-block step is accepted."""
    import numpy as np
    from drift_aware_kv_gb300 import polestar as P
    from drift_aware_kv_gb300 import synth
    w = synth.WORKLOADS["mini_l2_d512_bf16"]
    W = [{k: v.cuda() for k, v in lw.items()} for lw in synth.make_weights(w)]
    ps = P.Polestar(w, W)
    g = torch.Generator().manual_seed(3)
    Wm, N, K, H, B, d = w.prefix_win + w.suffix_win, w.seq_len, w.K, w.n_heads, w.block, w.d_model
    shapes = {P.BUF_KV: ((w.batch, N, 2, w.n_kv_heads * w.head_dim), torch.bfloat16, True),
              P.BUF_LABELS: ((w.batch, Wm), torch.uint8, True),
              P.BUF_CENTROID: ((w.batch, K, d), torch.float32, True),
              P.BUF_CSUM: ((w.batch, K, d), torch.float32, True),
              P.BUF_ANCHOR: ((w.batch, K, d), torch.float32, True),
              P.BUF_CODES: ((w.batch, Wm, d // 2), torch.uint8, True),
              P.BUF_SCALES: ((w.batch, Wm, d // 16), torch.uint8, True),
              P.BUF_PROXY: ((w.batch, K, H, N), torch.float32, True),
              P.BUF_PROXY_LSE: ((w.batch, K, H), torch.float32, True),
              P.BUF_ACTIVE_PREV: ((w.batch, B, H, N), torch.float32, False),
              P.BUF_ACTIVE_LSE: ((w.batch, B, H), torch.float32, False),
              P.BUF_THETA: ((w.batch, B, w.hist), torch.float32, False),
              P.BUF_THETA_N: ((w.batch, B), torch.int32, False)}
    for which, (shape, dt, layered) in shapes.items():
        for l in (range(w.n_layers) if layered else [0]):
            if dt in (torch.uint8, torch.int32):
                x = torch.randint(0, 5, shape, generator=g).to(dt)
            else:
                x = torch.randn(shape, generator=g).to(dt)
            ps.write(which, l, x)
            assert torch.equal(ps.read(which, l, shape, dt), x), which
    with pytest.raises(P.PolestarError):
        ps.write(P.BUF_CONF, 0, torch.zeros(w.batch, 2 * B))  # an output, not state
    ps.enter_block(1, [2] * w.batch)
    tr = synth.Trajectory(w)
    st = tr.next_step()
    ps.calibrate_step(st["x0"].to(torch.bfloat16).cuda(), [1] * w.batch, 1, False)
    torch.cuda.synchronize()
    assert list(ps.last_out.fire[i] for i in range(w.batch)) == [0] * w.batch  # cum 2 + 1 = 3 does not exceed 3
    ps.close()
