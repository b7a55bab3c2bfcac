"""Full-size workloads through the C ABI (LLaDA-8B shape at batch 1, 8 and 32 with
N up to 2048; Dream-7B shape with 28/4 grouped-query heads at batch 4).

The CPU oracle cannot run a 32-layer step in seconds, so these runs are checked
through outputs the oracle computes one by one on the caller's inputs
(confidence of sampled logit rows) and through properties that hold at any
size: the tau_upd trigger (§4.1 "Update Schedule"), KL drift >= 0 (Eq. 4), top-k
sets of distinct clusters whose members are exactly the selected rows (§4.1),
the last K-means update (every non-empty cluster's member sum, unit centroid
and anchor follow from the final labels; ten Lloyd iterations need not reach
a fixed point, so labels are not compared with the final centroids), NVFP4
codes on the E2M1 grid within half a grid step of the block-entry inputs
(App. C.3), and the commit gate recomputed from the exported c, Delta and
tau_d (§4.2)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from oracle import polestar_oracle as O  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from drift_aware_kv_gb300.build import build
    build()


def _check_entry(ps, w, nw, Wmax):
    from drift_aware_kv_gb300 import polestar as P
    b, d, K = w.batch, w.d_model, w.K
    for l in (0, w.n_layers // 2, w.n_layers - 1):
        lab = ps.read(P.BUF_LABELS, l, (b, Wmax), torch.uint8).numpy()[:, :nw]
        z = ps.read(P.BUF_CENTROID, l, (b, K, d), torch.float32).numpy()
        Hw = ps.read(P.BUF_WINDOW_H, l, (b, Wmax, d), torch.float32).numpy()[:, :nw]
        A = ps.read(P.BUF_ANCHOR, l, (b, K, d), torch.float32).numpy()
        codes = ps.read(P.BUF_CODES, l, (b, Wmax, d // 2), torch.uint8).numpy()[:, :nw]
        scales = ps.read(P.BUF_SCALES, l, (b, Wmax, d // 16), torch.uint8).numpy()[:, :nw]
        assert np.allclose(np.linalg.norm(z, axis=-1), 1.0, atol=1e-4)
        csum = ps.read(P.BUF_CSUM, l, (b, K, d), torch.float32).numpy()
        for s in range(min(b, 4)):
            X = Hw[s] / np.linalg.norm(Hw[s], axis=1, keepdims=True)
            # the last update of spherical K-means: every non-empty cluster's sum,
            # unit centroid and anchor follow from the final labels (whether or
            # not the iterations have converged)
            for c in range(K):
                mem = lab[s] == c
                if not mem.any():
                    continue
                ssum = X[mem].astype(np.float64).sum(0)
                assert np.allclose(csum[s, c], ssum, rtol=1e-4, atol=1e-4 * np.abs(ssum).max())
                zc = ssum / np.linalg.norm(ssum)
                assert float(zc @ z[s, c]) > 1 - 1e-6
                assert np.allclose(A[s, c], Hw[s][mem].astype(np.float64).mean(0), rtol=1e-4,
                                   atol=1e-4 * np.abs(Hw[s][mem]).max())
            c = np.stack([codes[s] & 0xF, codes[s] >> 4], -1).reshape(nw, d)
            sv = O.e4m3_value(scales[s]).reshape(nw, d // 16, 1)
            dec = (O.e2m1_value(c).reshape(nw, d // 16, 16) * sv).reshape(nw, d)
            r = Hw[s] - A[s][lab[s]]
            step = np.where(np.abs(dec) >= 4 * np.repeat(sv.reshape(nw, -1), 16, 1), 2.0,
                            np.where(np.abs(dec) >= 2 * np.repeat(sv.reshape(nw, -1), 16, 1), 1.0, 0.5))
            bound = step / 2 * np.repeat(sv.reshape(nw, -1), 16, 1)
            over = np.abs(r) > 6 * np.repeat(sv.reshape(nw, -1), 16, 1)
            assert np.all((np.abs(r - dec) <= bound * (1 + 1e-5) + 1e-6) | over)


def _check_step(ps, w, out, st, cum):
    from drift_aware_kv_gb300 import polestar as P
    b, L, K = w.batch, w.n_layers, w.K
    nw, Wmax = out.win_len, out.win_max
    fire = [bool(out.fire[s]) for s in range(b)]
    for s in range(b):
        cum[s] += st["n_unmasked"][s]
        want = cum[s] > w.tau_upd
        assert fire[s] == want
        if want:
            cum[s] = 0
    for l in (0, L - 1):
        D = ps.read(P.BUF_DRIFT, l, (b, K), torch.float32).numpy()
        tk = ps.read(P.BUF_TOPK, l, (b, w.topk), torch.int32).numpy()
        sel = ps.read(P.BUF_SELECTED, l, (b, Wmax), torch.uint8).numpy()[:, :nw]
        lab = ps.read(P.BUF_LABELS, l, (b, Wmax), torch.uint8).numpy()[:, :nw]
        for s in range(b):
            if not fire[s]:
                continue
            assert np.all(np.isfinite(D[s])) and np.all(D[s] >= -1e-6)
            assert len(set(tk[s].tolist())) == w.topk
            order = sorted(range(K), key=lambda c: (-D[s][c], c))[: w.topk]
            assert sorted(order) == sorted(tk[s].tolist())
            assert np.array_equal(sel[s].astype(bool), np.isin(lab[s], tk[s]))
    delta = ps.read(P.BUF_DELTA, 0, (b, w.block), torch.float32).numpy()
    assert np.all(np.isfinite(delta)) and np.all(delta >= -1e-6)
    return fire


def _check_commit(ps, w, st, cm, entry):
    from drift_aware_kv_gb300 import polestar as P
    b, B = w.batch, w.block
    conf = ps.read(P.BUF_CONF, 0, (b, 2 * B), torch.float32).numpy()
    drel = ps.read(P.BUF_DREL, 0, (b, 2 * B), torch.float32).numpy()
    taud = ps.read(P.BUF_TAUD, 0, (b, 2 * B), torch.float32).numpy()
    start = w.prompt_len + st["block_index"] * B
    for s in range(min(b, 3)):
        rows = [0, 7, B - 1, B]
        c_o = O.confidence(st["logits"][s, rows].numpy())  # one by one from the caller's logits
        assert np.allclose(conf[s, rows], c_o, rtol=2e-6, atol=1e-7)
        m = st["masked"][s].numpy()[start:start + B]
        got = cm[s, :B].astype(bool)
        if entry:
            want = m & (conf[s, :B] >= w.tau_s)
        else:
            assert np.allclose(taud[s, :B], w.alpha * (w.tau_s - conf[s, :B]) ** 2, rtol=1e-5, atol=1e-7)
            want = m & ((conf[s, :B] >= w.tau_s) | (drel[s, :B] >= taud[s, :B]))
        assert np.array_equal(got, want)


@pytest.mark.parametrize("name,steps", [("llada8b_p512_g256_b1", 10), ("llada8b_p512_g512_b8", 6),
                                        ("dream7b_p512_g256_b4", 6), ("llada8b_p1024_g1024_b32", 3)])
def test_fullsize_workload(name, steps):
    from drift_aware_kv_gb300 import polestar as P
    from drift_aware_kv_gb300 import synth
    w = synth.WORKLOADS[name]
    W = synth.make_weights(w, "cuda")
    ps = P.Polestar(w, W)
    tr = synth.Trajectory(w)
    dt = synth.torch_dtype(w)
    cum = [0] * w.batch
    fires = 0
    cm = torch.zeros(w.batch, 2 * w.block, dtype=torch.uint8, device="cuda")
    for _ in range(steps):
        st = tr.next_step()
        out = ps.calibrate_step(st["x0"].to(dt).cuda(), st["n_unmasked"], st["block_index"], st["block_entry"])
        ps.commit(st["logits"].cuda(), st["masked"].to(torch.uint8).cuda(), cm)
        torch.cuda.synchronize()
        if st["block_entry"]:
            cum = [0] * w.batch
            _check_entry(ps, w, out.win_len, out.win_max)
        else:
            fires += sum(_check_step(ps, w, out, st, cum))
        _check_commit(ps, w, st, cm.cpu().numpy(), st["block_entry"])
    ps.close()
    assert fires >= 1
