"""NVFP4 residual store in pinned host memory (§4.1 "Cluster and Quantize Hidden
States": the quantised residuals are offloaded and fetched back on use).

With host_offload the kernels are the same and only the store's location
changes (host memory plus a two-layer device ring filled on the side stream),
so every output must be bit-identical to the device-resident run: codes,
scales, labels, drift, top-k, selections, deltas and commit masks, step by
step, including with a separate side stream."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from drift_aware_kv_gb300.build import build
    build()


def _state(ps, w, out):
    from drift_aware_kv_gb300 import polestar as P
    b, d, Wmax = w.batch, w.d_model, out.win_max
    st = {}
    for l in range(w.n_layers):
        st[("codes", l)] = ps.read(P.BUF_CODES, l, (b, Wmax, d // 2), torch.uint8).numpy()
        st[("scales", l)] = ps.read(P.BUF_SCALES, l, (b, Wmax, d // 16), torch.uint8).numpy()
        st[("labels", l)] = ps.read(P.BUF_LABELS, l, (b, Wmax), torch.uint8).numpy()
        st[("drift", l)] = ps.read(P.BUF_DRIFT, l, (b, w.K), torch.float32).numpy()
        st[("topk", l)] = ps.read(P.BUF_TOPK, l, (b, w.topk), torch.int32).numpy()
        st[("selected", l)] = ps.read(P.BUF_SELECTED, l, (b, Wmax), torch.uint8).numpy()
        st[("centroid", l)] = ps.read(P.BUF_CENTROID, l, (b, w.K, d), torch.float32).numpy()
    st["delta"] = ps.read(P.BUF_DELTA, 0, (b, w.block), torch.float32).numpy()
    return st


@pytest.mark.parametrize("name,steps,side", [("tiny_l1_d256_fp32", 16, True), ("mini_l2_d512_bf16", 14, True),
                                             ("mini_gqa_l2_d448_bf16", 12, False),
                                             ("llada8b_p512_g256_b1", 5, True)])
def test_host_offload_is_bit_identical(name, steps, side):
    from drift_aware_kv_gb300 import polestar as P
    from drift_aware_kv_gb300 import synth
    w = synth.WORKLOADS[name]
    W = synth.make_weights(w, "cuda")
    side_stream = torch.cuda.Stream() if side else None
    ref = P.Polestar(w, W)
    off = P.Polestar(w, W, side_stream=side_stream, host_offload=True)
    tr = synth.Trajectory(w)
    dt = synth.torch_dtype(w)
    cm_r = torch.zeros(w.batch, 2 * w.block, dtype=torch.uint8, device="cuda")
    cm_o = torch.zeros_like(cm_r)
    fired = 0
    for _ in range(steps):
        st = tr.next_step()
        if st is None:
            break
        x0 = st["x0"].to(dt).cuda()
        logits, masked = st["logits"].cuda(), st["masked"].to(torch.uint8).cuda()
        out_r = ref.calibrate_step(x0, st["n_unmasked"], st["block_index"], st["block_entry"])
        fire_r = [bool(out_r.fire[s]) for s in range(w.batch)]
        ref.commit(logits, masked, cm_r)
        out_o = off.calibrate_step(x0, st["n_unmasked"], st["block_index"], st["block_entry"])
        fire_o = [bool(out_o.fire[s]) for s in range(w.batch)]
        off.commit(logits, masked, cm_o)
        torch.cuda.synchronize()
        assert fire_r == fire_o
        fired += sum(fire_r) if not st["block_entry"] else 0
        a, b = _state(ref, w, out_r), _state(off, w, out_o)
        for k in a:
            assert np.array_equal(a[k], b[k]), (st["t"], k)
        assert torch.equal(cm_r, cm_o)
    ref.close()
    off.close()
    assert fired >= 1


@pytest.mark.parametrize("name,steps", [("tiny_l1_d256_fp32", 16), ("mini_l2_d512_bf16", 14)])
def test_step_host_is_bit_identical(name, steps):
    """polestar_step_host (host inputs, the commit's inputs copied on the
    context's copy stream while the calibration computes) against the same
    steps on device buffers: identical state and commit masks at every step.
    One set of pinned host buffers is rewritten for every step, as a caller
    reusing its staging buffers does once the call has returned."""
    from drift_aware_kv_gb300 import polestar as P
    from drift_aware_kv_gb300 import synth
    w = synth.WORKLOADS[name]
    W = synth.make_weights(w, "cuda")
    ref = P.Polestar(w, W)
    hst = P.Polestar(w, W)
    tr = synth.Trajectory(w)
    dt = synth.torch_dtype(w)
    cm_r = torch.zeros(w.batch, 2 * w.block, dtype=torch.uint8, device="cuda")
    cm_h = torch.zeros(w.batch, 2 * w.block, dtype=torch.uint8).pin_memory()
    x0_h = logits_h = masked_h = None
    for _ in range(steps):
        st = tr.next_step()
        if st is None:
            break
        x0 = st["x0"].to(dt)
        logits, masked = st["logits"].float(), st["masked"].to(torch.uint8)
        if x0_h is None:
            x0_h = torch.empty_like(x0).pin_memory()
            logits_h = torch.empty_like(logits).pin_memory()
            masked_h = torch.empty_like(masked).pin_memory()
        x0_h.copy_(x0)
        logits_h.copy_(logits)
        masked_h.copy_(masked)
        out_r = ref.calibrate_step(x0.cuda(), st["n_unmasked"], st["block_index"], st["block_entry"])
        ref.commit(logits.cuda(), masked.cuda(), cm_r)
        hst.step_host(x0_h, st["n_unmasked"], st["block_index"], st["block_entry"], logits_h, masked_h, cm_h)
        torch.cuda.synchronize()
        a, b = _state(ref, w, out_r), _state(hst, w, out_r)
        for k in a:
            assert np.array_equal(a[k], b[k]), (st["t"], k)
        assert torch.equal(cm_r.cpu(), cm_h), st["t"]
    ref.close()
    hst.close()
