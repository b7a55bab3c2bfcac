"""Bounded device waits: a wait that runs out is an error status, not a hang.

Every mbarrier wait of the projection kernels gives up after a bound, records a
code in the context's device error word and lets its kernel return; the next
call on the context reports POLESTAR_ERR_TIMEOUT and leaves the context as it
was.  The test shortens the bound through the library's hook and runs a kernel
whose barrier nobody ever arrives on -- no fault, no trap, no endless loop."""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from drift_aware_kv_gb300.build import build
    build()


def _steps(w, n):
    from drift_aware_kv_gb300 import synth
    tr = synth.Trajectory(w)
    return [tr.next_step() for _ in range(n)]


def test_wait_that_runs_out_reports_timeout_and_context_stays_usable():
    from drift_aware_kv_gb300 import polestar as P
    from drift_aware_kv_gb300 import synth
    w = synth.WORKLOADS["mini_l2_d512_bf16"]
    W = [{k: v.cuda() for k, v in lw.items()} for lw in synth.make_weights(w)]
    steps = _steps(w, 3)
    dt = synth.torch_dtype(w)
    ref = P.Polestar(w, W)
    ps = P.Polestar(w, W)
    for st in steps[:2]:
        ref.calibrate_step(st["x0"].to(dt).cuda(), st["n_unmasked"], st["block_index"], st["block_entry"])
        ps.calibrate_step(st["x0"].to(dt).cuda(), st["n_unmasked"], st["block_index"], st["block_entry"])
    assert ps.lib.polestar_debug_stalled_wait(ps.ctx, 2_000_000) == P.OK  # ~1 ms at 2 GHz
    torch.cuda.synchronize()
    st = steps[2]
    x0 = st["x0"].to(dt).cuda()
    with pytest.raises(P.PolestarError) as ei:
        ps.calibrate_step(x0, st["n_unmasked"], st["block_index"], st["block_entry"])
    assert ei.value.status == P.ERR_TIMEOUT and "timed out (code 99)" in str(ei.value)
    # the failed call changed nothing: the same step now runs and matches a
    # context that never saw the stalled wait, bit for bit
    ps.calibrate_step(x0, st["n_unmasked"], st["block_index"], st["block_entry"])
    ref.calibrate_step(x0, st["n_unmasked"], st["block_index"], st["block_entry"])
    torch.cuda.synchronize()
    for l in range(w.n_layers):
        shape = (w.batch, w.seq_len, 2, w.n_kv_heads * w.head_dim)
        assert torch.equal(ps.read(P.BUF_KV, l, shape, dt), ref.read(P.BUF_KV, l, shape, dt))
    cm = torch.zeros(w.batch, 2 * w.block, dtype=torch.uint8, device="cuda")
    ps.commit(st["logits"].cuda(), st["masked"].to(torch.uint8).cuda(), cm)
    torch.cuda.synchronize()
    ps.close()
    ref.close()


def test_stalled_wait_rejects_bad_arguments():
    from drift_aware_kv_gb300 import polestar as P
    from drift_aware_kv_gb300 import synth
    w = synth.WORKLOADS["mini_l2_d512_bf16"]
    W = [{k: v.cuda() for k, v in lw.items()} for lw in synth.make_weights(w)]
    ps = P.Polestar(w, W)
    assert ps.lib.polestar_debug_stalled_wait(ps.ctx, 0) == P.ERR_INVALID_ARG
    assert ps.lib.polestar_debug_stalled_wait(ps.ctx, -5) == P.ERR_INVALID_ARG
    ps.close()
