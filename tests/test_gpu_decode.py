"""GPU parity of closed-loop decoding (Algorithm 1 in full: embedding, layer
loop, final norm + LM head, commit gate, progress rule, greedy tokens) against
the CPU oracle, through the C ABI (see tests/parity.py for the bar)."""
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from drift_aware_kv_gb300.build import build
    build()


def test_decode_tokens_on_shared_logits():
    """Progress rule, greedy ids, token / mask update and counts, bit-exact
    against the oracle when both sides score the same logits (the synthetic
    trajectory's), over a 14-step bf16 trajectory."""
    from drift_aware_kv_gb300 import synth
    from parity import DecodeTokensLockstep
    w = synth.WORKLOADS["mini_l2_d512_bf16"].replace(n_steps=None)
    ls = DecodeTokensLockstep(w, kv_tol=1e-2, act_tol=1e-2)
    rep = ls.run()
    ls.lib.close()
    print(rep, "progress steps", ls.progress_steps, "tokens", ls.tokens_checked)
    assert rep.compared >= 8 and ls.tokens_checked >= 20, rep
    assert ls.progress_steps >= 1


def _closed_loop(name, **tol):
    from drift_aware_kv_gb300 import synth
    from parity import ClosedLoop
    w = synth.WORKLOADS[name]
    cl = ClosedLoop(w, **tol)
    try:
        rep = cl.run()
    except AssertionError:
        print(name, "at failure:", cl.rep, "kinds", cl.steps_by_kind)
        raise
    cl.lib.close()
    print(name, rep, "kinds", cl.steps_by_kind, "max logit err", cl.max_logit_err)
    return cl, rep


def test_closed_loop_fp32():
    """Whole generation (2 sequences, 4 blocks of 32) in fp32: every step
    compared, decisions exact up to counted ties; the gate's confidence and
    drift branches, suffix commits and the progress rule all occur."""
    cl, rep = _closed_loop("loop_l1_d256_fp32", kv_tol=1e-5, act_tol=1e-5, logit_tol=1e-4, elem_tol=1e-4)
    # masked positions share one input row, so K-means distances and cluster
    # drifts can tie exactly: such steps are near ties, the rest compare
    assert rep.steps >= 8 and rep.compared >= 0.8 * rep.steps, rep
    assert rep.near_ties + rep.sensitivity_ties == rep.resyncs
    k = cl.steps_by_kind
    assert k["gate"] > 0 and k["suffix"] > 0 and k["progress"] > 0, k
    assert rep.fires >= 2, rep


def test_closed_loop_bf16():
    """The same closed loop on a two-layer bf16 stack: logits within 2e-2
    relative L2 (or the oracle's perturbed copies' band); decisions whose oracle
    margin lies outside what that difference allows must agree."""
    cl, rep = _closed_loop("loop_l2_d512_bf16", kv_tol=1e-2, act_tol=1e-2, logit_tol=2e-2, elem_tol=4e-2)
    assert rep.steps >= 8 and rep.compared >= rep.steps // 2, rep
    assert rep.near_ties + rep.sensitivity_ties == rep.resyncs
    assert rep.fires >= 2, rep
