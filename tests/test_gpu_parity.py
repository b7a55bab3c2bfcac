"""GPU parity: the CUDA library through its C ABI against the CPU oracle, in
lockstep over seeded synthetic trajectories (see tests/parity.py for the bar)."""
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from drift_aware_kv_gb300.build import build
    build()


def _run(name, kv_tol, act_tol, **kw):
    from drift_aware_kv_gb300 import synth
    from parity import Lockstep
    w = synth.WORKLOADS[name].replace(**kw)
    ls = Lockstep(w, kv_tol=kv_tol, act_tol=act_tol)
    rep = ls.run()
    ls.lib.close()
    print(name, f"near ties {rep.near_ties}, sensitivity ties {rep.sensitivity_ties}", rep)
    return rep


def test_tiny_fp32_trajectory():
    """Single-layer fp32 workload, 16 steps: every decision exact, fp32 tolerances."""
    rep = _run("tiny_l1_d256_fp32", kv_tol=1e-5, act_tol=1e-5)
    assert rep.compared >= 12 and rep.fires >= 2, rep
    assert rep.near_ties <= 1


@pytest.mark.parametrize("name", ["mini_l2_d512_bf16", "mini_gqa_l2_d448_bf16"])
def test_mini_bf16_trajectory(name):
    """Two-layer bf16 stacks (MHA and 7:1 GQA): decisions exact up to counted near
    ties and sensitivity ties (the oracle's own perturbed copies); KL within
    1e-5 + 1e-3 rel plus the oracle-measured band; K/V, active outputs and
    update packets within 1e-2 relative L2."""
    rep = _run(name, kv_tol=1e-2, act_tol=1e-2, n_steps=None)
    assert rep.compared >= 8 and rep.fires >= 3, rep
    assert rep.near_ties + rep.sensitivity_ties <= 3


def test_mini_bf16_trajectory_nonunit_norm_gains():
    """The same lockstep with distinct, non-unit RMSNorm gains per norm and layer
    (the benchmark shapes use gains 1): a swap of the attention and FFN norms,
    or a gain applied twice or not at all, cannot pass."""
    rep = _run("mini_l2_d512_bf16", kv_tol=1e-2, act_tol=1e-2, n_steps=None, norm_gain_std=0.3)
    assert rep.compared >= 8 and rep.fires >= 3, rep
    assert rep.near_ties + rep.sensitivity_ties <= 3


def test_mini_bf16_trajectory_tcgen05_attention():
    """The same lockstep with every attention launch (within-block rows with KL,
    block entries, proxy baselines) on the tcgen05 kernel (head size 128)."""
    from drift_aware_kv_gb300 import polestar as P
    old = P.attention_impl(2)
    try:
        rep = _run("mini_l2_d512_bf16", kv_tol=1e-2, act_tol=1e-2, n_steps=None)
    finally:
        P.attention_impl(old)
    assert rep.compared >= 8 and rep.fires >= 3, rep
    assert rep.near_ties + rep.sensitivity_ties <= 3
