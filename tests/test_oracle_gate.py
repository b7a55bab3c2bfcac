"""Closed-form cases of the oracle's commit gate (Polestar-Commit, §4.2 of
"Polestar: Drift-Aware Cache Calibration and Token Commitment for Efficient
Inference of Diffusion LLMs"; the commit phases of Algorithm 1), on a hand-built
state: the current-block rule (confidence at or above tau_s, or drift delta at or
above the dynamic threshold), the drift history (mean of the last h drifts, the
current one excluded, an empty history counting as 0, then the push), the
suffix-block rule (a refreshing step, a selected cluster, confidence at or above
tau_suf) and the block-entry rule (confidence alone)."""
import math

import numpy as np

from drift_aware_kv_gb300 import synth
from oracle import polestar_oracle as O

CFG = synth.WORKLOADS["tiny_l1_d256_fp32"]  # B = 32, prompt 64, window 64 + 32, V = 512
B, V = CFG.block, CFG.vocab


def _logits_for(conf):
    """Rows whose max softmax probability is conf (one raised entry, the rest 0)."""
    conf = np.asarray(conf, dtype=np.float64)
    lg = np.zeros((len(conf), V))
    lg[:, 0] = np.log(conf * (V - 1) / (1.0 - conf))
    return lg


def _oracle(block_entry=False, fire=True):
    orc = O.PolestarOracle.__new__(O.PolestarOracle)
    orc.cfg, orc.N = CFG, CFG.seq_len
    orc.block, orc.block_entry = 0, block_entry
    st = O.SeqState(kv=[])
    st.theta = [[] for _ in range(B)]
    st.delta = np.zeros(B)
    st.fire = fire
    st.sel_last = np.zeros(len(orc.window(0)), dtype=bool)
    orc.seqs = [st]
    return orc, st


def test_current_block_rule_and_history():
    orc, st = _oracle()
    conf = np.full(2 * B, 0.6)
    masked = np.zeros(CFG.seq_len, dtype=bool)
    masked[64:128] = True
    # j = 0: confident enough alone
    conf[0] = 0.95
    # j = 1..3: c = 0.8 -> tau_d = alpha (tau_s - c)^2 = 0.1 (up to rounding of c)
    conf[1:4] = 0.8
    td = O.drift_threshold(_conf_of(0.8), CFG.tau_s, CFG.alpha)
    st.delta[1], st.delta[2], st.delta[3] = 0.2, 0.05, td  # above, below, exactly at tau_d
    # j = 4: history [0.1, 0.3] -> Delta = 0.5 - 0.2 = 0.3 >= tau_d(0.8)
    conf[4] = 0.8
    st.theta[4] = [0.1, 0.3]
    st.delta[4] = 0.5
    # j = 5: only the last h = 5 drifts count: [9, 0, 0, 0, 0, 0] -> mean 0, Delta = 0.12
    conf[5] = 0.8
    st.theta[5] = [9.0, 0, 0, 0, 0, 0]
    st.delta[5] = 0.12
    # j = 6: same drift but the old entry inside the window: mean 9/5 -> Delta < 0
    conf[6] = 0.8
    st.theta[6] = [9.0, 0, 0, 0, 0]
    st.delta[6] = 0.12
    # j = 7: would commit, but already unmasked
    conf[7] = 0.95
    masked[64 + 7] = False
    out = orc.commit(_logits_for(conf)[None], masked[None])[0]
    m = out["commit"]
    assert list(m[:8]) == [True, True, False, True, True, True, False, False]
    assert math.isclose(out["tau_d"][1], 0.1, rel_tol=0, abs_tol=1e-9)
    assert math.isclose(out["delta_rel"][4], 0.3, abs_tol=1e-15)
    assert math.isclose(out["delta_rel"][5], 0.12, abs_tol=1e-15)
    assert math.isclose(out["delta_rel"][6], 0.12 - 9.0 / 5, abs_tol=1e-12)
    # the current drift is pushed after use; the history keeps the last h entries
    assert st.theta[4] == [0.1, 0.3, 0.5]
    assert st.theta[5] == [0, 0, 0, 0, 0.12]


def _conf_of(c):
    """The confidence the oracle computes for a row built to have max-prob c."""
    return float(O.confidence(_logits_for([c]))[0])


def test_suffix_block_rule():
    orc, st = _oracle(fire=True)
    win = orc.window(0)
    suffix = [wi for wi, p in enumerate(win) if p >= 96]  # suffix positions 96..127
    conf = np.full(2 * B, 0.6)
    masked = np.ones(CFG.seq_len, dtype=bool)
    # suffix rows (j = B + i for position 96 + i)
    conf[B + 0], conf[B + 1], conf[B + 2] = 0.95, 0.95, 0.85
    st.sel_last[suffix[0]] = True   # selected, confident: commit
    st.sel_last[suffix[2]] = True   # selected, below tau_suf: no
    # suffix[1] confident but its cluster not selected: no
    out = orc.commit(_logits_for(conf)[None], masked[None])[0]["commit"]
    assert list(out[B:B + 3]) == [True, False, False]
    assert not out[B + 3:].any()
    # a step without refresh commits no suffix token
    orc2, st2 = _oracle(fire=False)
    st2.sel_last[:] = True
    out2 = orc2.commit(_logits_for(conf)[None], masked[None])[0]["commit"]
    assert not out2[B:].any()


def test_block_entry_rule_is_confidence_only():
    orc, st = _oracle(block_entry=True)
    conf = np.full(2 * B, 0.6)
    conf[:3] = [0.95, 0.85, 0.91]
    st.delta[:] = 10.0  # drift plays no part at block entry
    masked = np.ones(CFG.seq_len, dtype=bool)
    out = orc.commit(_logits_for(conf)[None], masked[None])[0]["commit"]
    assert list(out[:3]) == [True, False, True] and not out[3:].any()
