"""Fixtures under tests/golden/: the paper's Table 5 defaults (printed values) and
the §4.2 dynamic threshold at those defaults (values derived by hand from the
printed formula).  The library's default workloads, the C header's documented
defaults and the oracle's gate must agree with them."""
import os
import re

import numpy as np

from drift_aware_kv_gb300 import synth
from oracle import polestar_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


def _pairs(name):
    out = []
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def test_workload_defaults_follow_table5():
    t = {k: v for k, v in _pairs("table5_defaults.txt")}
    for w in synth.WORKLOADS.values():
        assert w.block == int(t["block"])
        assert w.prefix_win == int(t["prefix_win_blocks"]) * w.block
        assert w.suffix_win == int(t["suffix_win_blocks"]) * w.block
        assert (w.K, w.topk, w.tau_upd, w.hist) == (int(t["K"]), int(t["topk"]), int(t["tau_upd"]), int(t["hist"]))
        assert (w.tau_s, w.alpha, w.tau_suf) == (float(t["tau_s"]), float(t["alpha"]), float(t["tau_suf"]))
    assert t["residual_format"] == "nvfp4"


def test_header_documents_table5_defaults():
    """include/polestar.h gives each hyper-parameter's default in brackets."""
    t = {k: v for k, v in _pairs("table5_defaults.txt")}
    hdr = open(os.path.join(os.path.dirname(HERE), "include", "polestar.h")).read()
    for field, key in (("block", "block"), ("K", "K"), ("topk", "topk"), ("tau_upd", "tau_upd"), ("hist", "hist"),
                       ("tau_s", "tau_s"), ("tau_suf", "tau_suf"), ("alpha", "alpha")):
        m = re.search(r"\b" + field + r";[^\[]*\[([0-9.]+)\]", hdr)
        assert m, field
        assert float(m.group(1)) == float(t[key]), field


def test_gate_threshold_at_defaults():
    t = {k: v for k, v in _pairs("table5_defaults.txt")}
    for c, td in _pairs("gate_thresholds.txt"):
        got = O.drift_threshold(float(c), float(t["tau_s"]), float(t["alpha"]))
        assert np.isclose(got, float(td), rtol=0, atol=1e-12), (c, got)
