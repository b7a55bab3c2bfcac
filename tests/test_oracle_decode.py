"""Pins of the oracle's closed-loop decoding steps (Eq. 1 greedy reconstruction,
the progress rule, the token / mask update, the layer-0 inputs, the LM head),
each against hand-worked cases or closed forms, not against the oracle's own
formulas."""
import numpy as np

from oracle import polestar_oracle as O


def test_greedy_tokens_first_maximum_and_margin():
    l = np.array([[1.0, 3.0, 3.0, -2.0],    # tie between ids 1 and 2 -> 1, margin 0
                  [0.5, -1.0, 2.0, 1.5],     # id 2, gap 0.5 over |2|
                  [-4.0, -1.0, -3.0, -2.0]])  # all negative: id 1, gap 1 over |-1|
    ids, margin = O.greedy_tokens(l)
    assert ids.tolist() == [1, 2, 1]
    assert margin.tolist() == [0.0, 0.25, 1.0]


def test_progress_rule_cases():
    conf = np.array([0.3, 0.8, 0.8, 0.1])
    # nothing committed, all masked: the most confident, lower position on a tie
    assert O.progress_rule([0, 0, 0, 0], conf, [1, 1, 1, 1]).tolist() == [False, True, False, False]
    # position 1 no longer masked: position 2
    assert O.progress_rule([0, 0, 0, 0], conf, [1, 0, 1, 1]).tolist() == [False, False, True, False]
    # a committed masked token already makes progress: unchanged
    assert O.progress_rule([0, 0, 0, 1], conf, [1, 1, 1, 1]).tolist() == [False, False, False, True]
    # nothing masked: nothing to commit
    assert O.progress_rule([0, 0, 0, 0], conf, [0, 0, 0, 0]).tolist() == [False] * 4
    # a commit flag on an unmasked position is no progress: the rule still fires
    assert O.progress_rule([1, 0, 0, 0], conf, [0, 0, 0, 1]).tolist() == [True, False, False, True]


def test_apply_commits_hand_case():
    tokens = np.array([7, 7, 0, 0, 0, 0])
    masked = np.array([False, False, True, True, True, True])
    # 2B = 4 rows from position 2; row 3 lies past the end (position 6)
    n = O.apply_commits(tokens, masked, np.array([1, 0, 1, 1], dtype=bool), np.array([11, 12, 13, 14]), start=3)
    assert n == 2
    assert tokens.tolist() == [7, 7, 0, 11, 0, 13]
    assert masked.tolist() == [False, False, True, False, True, False]
    # a committed row whose position is no longer masked changes nothing
    n = O.apply_commits(tokens, masked, np.array([1, 1, 0, 0], dtype=bool), np.array([21, 22, 23, 24]), start=0)
    assert n == 0 and tokens.tolist() == [7, 7, 0, 11, 0, 13]


def test_embed_inputs_hand_case():
    E = np.arange(12, dtype=np.float64).reshape(4, 3)
    m = np.array([-1.0, -2.0, -3.0])
    x = O.embed_inputs(np.array([2, 0, 3]), np.array([False, True, False]), E, m)
    assert x.tolist() == [[6, 7, 8], [-1, -2, -3], [9, 10, 11]]


def test_lm_logits_closed_form():
    """A row c * s (s in {+1, -1}^d) has RMS |c|, so its normalised form is
    sign(c) * s * gain; with a +-1 LM head the logits are integer sums."""
    d = 8
    s = np.array([1, -1, 1, 1, -1, -1, 1, -1], dtype=np.float64)
    gain = np.array([1, 2, 1, 2, 1, 2, 1, 2], dtype=np.float64)
    W = np.array([[1] * 8, [1, -1] * 4, [-1] * 8], dtype=np.float64)
    for c in (3.0, -0.5):
        x = np.sign(c) * s * gain
        want = W @ x
        got = O.lm_logits((c * s)[None], W, gain, eps=0.0, bf16=False)[0]
        assert np.allclose(got, want, rtol=0, atol=1e-12), (got, want)
    # the bf16 rounding of the normalised row: 1/3 gains -> nearest bf16 values
    g3 = np.full(d, 1.0 / 3.0)
    got = O.lm_logits(s[None], np.eye(d), g3, eps=0.0, bf16=True)[0]
    assert np.all(np.abs(got) == 0.333984375)  # bf16(1/3) = 0x3EAB
